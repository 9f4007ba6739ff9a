"""How far bf16 rounding decisions taken the other way move the drafter's logits.

Run by hand (CPU, oracle only; about half a minute for the Qwen3-8B-shaped workload):

    python tests/rounding_sensitivity.py [workload] [relative perturbation]

The oracle is run twice on the same sequence: once as is, once with every value
multiplied by (1 + rel * N(0, 1)) just before each bf16 rounding point of the contract,
which is what an fp32 (rather than fp64) evaluation of the same formulas does to the
pre-rounding values.  Values lying that close to a rounding boundary round the other
way; over a long context and several layers those one-ulp flips add up.  The printed
maximum logit change is what the GPU parity tests allow as the margin below which a
GPU draft may legitimately differ from the oracle's (they measure it per row from the
GPU's own final hidden state).
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), ".."))

from oracle import dflash_oracle as O  # noqa: E402
from oracle import run as orun  # noqa: E402
from workload import configs  # noqa: E402


def sensitivity(w, rel=1e-7, b=0, seed=1):
    W = orun.host_weights(w)
    base = orun.draft_sequence(w, W, b)
    orig = O._maybe_bf16
    rng = np.random.default_rng(seed)

    def perturbed(x, bf16):
        x = np.asarray(x, dtype=np.float64)
        if bf16:
            x = x * (1.0 + rel * rng.standard_normal(x.shape))
        return orig(x, bf16)

    O._maybe_bf16 = perturbed
    try:
        pert = orun.draft_sequence(w, W, b)
    finally:
        O._maybe_bf16 = orig
    dh = pert["h"] - base["h"]
    return {
        "h_rms_rel": float(np.sqrt((dh ** 2).mean() / (base["h"] ** 2).mean())),
        "h_normwise": float(np.abs(dh).max() / np.abs(base["h"]).max()),
        "max_logit_change": float(np.abs(pert["z"] - base["z"]).max()),
        "drafts_changed": int((pert["draft"] != base["draft"]).sum()),
        "k_flip_frac": float(np.mean([(pert["K"][l] != base["K"][l]).mean()
                                      for l in range(w.n_layers)])),
    }


if __name__ == "__main__":
    name = sys.argv[1] if len(sys.argv) > 1 else "qwen3-8b-shaped-b1"
    rel = float(sys.argv[2]) if len(sys.argv) > 2 else 1e-7
    w = configs.BY_NAME[name]
    print(name, rel, sensitivity(w, rel))
