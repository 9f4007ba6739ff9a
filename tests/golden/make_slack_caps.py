"""Writes tests/golden/slack_caps.json: per workload, the largest change of the drafter's
logits that bf16 rounding decisions taken the other way cause, measured on the oracle
alone (no GPU, no value from the CUDA path).

For every checked sequence of a workload the fp64 oracle runs once as is and then with
every value multiplied by (1 + rel * N(0, 1)) just before each bf16 rounding point of
the rounding contract (fused features, injected K/V, RMSNorm outputs that feed a
projection, q/k/v after RoPE, the attention output, the SwiGLU product, the final
hidden state), which is what evaluating the same formulas with fp32 instead of fp64
sums does to those values.  Values that close to a rounding boundary round the other
way; the stored figure is the largest |z_perturbed - z| over the rows, the vocabulary,
the sequences, the seeds and rel in {1e-7, 1e-6}.  The GPU parity tests allow their own
logit deviation up to a stated multiple of it (tests/parity_plan.py).

    python tests/golden/make_slack_caps.py [--only NAME ...] [--seeds N] [--out FILE]
    python tests/golden/make_slack_caps.py --merge FILE ...   # into slack_caps.json

(--out writes the named workloads to a separate file, so that several workloads can
be measured by parallel processes and merged afterwards.)

Fp32 workloads have no rounding point beyond fp32 storage of the inputs (the perturbed
run equals the plain one); their figure is instead the largest logit change that the
fp32 tolerance on the final hidden state admits: |dz_v| <= ||dh||_2 ||W_lm[v]||_2 with
every |dh_i| at 1e-4 max|h| (the normwise tolerance), i.e. sqrt(d) 1e-4 max|h|
max_v ||W_lm[v]||_2.
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(HERE))

from oracle import dflash_oracle as O  # noqa: E402
from oracle import run as orun  # noqa: E402
from workload import configs, inputs  # noqa: E402

import parity_plan  # noqa: E402

RELS = (1e-7, 1e-6)


INPUT = "input:"   # name prefix of the input-fusion variant of a workload

# the workloads whose input-fusion variant the GPU tests compare
INPUT_FUSION = ["tiny-f32", "small-bf16-hd128", "small-bf16-b1", "small-bf16-hd64-g8-b6-tc",
                "small-bf16-b20-tc256", "qwen3-8b-shaped-b1"]


def draft_of(w, variant):
    return orun.draft_sequence_input if variant == "input" else orun.draft_sequence


def perturbed_run(w, W, b, rel, seed, variant="kv"):
    """The oracle's draft of sequence b with every pre-rounding value perturbed by a
    relative rel * N(0, 1) (seeded)."""
    orig = O._maybe_bf16
    rng = np.random.default_rng(seed)

    def perturbed(x, bf16):
        x = np.asarray(x, dtype=np.float64)
        if bf16:
            x = x * (1.0 + rel * rng.standard_normal(x.shape))
        return orig(x, bf16)

    O._maybe_bf16 = perturbed
    try:
        return draft_of(w, variant)(w, W, b)
    finally:
        O._maybe_bf16 = orig


# sequences studied per large workload (the oracle takes minutes per run at 8k-16k
# contexts): the shortest, the median and the longest context of the GPU tests' sample
N_STUDIED = 3


def sequences_of(w):
    """The sequences whose rounding sensitivity is measured: every sequence of a small
    workload; for a large one the shortest, median and longest of the sequences the GPU
    tests compare with the full oracle."""
    small = w.name in configs.PARITY_SMALL or w.name.removesuffix("-fp8") in configs.PARITY_SMALL
    if small or w.batch <= N_STUDIED:
        return list(range(w.batch))
    lens = inputs.ctx_lens(w).numpy()
    sample = parity_plan.sampled_sequences(lens)
    if len(sample) <= N_STUDIED:
        return sample
    order = sorted(sample, key=lambda b: (lens[b], b))
    return sorted({order[0], order[len(order) // 2], order[-1]})


def study(w, seeds, variant="kv"):
    W = orun.host_weights(w)
    # every run of a sequence draws the same context features: draw them once
    draw = inputs.ctx_hidden
    cache = {}

    def ctx_hidden(w_, b, p0, p1, device="cpu"):
        key = (w_.name, b, p0, p1, device)
        if key not in cache:
            cache.clear()
            cache[key] = draw(w_, b, p0, p1, device)
        return cache[key]

    inputs.ctx_hidden = ctx_hidden
    try:
        return _study(w, W, seeds, variant)
    finally:
        inputs.ctx_hidden = draw


def _study(w, W, seeds, variant):
    per_seq = {}
    for b in sequences_of(w):
        base = draft_of(w, variant)(w, W, b)
        worst = 0.0
        if w.dtype != "bf16":
            wl = np.asarray(W["lm_head"], dtype=np.float64)
            worst = float(np.sqrt(w.d_model) * 1e-4 * np.abs(base["h"]).max()
                          * np.sqrt((wl * wl).sum(axis=1)).max())
        for rel in (RELS if w.dtype == "bf16" else ()):
            for s in range(seeds if rel == RELS[0] else 1):
                p = perturbed_run(w, W, b, rel, 1000 * b + s + 1, variant)
                worst = max(worst, float(np.abs(p["z"] - base["z"]).max()))
        per_seq[str(b)] = {"worst_logit_change": worst, "ctx_len": int(base["T"]),
                           "rows_margin_below_2cap": None,
                           "min_margin": float(base["margin"].min())}
        per_seq[str(b)]["_margin"] = base["margin"].tolist()
    worst = max(v["worst_logit_change"] for v in per_seq.values())
    cap2 = 2 * parity_plan.CAP_FACTOR * worst
    for v in per_seq.values():
        v["rows_margin_below_2cap"] = int(sum(m < max(1e-2, cap2) for m in v.pop("_margin")))
    return {"worst_logit_change": worst, "sequences": per_seq}


def all_workloads():
    ws = dict(configs.PARITY_SMALL)
    ws.update({w.name: w for w in configs.ALL if w.name not in ws})
    ws.update(configs.ONE_LAYER)
    ws.update({INPUT + n: ws[n] for n in INPUT_FUSION})
    ws.update(configs.FP8)
    return ws


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--only", nargs="*")
    ap.add_argument("--seeds", type=int, default=2)
    ap.add_argument("--out", default=parity_plan.CAPS_FILE)
    ap.add_argument("--merge", nargs="*")
    args = ap.parse_args()
    if args.merge:
        out = parity_plan.load_caps()
        for f in args.merge:
            with open(f) as fh:
                out["workloads"].update(json.load(fh)["workloads"])
        with open(parity_plan.CAPS_FILE, "w") as fh:
            json.dump(out, fh, indent=1, sort_keys=True)
        return
    ws = all_workloads()
    names = args.only or list(ws)
    out = {}
    if os.path.exists(args.out):
        with open(args.out) as fh:
            out = json.load(fh)
    out.setdefault("workloads", {})
    out["method"] = ("max |z_perturbed - z| of the fp64 oracle, pre-rounding values scaled "
                     "by 1 + rel*N(0,1), rel in %s, %d seed(s) at 1e-7" % (list(RELS), args.seeds))
    out["cap_factor"] = parity_plan.CAP_FACTOR
    for name in names:
        t0 = time.time()
        variant = "input" if name.startswith(INPUT) else "kv"
        out["workloads"][name] = study(ws[name], args.seeds, variant)
        out["workloads"][name]["seconds"] = round(time.time() - t0, 1)
        print(name, out["workloads"][name]["worst_logit_change"],
              f"{time.time() - t0:.0f}s", flush=True)
        with open(args.out, "w") as f:
            json.dump(out, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main()
