"""The stored logit-slack caps (tests/golden/slack_caps.json) against the oracle-only
study that writes them (tests/golden/make_slack_caps.py): every workload the GPU parity
tests compare has a cap, the stored figures of small workloads are reproduced exactly,
the caps were measured on the sequences the GPU tests sample, and the study measures
what it claims (no change without perturbation, a change that saturates rather than
grows with the perturbation)."""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden"))

import make_slack_caps as M  # noqa: E402
import parity_plan  # noqa: E402
from oracle import run as orun  # noqa: E402
from workload import configs, inputs  # noqa: E402


def test_every_parity_workload_has_a_cap():
    caps = parity_plan.load_caps()["workloads"]
    for name in M.all_workloads():
        assert name in caps, name
        assert caps[name]["worst_logit_change"] > 0.0, name


@pytest.mark.parametrize("name", ["small-bf16-b1", "small-bf16-hd64-g8", "tiny-f32"])
def test_stored_caps_are_reproduced(name):
    stored = parity_plan.load_caps()["workloads"][name]
    again = M.study(M.all_workloads()[name], seeds=2)
    assert again["worst_logit_change"] == pytest.approx(stored["worst_logit_change"], rel=1e-9)


def test_caps_cover_the_sampled_sequences():
    """Each large workload's cap was measured on sequences the GPU tests compare,
    including the shortest and the longest context of their sample."""
    caps = parity_plan.load_caps()["workloads"]
    for w in list(configs.ALL[1:]) + list(configs.ONE_LAYER.values()):
        lens = inputs.ctx_lens(w).numpy()
        sample = parity_plan.sampled_sequences(lens)
        have = {int(b) for b in caps[w.name]["sequences"]}
        assert have == set(M.sequences_of(w)) and have <= set(sample), w.name
        assert {min(sample, key=lambda b: (lens[b], b)),
                max(sample, key=lambda b: (lens[b], b))} <= have, w.name


def test_unperturbed_run_changes_nothing():
    w = configs.PARITY_SMALL["small-bf16-b1"]
    W = orun.host_weights(w)
    base = orun.draft_sequence(w, W, 0)
    same = M.perturbed_run(w, W, 0, 0.0, 1)
    assert np.array_equal(same["z"], base["z"])


def test_logit_change_saturates_with_the_perturbation():
    """Sub-ulp perturbations flip rounding decisions; the resulting logit change is of
    the same size for relative perturbations 100x apart, which is why a fixed cap holds
    whatever the exact size of the fp32 evaluation error."""
    w = configs.PARITY_SMALL["small-bf16-b1"]
    W = orun.host_weights(w)
    base = orun.draft_sequence(w, W, 0)
    ch = [np.abs(M.perturbed_run(w, W, 0, rel, 7)["z"] - base["z"]).max()
          for rel in (1e-7, 1e-5)]
    assert 0.0 < ch[0] and ch[1] < 2.0 * ch[0], ch
    assert ch[1] < parity_plan.CAP_FACTOR * parity_plan.load_caps()["workloads"][
        "small-bf16-b1"]["worst_logit_change"] * 2
