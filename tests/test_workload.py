"""Synthetic input generator and workload helpers (CPU)."""
import ast
import os

import numpy as np
import torch

from workload import configs, inputs, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_hash_matches_python_integer_reference():
    idx = [0, 1, 2, 3, 2 ** 31 - 1, 2 ** 31, 2 ** 33 + 5, 12345678901, 2 ** 62 + 3]
    h = synth.hash_at(7, "w_fuse", torch.tensor(idx, dtype=torch.int64))
    key = synth.stream_key(7, "w_fuse")
    ref = [synth._s64(synth.mix64_int(key + i * synth.GOLDEN)) for i in idx]
    assert h.tolist() == ref


def test_splitmix64_known_value():
    # SplitMix64 with state 0: first output is mix64(0 + golden) = 0xE220A8397B1DCDAF
    assert synth.mix64_int(synth.GOLDEN) == 0xE220A8397B1DCDAF


def test_normal_stream_statistics_and_slicing():
    x = synth.normal(3, "t", (1000, 300), std=2.0)
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 2.0) < 0.02
    part = synth.normal(3, "t", (1000, 300), std=2.0, rows=(500, 503))
    assert torch.equal(part, x[500:503])
    g = synth.normal(3, "g", (4096,), std=0.02, mean=1.0, dtype=torch.bfloat16)
    assert abs(float(g.float().mean()) - 1.0) < 2e-3
    assert not torch.equal(synth.normal(3, "a", (64,)), synth.normal(3, "b", (64,)))


def test_uniform_and_integers_ranges():
    u = synth.uniform(4, "uniforms", (64, 16, 2))
    assert float(u.min()) >= 0.0 and float(u.max()) < 1.0 and abs(float(u.mean()) - 0.5) < 0.01
    n = synth.integers(2, "ctx_len", (5000,), 512, 4096)
    assert int(n.min()) >= 512 and int(n.max()) <= 4096
    p = synth.permutation(2, "pages", 1000)
    assert sorted(p.tolist()) == list(range(1000))


def test_page_table_covers_each_context_once():
    w = configs.small_bf16()
    lens = inputs.ctx_lens(w)
    table, total = inputs.page_table(w, lens)
    used = []
    for b, t in enumerate(lens.tolist()):
        npg = -(-t // w.page_size)
        used += table[b, :npg].tolist()
        assert (table[b, npg:] == -1).all()
    assert sorted(used) == list(range(total))


def test_planting_makes_the_draft_the_strict_row_maximum():
    w = configs.QWEN3_8B_B1.scaled(vocab=4096)
    z = inputs.logits_noise(w)
    d = torch.randint(0, w.vocab, (1, w.block_size))
    mask = inputs.plant_mask(w)
    inputs.plant(w, z, d, mask)
    for i in range(w.block_size):
        row = z[0, i].float()
        if mask[0, i]:
            top = row[d[0, i]]
            others = torch.cat([row[:d[0, i]], row[d[0, i] + 1:]])
            assert float(top) > float(others.max())


def test_oracle_is_independent_of_torch_and_the_cuda_package():
    src = open(os.path.join(ROOT, "oracle", "dflash_oracle.py")).read()
    mods = set()
    for node in ast.walk(ast.parse(src)):
        if isinstance(node, ast.Import):
            mods |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom):
            mods.add((node.module or "").split(".")[0])
    assert mods <= {"__future__", "numpy"}, mods


def test_configs_match_the_named_workloads():
    c = configs.BY_NAME
    assert c["tiny-f32"].fuse_in == 768 and c["tiny-f32"].dtype == "f32"
    q = c["qwen3-8b-shaped-b1"]
    assert (q.fuse_in, q.n_layers, q.vocab, q.block_size, q.ctx_len) == (20480, 5, 151936, 16, 2048)
    g = c["gpt-oss-120b-shaped-b64-t1"]
    assert (g.d_model, g.q_width, g.temperature, g.batch, g.ctx_len) == (2880, 4096, 1.0, 64, 16384)
    assert np.isclose((1 - 0.8 ** 16) / (1 - 0.8), 4.859, atol=1e-3)
