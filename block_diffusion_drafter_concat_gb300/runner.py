"""One DFlash draft + verify step on a seeded synthetic workload, end to end on the GPU.

StepRunner owns the device state of a workload: random-init weights of the named
shape, the paged KV cache, the page table, the per-step inputs (the S newest target
hidden features of every sequence and the target's verify logits) and the outputs.
``step()`` enqueues the whole path as libdflash calls on the current stream:

  dflash_inject_draft (fuse + inject the S new context rows of every sequence, then the
  drafter's block pass)  -> dflash_lm_head_argmax
  -> dflash_verify_greedy, or dflash_verify_sample at temperature > 0.

``capture()`` records that sequence into a CUDA graph.  Inputs come from the seeded
counter-based generator, drawn directly on the device.
"""
from __future__ import annotations

import torch

from workload import inputs
from workload.configs import Workload

from . import BF16, F32, Drafter, KVCache, last_launch_count, pack_fp8

PREFILL_CHUNK = 4096


FP8_MATRICES = ("w_fuse", "w_q", "w_k", "w_v", "w_o", "w_gate", "w_up", "w_down", "lm_head")


def drafter_config(w: Workload) -> dict:
    return dict(d_model=w.d_model, n_layers=w.n_layers, n_q_heads=w.n_q_heads,
                n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, ffn_dim=w.ffn_dim,
                vocab=w.vocab, block_size=w.block_size, n_target_layers=w.n_target_layers,
                target_width=w.target_width, page_size=w.page_size,
                max_position=w.max_position, rope_theta=w.rope_theta, rms_eps=w.rms_eps,
                dtype=BF16 if w.dtype == "bf16" else F32,
                weight_format=1 if w.weight_format == "fp8" else 0)


def packed_weights(weights: dict) -> dict:
    """Projection matrices replaced by their packed FP8 form (dflash_pack_fp8, on the
    device); embedding and gains unchanged."""
    return {n: pack_fp8(t) if n.split(".")[-1] in FP8_MATRICES else t
            for n, t in weights.items()}


class StepRunner:
    """variant "kv": the DFlash step (context features injected into every layer's K/V);
    "input": the input-fusion variant (the S new context rows run through the layer
    stack as input, dflash_inject_inputs, before the block is drafted)."""

    def __init__(self, w: Workload, device="cuda", prefill=True, weights=None, variant="kv"):
        assert variant in ("kv", "input")
        self.variant = variant
        self.w = w
        self.device = device
        self.dt = inputs.torch_dtype(w)
        S, B = w.block_size, w.batch
        self.weights = weights if weights is not None else inputs.weights(w, device)
        if w.weight_format == "fp8":
            self.weights = packed_weights(self.weights)
        self.drafter = Drafter(drafter_config(w), self.weights)
        self.lens = inputs.ctx_lens(w)
        assert int(self.lens.min()) >= S, "each context must hold at least one block"
        table, total = inputs.page_table(w, self.lens)
        self.table_host = table
        self.page_table = table.to(device)
        self.cache = KVCache(w.n_layers, total, w.n_kv_heads, w.head_dim, self.dt, device)
        self.ws = self.drafter.workspace(max(w.rows, PREFILL_CHUNK), B, w.max_pages, device)
        # step inputs: the S newest context rows of every sequence
        pos, slots = [], []
        for b in range(B):
            t = int(self.lens[b])
            p = torch.arange(t - S, t)
            pos.append(p)
            slots.append(inputs.slots_for(w, table, b, p))
        self.positions = torch.cat(pos).to(torch.int32).to(device)
        self.slots = torch.cat(slots).to(torch.int32).to(device)
        self.x_step = torch.cat([inputs.ctx_hidden(w, b, int(self.lens[b]) - S, int(self.lens[b]),
                                                   device) for b in range(B)])
        self.block_ids = inputs.block_ids(w).to(device)
        self.ctx_lens = self.lens.to(torch.int32).to(device)
        self.ctx_before = (self.lens - S).to(torch.int32).to(device)
        M, d = w.rows, w.d_model
        self.fused = torch.empty(M, d, dtype=self.dt, device=device)
        self.hidden = torch.empty(M, d, dtype=self.dt, device=device)
        self.draft = torch.empty(B, S, dtype=torch.int32, device=device)
        self.dmax = torch.empty(M, dtype=torch.float32, device=device)
        self.dlse = torch.empty(M, dtype=torch.float32, device=device)
        self.out_tokens = torch.empty(B, S, dtype=torch.int32, device=device)
        self.n_acc = torch.empty(B, dtype=torch.int32, device=device)
        self.n_emit = torch.empty(B, dtype=torch.int32, device=device)
        self.logits = inputs.logits_noise(w, device=device)
        self.uniforms = inputs.uniforms(w, device=device)
        self.launches = 0
        self.graph = None
        # copy the fused step rows out (parity tests read them; the benchmark does not)
        self.keep_fused = True
        if prefill:
            self.prefill()

    # ------------------------------------------------------------------ setup
    def prefill(self):
        """Injects context positions [0, T_b - S) of every sequence (untimed setup)."""
        w = self.w
        if self.variant == "input":
            return self._prefill_inputs()
        for b in range(w.batch):
            t = int(self.lens[b]) - w.block_size
            for p0 in range(0, t, PREFILL_CHUNK):
                p1 = min(t, p0 + PREFILL_CHUNK)
                x = inputs.ctx_hidden(w, b, p0, p1, self.device)
                p = torch.arange(p0, p1)
                s = inputs.slots_for(w, self.table_host, b, p)
                self.drafter.inject_kv(p.to(torch.int32).to(self.device),
                                       s.to(torch.int32).to(self.device), self.cache, self.ws,
                                       x_cat=x)

    def _prefill_inputs(self):
        """Input fusion: the context runs through the layer stack in causal chunks of S
        rows (identical to one causal pass).  Chunk c0 puts sequence b at position
        min(c0, T_b - S): a sequence whose context is done recomputes its last chunk
        (the same values), so no row leaves its pages."""
        w, S = self.w, self.w.block_size
        lens = [int(t) for t in self.lens]
        x = torch.empty(w.rows, w.fuse_in, dtype=self.dt, device=self.device)
        for c0 in range(0, max(lens) - S, S):
            starts = [min(c0, t - S) for t in lens]
            for b, p0 in enumerate(starts):
                x[b * S:(b + 1) * S] = inputs.ctx_hidden(w, b, p0, p0 + S, self.device)
            ctx = torch.tensor(starts, dtype=torch.int32, device=self.device)
            self.drafter.inject_inputs(x, ctx, self.page_table, self.cache, self.ws)

    def plant(self, drafts, mask=None):
        """Regenerates the verify logits and plants agreement with `drafts` [B, S]."""
        w = self.w
        self.logits = inputs.logits_noise(w, device=self.device)
        mask = inputs.plant_mask(w) if mask is None else mask
        inputs.plant(w, self.logits, torch.as_tensor(drafts).cpu(), mask)

    # ------------------------------------------------------------------ the step
    def step(self):
        w, d = self.w, self.drafter
        n = 0
        if self.variant == "input":
            d.inject_inputs(self.x_step, self.ctx_before, self.page_table, self.cache, self.ws,
                            fused_out=self.fused)
            n += last_launch_count()
            d.draft_block(self.block_ids, self.ctx_lens, self.page_table, self.cache,
                          self.hidden, self.ws)
        else:
            # injection and draft in one call (W_k / W_v read once where the rows fit one
            # weight-streaming tile)
            d.inject_draft(self.x_step, self.positions, self.slots, self.block_ids,
                           self.ctx_lens, self.page_table, self.cache, self.hidden, self.ws,
                           fused_out=self.fused if self.keep_fused else None)
        n += last_launch_count()
        sample = w.temperature > 0
        tau = w.temperature if sample else 1.0
        d.lm_head_argmax(self.hidden, self.draft.view(-1), self.ws, self.dmax,
                         self.dlse if sample else None, tau)
        n += last_launch_count()
        if sample:
            d.verify_sample(self.draft, self.hidden, self.dmax, self.dlse, self.logits,
                            self.uniforms, tau, self.out_tokens, self.n_acc, self.n_emit, self.ws)
        else:
            d.verify_greedy(self.draft, self.logits, self.out_tokens, self.n_acc, self.n_emit,
                            self.ws)
        n += last_launch_count()
        self.launches = n

    def timed_calls(self, reps=3):
        """Median device time (us) of each library call of an eager step, each timed
        alone between CUDA events on the current stream."""
        w, d = self.w, self.drafter
        sample = w.temperature > 0
        tau = w.temperature if sample else 1.0
        calls = {
            "inject": (lambda: d.inject_inputs(self.x_step, self.ctx_before, self.page_table,
                                               self.cache, self.ws, fused_out=self.fused))
                      if self.variant == "input" else
                      (lambda: d.inject_kv(self.positions, self.slots, self.cache, self.ws,
                                           x_cat=self.x_step, fused_out=self.fused)),
            "draft_block": lambda: d.draft_block(self.block_ids, self.ctx_lens, self.page_table,
                                                 self.cache, self.hidden, self.ws),
            "inject_draft": lambda: d.inject_draft(self.x_step, self.positions, self.slots,
                                                   self.block_ids, self.ctx_lens,
                                                   self.page_table, self.cache, self.hidden,
                                                   self.ws),
            "lm_head_argmax": lambda: d.lm_head_argmax(self.hidden, self.draft.view(-1), self.ws,
                                                       self.dmax, self.dlse if sample else None,
                                                       tau),
            "verify": (lambda: d.verify_sample(self.draft, self.hidden, self.dmax, self.dlse,
                                               self.logits, self.uniforms, tau, self.out_tokens,
                                               self.n_acc, self.n_emit, self.ws)) if sample else
                      (lambda: d.verify_greedy(self.draft, self.logits, self.out_tokens,
                                               self.n_acc, self.n_emit, self.ws)),
        }
        st = torch.cuda.current_stream()
        out = {}
        for name, fn in calls.items():
            ts = []
            for _ in range(reps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(st)
                fn()
                b.record(st)
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b) * 1e3)
            out[name] = sorted(ts)[len(ts) // 2]
        return out

    def capture(self):
        """Records step() into a CUDA graph (after one eager warm-up step)."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.step()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step()
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()


# ---------------------------------------------------------------------- roofline model
def weight_bytes(w: Workload) -> int:
    """Bytes of every weight one step streams once (the embedding contributes only the
    block's rows).  FP8 projection matrices: one byte per element plus a 4-byte scale
    per row."""
    e = 2 if w.dtype == "bf16" else 4
    d, F = w.d_model, w.ffn_dim
    mats = [(d, w.fuse_in)] + w.n_layers * [(w.q_width, d), (w.kv_width, d), (w.kv_width, d),
                                            (d, w.q_width), (F, d), (F, d), (d, F)] + [(w.vocab, d)]
    if w.weight_format == "fp8":
        proj = sum(r * c + 4 * r for r, c in mats)
    else:
        proj = e * sum(r * c for r, c in mats)
    return proj + e * (d + w.n_layers * 2 * d + d + w.rows * d)


def step_bytes(w: Workload, lens=None) -> int:
    """Algorithmic HBM bytes of one step: weights once, context K/V read once, the S
    new K/V rows written, target hidden features and verify logits read, outputs."""
    e = 2 if w.dtype == "bf16" else 4
    lens = inputs.ctx_lens(w) if lens is None else lens
    kv_row = w.n_layers * 2 * w.kv_width * e
    ctx = int(lens.sum()) * kv_row
    new = w.rows * kv_row
    return (weight_bytes(w) + ctx + new + w.rows * w.fuse_in * e + w.rows * w.vocab * e
            + w.rows * w.d_model * e + w.rows * 4 * 4)


def step_flops(w: Workload, lens=None) -> int:
    lens = inputs.ctx_lens(w) if lens is None else lens
    d, F, R = w.d_model, w.ffn_dim, w.rows
    lin = 2 * R * (d * w.fuse_in + w.n_layers * (2 * w.kv_width * d)
                   + w.n_layers * (w.q_width * d + 2 * w.kv_width * d + d * w.q_width
                                   + 3 * F * d) + w.vocab * d)
    keys = int(lens.sum()) + w.batch * w.block_size
    attn = w.n_layers * 4 * w.block_size * w.n_q_heads * w.head_dim * keys
    return lin + attn


def lm_head_bytes(w: Workload) -> int:
    """Algorithmic bytes of one LM-head launch: the head's weights (FP8: one byte per
    element plus a 4-byte scale per row), the hidden rows, and the per-row token, max and
    log-sum-exp outputs."""
    e = 2 if w.dtype == "bf16" else 4
    head = (w.vocab * w.d_model + 4 * w.vocab) if w.weight_format == "fp8" else e * w.vocab * w.d_model
    return head + e * w.rows * w.d_model + w.rows * 12


def main(argv=None):
    """Runs a few eager steps of a named workload (the command that the ncu captures in
    the profile summaries run):

        python -m block_diffusion_drafter_concat_gb300.runner --workload NAME
               [--layers N] [--steps K]
    """
    import argparse
    import dataclasses

    from workload import configs

    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="qwen3-8b-shaped-b1")
    ap.add_argument("--layers", type=int, default=0, help="drafter layers (0 = the workload's)")
    ap.add_argument("--steps", type=int, default=3)
    a = ap.parse_args(argv)
    w = configs.named(a.workload)
    if a.layers:
        w = dataclasses.replace(w, n_layers=a.layers)
    r = StepRunner(w)
    for _ in range(a.steps):
        r.step()
    torch.cuda.synchronize()
    err = r.drafter.device_error()
    print(f"{w.name} layers={w.n_layers}: {a.steps} steps, {r.launches} launches per step, "
          f"device error {err}")
    if err:
        raise SystemExit(1)


if __name__ == "__main__":
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    main()
