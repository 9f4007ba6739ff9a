"""The greedy speculative loop on the GPU: a DFlash drafter and a random causal target
transformer, every step one dflash_spec_step call (draft -> target pass -> verify ->
commit -> inject), so a run of steps is a chain of device work with no host
synchronisation in between (``capture()`` records one step in a CUDA graph).

SpecRunner owns the device state of a SpecWorkload: the two handles (the drafter's
embedding and LM head are the target's tensors), both paged caches, one page table,
the prompt, the loop state and the planted-agreement uniforms.  ``prefill()`` runs the
target causally over the prompt (all but its last token, in block_size chunks) and
injects the tap features of every chunk into the drafter's cache.
"""
from __future__ import annotations

import ctypes

import torch

from workload import inputs
from workload.configs import SpecWorkload

from . import Drafter, KVCache, SpecState, _check, _ptr, _stream, last_launch_count
from .runner import drafter_config


class SpecRunner:
    def __init__(self, sw: SpecWorkload, device="cuda", plant=True):
        self.sw = sw
        w, wt = sw.drafter, sw.target
        self.device = device
        dt = inputs.torch_dtype(w)
        B, S = w.batch, w.block_size
        self.tw = inputs.target_weights(sw, device)
        self.dw = inputs.loop_drafter_weights(sw, self.tw, device)
        dcfg = drafter_config(w)
        dcfg["max_position"] = sw.max_position
        tcfg = drafter_config(wt)
        tcfg["max_position"] = sw.max_position
        self.drafter = Drafter(dcfg, self.dw)
        self.target = Drafter(tcfg, self.tw)
        self.max_pages = -(-sw.max_position // 16)
        npg = B * self.max_pages
        self.table = (torch.arange(B, dtype=torch.int32)[:, None] * self.max_pages
                      + torch.arange(self.max_pages, dtype=torch.int32)[None, :]).to(device)
        self.dcache = KVCache(w.n_layers, npg, w.n_kv_heads, w.head_dim, dt, device)
        self.tcache = KVCache(wt.n_layers, npg, wt.n_kv_heads, wt.head_dim, dt, device)
        self.dws = self.drafter.workspace(B * S, B, self.max_pages, device)
        self.tws = self.target.workspace(B * S, B, self.max_pages, device)
        lib = self.drafter.lib
        n = ctypes.c_size_t()
        _check(lib.dflash_spec_workspace_size(self.drafter.h, self.target.h, B, self.max_pages,
                                              ctypes.byref(n)))
        self.ws = torch.empty(n.value, dtype=torch.uint8, device=device)
        _check(lib.dflash_spec_workspace_init(self.drafter.h, self.target.h, B, self.max_pages,
                                              _ptr(self.ws), self.ws.numel(), _stream()))
        self.prompt = inputs.prompt_tokens(sw)
        self.block_ids = torch.full((B, S), w.mask_id, dtype=torch.int32)
        self.block_ids[:, 0] = self.prompt[:, -1].to(torch.int32)
        self.block_ids = self.block_ids.to(device)
        self.ctx_lens = torch.full((B,), sw.prompt_len - 1, dtype=torch.int32, device=device)
        self.max_new = (sw.steps + 1) * S
        self.generated = torch.full((B, self.max_new), -1, dtype=torch.int32, device=device)
        self.n_generated = torch.zeros(B, dtype=torch.int32, device=device)
        self.n_emitted = torch.zeros(B, dtype=torch.int32, device=device)
        self.drafts = torch.zeros(B, S, dtype=torch.int32, device=device)
        self.step_ctr = torch.zeros(1, dtype=torch.int32, device=device)
        self.plant_u = inputs.loop_uniforms(sw, device) if plant else None
        self._taps = (ctypes.c_int32 * len(sw.tap_layers))(*sw.tap_layers)
        self.state = SpecState(
            batch=B, block_ids=_ptr(self.block_ids), ctx_lens=_ptr(self.ctx_lens),
            page_table=_ptr(self.table), max_pages=self.max_pages, num_pages=npg,
            d_k_pool=self.dcache._kp, d_v_pool=self.dcache._vp,
            t_k_pool=self.tcache._kp, t_v_pool=self.tcache._vp,
            tap_layers=ctypes.cast(self._taps, ctypes.c_void_p), mask_id=w.mask_id,
            generated=_ptr(self.generated), max_new=self.max_new,
            n_generated=_ptr(self.n_generated), n_emitted=_ptr(self.n_emitted),
            drafts=_ptr(self.drafts), step=_ptr(self.step_ctr),
            plant_u=_ptr(self.plant_u), plant_steps=sw.steps if plant else 0,
            plant_p=sw.plant_p if plant else 0.0)
        self.launches = 0
        self.graph = None

    # ------------------------------------------------------------------ setup
    def prefill(self):
        """Both caches take the prompt but its last token: the target runs causally over
        it in block_size chunks (the last chunk padded with mask ids, whose cache rows
        lie past the context and are overwritten by the first step), and each chunk's
        tap features are injected into the drafter's cache."""
        sw, w = self.sw, self.sw.drafter
        B, S, T = w.batch, w.block_size, sw.prompt_len - 1
        taps = torch.empty(B * S, w.fuse_in, dtype=inputs.torch_dtype(w), device=self.device)
        prompt = self.prompt.to(torch.int32)
        for c0 in range(0, T, S):
            ids = torch.full((B, S), w.mask_id, dtype=torch.int32)
            n = min(S, T - c0)
            ids[:, :n] = prompt[:, c0:c0 + n]
            ctx = torch.full((B,), c0, dtype=torch.int32, device=self.device)
            self.target.target_forward(ids.to(self.device), ctx, self.table, self.tcache,
                                       self.tws, sw.tap_layers, taps)
            pos = (c0 + torch.arange(S, dtype=torch.int32)).repeat(B)
            slots = (self.table.cpu().to(torch.int64)[torch.arange(B).repeat_interleave(S),
                                                      pos.to(torch.int64) // 16] * 16
                     + pos.to(torch.int64) % 16).to(torch.int32)
            self.drafter.inject_kv(pos.to(self.device), slots.to(self.device), self.dcache,
                                   self.dws, x_cat=taps)

    # ------------------------------------------------------------------ the loop
    def step(self):
        _check(self.drafter.lib.dflash_spec_step(self.drafter.h, self.target.h,
                                                 ctypes.byref(self.state), _ptr(self.ws),
                                                 self.ws.numel(), _stream()))
        self.launches = last_launch_count()

    def capture(self):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            self.step()
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()
