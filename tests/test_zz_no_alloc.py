"""The no-allocation greedy verification entry point, through the C ABI.

dflash_verify_greedy_static exists for callers that cannot call cudaMalloc where they
verify (a host runtime that only owns fixed buffers, an allocator frozen under a memory
budget, a plain C caller without an allocator): it keeps its scratch in a fixed device
array inside the library.  This checks it against dflash_verify_greedy (which takes a
caller workspace) on two calls in a row; the outputs are integers, so they must match
exactly.  Kept in its own file so that it runs after every other test.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _inputs(S, V, B=7, seed=11):
    g = torch.Generator().manual_seed(seed)
    logits = (torch.randint(0, 7, (B, S, V), generator=g).float() - 3).to(torch.bfloat16)
    draft = logits.float().argmax(-1)
    draft[1, 0] = (draft[1, 0] + 1) % V
    draft[3, 9] = (draft[3, 9] + 5) % V
    draft[5] = torch.randint(0, V, (S,), generator=g)
    return draft.to(torch.int32), logits


def test_static_scratch_verify_matches_workspace_verify():
    import block_diffusion_drafter_concat_gb300 as pkg
    from block_diffusion_drafter_concat_gb300 import build
    from block_diffusion_drafter_concat_gb300.runner import StepRunner
    from workload import configs

    build.build()
    lib = pkg.load()
    r = StepRunner(configs.small_bf16(), prefill=False)
    S, V = r.w.block_size, r.w.vocab
    draft, logits = _inputs(S, V)
    B = draft.shape[0]
    d, lg = draft.cuda(), logits.cuda()
    ref = [torch.empty(B, S, dtype=torch.int32, device="cuda"),
           torch.empty(B, dtype=torch.int32, device="cuda"),
           torch.empty(B, dtype=torch.int32, device="cuda")]
    r.drafter.verify_greedy(d, lg, *ref, r.ws)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = [torch.full((B, S), -7, dtype=torch.int32, device="cuda"),
               torch.full((B,), -7, dtype=torch.int32, device="cuda"),
               torch.full((B,), -7, dtype=torch.int32, device="cuda")]
        st = lib.dflash_verify_greedy_static(r.drafter.h, ctypes.c_void_p(d.data_ptr()),
                                             ctypes.c_void_p(lg.data_ptr()), B,
                                             *[ctypes.c_void_p(t.data_ptr()) for t in out],
                                             stream)
        assert st == pkg.OK, lib.dflash_last_error()
        torch.cuda.synchronize()
        for a, b in zip(out, ref):
            assert torch.equal(a, b), (call, a, b)
    assert int(ref[2][0]) == S and int(ref[2][1]) == 1
    assert r.drafter.device_error() == 0
    # sizes beyond the fixed array are refused with a clear message
    big = 16384 // S + 1
    st = lib.dflash_verify_greedy_static(r.drafter.h, ctypes.c_void_p(d.data_ptr()),
                                         ctypes.c_void_p(lg.data_ptr()), big,
                                         *[ctypes.c_void_p(t.data_ptr()) for t in out], stream)
    assert st == pkg.EUNSUPPORTED
    assert b"static scratch" in lib.dflash_last_error()
