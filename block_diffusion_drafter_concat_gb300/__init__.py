"""Python binding of libdflash (ctypes): argument marshalling only.

Every step of the DFlash draft + verify path runs in the library's CUDA kernels; this
module turns torch tensors into device pointers and the current torch stream into a
cudaStream_t.  It never computes any part of the method and has no CPU fallback: a
missing library raises at load time.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdflash.so")

OK, EINVAL, EUNSUPPORTED, EWORKSPACE, ECUDA, EDEVICE = range(6)
F32, BF16 = 0, 1
DEV_ERRORS = {0: "ok", 1: "index out of range", 2: "position out of range", 3: "wait timeout"}

API = ["dflash_create", "dflash_destroy", "dflash_workspace_size", "dflash_workspace_init",
       "dflash_fuse_features", "dflash_inject_kv", "dflash_draft_block",
       "dflash_inject_draft", "dflash_inject_inputs", "dflash_target_forward", "dflash_spec_workspace_size",
       "dflash_spec_workspace_init", "dflash_spec_step",
       "dflash_lm_head_argmax", "dflash_verify_greedy", "dflash_verify_sample",
       "dflash_verify_greedy_static", "dflash_test_force_timeout", "dflash_fp8_packed_bytes",
       "dflash_pack_fp8",
       "dflash_get_device_error", "dflash_last_error", "dflash_last_launch_count"]


class DFlashError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"libdflash status {status}: {msg}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "d_model", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "ffn_dim", "vocab",
        "block_size", "n_target_layers", "target_width", "page_size", "max_position")] + [
        ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float), ("dtype", ctypes.c_int32),
        ("weight_format", ctypes.c_int32)]


_P = ctypes.c_void_p
_PP = ctypes.POINTER(ctypes.c_void_p)


class Weights(ctypes.Structure):
    _fields_ = [("w_fuse", _P), ("g_fuse", _P)] + [(n, _PP) for n in (
        "g_attn", "w_q", "w_k", "w_v", "w_o", "g_mlp", "w_gate", "w_up", "w_down")] + [
        ("g_final", _P), ("embed", _P), ("lm_head", _P)]


class SpecState(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("block_ids", _P), ("ctx_lens", _P),
                ("page_table", _P), ("max_pages", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("d_k_pool", _PP), ("d_v_pool", _PP), ("t_k_pool", _PP), ("t_v_pool", _PP),
                ("tap_layers", _P), ("mask_id", ctypes.c_int32), ("generated", _P),
                ("max_new", ctypes.c_int32), ("n_generated", _P), ("n_emitted", _P), ("drafts", _P),
                ("step", _P), ("plant_u", _P), ("plant_steps", ctypes.c_int32),
                ("plant_p", ctypes.c_float)]


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libdflash.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "block_diffusion_drafter_concat_gb300.build.build()")
    lib = ctypes.CDLL(path)
    i32, sz = ctypes.c_int32, ctypes.c_size_t
    P, PP = _P, _PP
    sig = {
        "dflash_create": [ctypes.POINTER(Config), ctypes.POINTER(Weights), ctypes.POINTER(P)],
        "dflash_destroy": [P],
        "dflash_workspace_size": [P, i32, i32, i32, ctypes.POINTER(sz)],
        "dflash_workspace_init": [P, P, sz, P],
        "dflash_fuse_features": [P, P, i32, P, P, sz, P],
        "dflash_inject_kv": [P, P, P, i32, P, P, i32, PP, PP, P, P, sz, P],
        "dflash_draft_block": [P, P, P, P, i32, i32, i32, PP, PP, P, P, sz, P],
        "dflash_inject_inputs": [P, P, P, P, i32, i32, i32, PP, PP, P, P, sz, P],
        "dflash_inject_draft": [P, P, i32, P, P, P, P, P, i32, i32, i32, PP, PP, P, P, P, sz, P],
        "dflash_spec_workspace_size": [P, P, i32, i32, ctypes.POINTER(sz)],
        "dflash_spec_workspace_init": [P, P, i32, i32, P, sz, P],
        "dflash_spec_step": [P, P, ctypes.POINTER(SpecState), P, sz, P],
        "dflash_target_forward": [P, P, P, P, i32, i32, i32, PP, PP, P, i32, P, P, P, sz, P],
        "dflash_lm_head_argmax": [P, P, i32, ctypes.c_float, P, P, P, P, sz, P],
        "dflash_verify_greedy": [P, P, P, i32, P, P, P, P, sz, P],
        "dflash_verify_sample": [P, P, P, P, P, P, P, ctypes.c_float, i32, P, P, P, P, sz, P],
        "dflash_verify_greedy_static": [P, P, P, i32, P, P, P, P],
        "dflash_test_force_timeout": [P, i32],
        "dflash_fp8_packed_bytes": [i32, i32, ctypes.POINTER(sz)],
        "dflash_pack_fp8": [P, i32, i32, P, P],
        "dflash_get_device_error": [P, ctypes.POINTER(i32), i32],
        "dflash_last_error": [],
        "dflash_last_launch_count": [],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int32
    lib.dflash_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status):
    if status != OK:
        raise DFlashError(status, load().dflash_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _ptr_array(ts: Sequence[torch.Tensor]):
    arr = (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    return ctypes.cast(arr, _PP), arr


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def pack_fp8(w: torch.Tensor) -> torch.Tensor:
    """The packed FP8 form of a bf16 [rows, cols] CUDA matrix (dflash_pack_fp8), as a
    uint8 CUDA tensor."""
    lib = load()
    rows, cols = w.shape
    n = ctypes.c_size_t()
    _check(lib.dflash_fp8_packed_bytes(rows, cols, ctypes.byref(n)))
    out = torch.empty(n.value, dtype=torch.uint8, device=w.device)
    _check(lib.dflash_pack_fp8(_ptr(w.contiguous()), rows, cols, _ptr(out), _stream()))
    return out


def unpack_fp8(packed: torch.Tensor, rows: int, cols: int):
    """(codes [rows, cols] uint8, scales [rows] fp32) views of a packed FP8 matrix."""
    ld = (cols + 15) // 16 * 16
    off = (rows * ld + 255) // 256 * 256
    codes = packed[:rows * ld].view(rows, ld)[:, :cols]
    scales = packed[off:off + 4 * rows].view(torch.float32)
    return codes, scales


def last_launch_count() -> int:
    return int(load().dflash_last_launch_count())


class KVCache:
    """Per-layer paged K and V pools, each [num_pages, n_kv_heads, 16, head_dim]."""

    def __init__(self, n_layers, num_pages, n_kv_heads, head_dim, dtype, device="cuda"):
        shape = (num_pages, n_kv_heads, 16, head_dim)
        self.num_pages = num_pages
        self.k = [torch.zeros(shape, dtype=dtype, device=device) for _ in range(n_layers)]
        self.v = [torch.zeros(shape, dtype=dtype, device=device) for _ in range(n_layers)]
        self._kp, self._ka = _ptr_array(self.k)
        self._vp, self._va = _ptr_array(self.v)


class Drafter:
    """A libdflash handle over borrowed device weights (kept alive here).

    ``weights`` maps the names w_fuse, g_fuse, l{l}.g_attn, l{l}.w_q, l{l}.w_k,
    l{l}.w_v, l{l}.w_o, l{l}.g_mlp, l{l}.w_gate, l{l}.w_up, l{l}.w_down, g_final, embed,
    lm_head to contiguous CUDA tensors of the config dtype (without w_fuse and g_fuse:
    a plain transformer, e.g. the target of the speculative loop)."""

    LAYER = ("g_attn", "w_q", "w_k", "w_v", "w_o", "g_mlp", "w_gate", "w_up", "w_down")

    def __init__(self, cfg: dict, weights: dict):
        lib = load()
        self.cfg = dict(cfg)
        self.dtype = torch.bfloat16 if cfg["dtype"] == BF16 else torch.float32
        self.c = Config(**{k: cfg.get(k, 0) for k, _ in Config._fields_})
        self._w = weights
        self._arrays = {}
        fields = {}
        for name in self.LAYER:
            ts = [weights[f"l{l}.{name}"] for l in range(cfg["n_layers"])]
            fields[name], self._arrays[name] = _ptr_array(ts)
        for name in ("w_fuse", "g_fuse", "g_final", "embed", "lm_head"):
            fields[name] = _ptr(weights.get(name))
        self.w = Weights(**fields)
        h = ctypes.c_void_p()
        _check(lib.dflash_create(ctypes.byref(self.c), ctypes.byref(self.w), ctypes.byref(h)))
        self.h = h
        self.lib = lib

    def close(self):
        if self.h:
            _check(self.lib.dflash_destroy(self.h))
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---------------------------------------------------------------- workspace
    def workspace_size(self, max_rows, max_batch, max_pages) -> int:
        n = ctypes.c_size_t()
        _check(self.lib.dflash_workspace_size(self.h, max_rows, max_batch, max_pages,
                                              ctypes.byref(n)))
        return n.value

    def workspace(self, max_rows, max_batch, max_pages, device="cuda"):
        ws = torch.empty(self.workspace_size(max_rows, max_batch, max_pages), dtype=torch.uint8,
                         device=device)
        self.workspace_init(ws)
        return ws

    def workspace_init(self, ws):
        _check(self.lib.dflash_workspace_init(self.h, _ptr(ws), ws.numel(), _stream()))

    # ---------------------------------------------------------------- the path
    def fuse_features(self, x_cat, fused, ws):
        _check(self.lib.dflash_fuse_features(self.h, _ptr(x_cat), x_cat.shape[0], _ptr(fused),
                                             _ptr(ws), ws.numel(), _stream()))
        return fused

    def inject_kv(self, positions, slots, cache: KVCache, ws, x_cat=None, fused=None,
                  fused_out=None):
        n = (x_cat if x_cat is not None else fused).shape[0]
        _check(self.lib.dflash_inject_kv(self.h, _ptr(x_cat), _ptr(fused), n, _ptr(positions),
                                         _ptr(slots), cache.num_pages, cache._kp, cache._vp,
                                         _ptr(fused_out), _ptr(ws), ws.numel(), _stream()))

    def draft_block(self, block_ids, ctx_lens, page_table, cache: KVCache, final_hidden, ws):
        _check(self.lib.dflash_draft_block(
            self.h, _ptr(block_ids), _ptr(ctx_lens), _ptr(page_table), page_table.shape[1],
            block_ids.shape[0], cache.num_pages, cache._kp, cache._vp, _ptr(final_hidden),
            _ptr(ws), ws.numel(), _stream()))
        return final_hidden

    def inject_draft(self, x_cat, positions, slots, block_ids, ctx_lens, page_table,
                     cache: KVCache, final_hidden, ws, fused_out=None):
        _check(self.lib.dflash_inject_draft(
            self.h, _ptr(x_cat), x_cat.shape[0], _ptr(positions), _ptr(slots), _ptr(block_ids),
            _ptr(ctx_lens), _ptr(page_table), page_table.shape[1], block_ids.shape[0],
            cache.num_pages, cache._kp, cache._vp, _ptr(fused_out), _ptr(final_hidden),
            _ptr(ws), ws.numel(), _stream()))
        return final_hidden

    def inject_inputs(self, x_cat, ctx_lens, page_table, cache: KVCache, ws, fused_out=None):
        _check(self.lib.dflash_inject_inputs(
            self.h, _ptr(x_cat), _ptr(ctx_lens), _ptr(page_table), page_table.shape[1],
            ctx_lens.shape[0], cache.num_pages, cache._kp, cache._vp, _ptr(fused_out), _ptr(ws),
            ws.numel(), _stream()))

    def target_forward(self, ids, ctx_lens, page_table, cache: KVCache, ws, tap_layers=(),
                       taps=None, logits=None):
        n = len(tap_layers)
        arr = (ctypes.c_int32 * max(1, n))(*tap_layers)
        _check(self.lib.dflash_target_forward(
            self.h, _ptr(ids), _ptr(ctx_lens), _ptr(page_table), page_table.shape[1],
            ids.shape[0], cache.num_pages, cache._kp, cache._vp,
            ctypes.cast(arr, ctypes.c_void_p) if n else None, n, _ptr(taps), _ptr(logits),
            _ptr(ws), ws.numel(), _stream()))

    def lm_head_argmax(self, hidden, tokens, ws, max_logit=None, lse=None, temperature=1.0):
        _check(self.lib.dflash_lm_head_argmax(self.h, _ptr(hidden), hidden.shape[0],
                                              float(temperature), _ptr(tokens), _ptr(max_logit),
                                              _ptr(lse), _ptr(ws), ws.numel(), _stream()))
        return tokens

    def verify_greedy(self, draft, target_logits, out_tokens, n_accepted, n_emitted, ws):
        _check(self.lib.dflash_verify_greedy(self.h, _ptr(draft), _ptr(target_logits),
                                             draft.shape[0], _ptr(out_tokens), _ptr(n_accepted),
                                             _ptr(n_emitted), _ptr(ws), ws.numel(), _stream()))

    def verify_sample(self, draft, hidden, draft_max, draft_lse, target_logits, uniforms,
                      temperature, out_tokens, n_accepted, n_emitted, ws):
        _check(self.lib.dflash_verify_sample(
            self.h, _ptr(draft), _ptr(hidden), _ptr(draft_max), _ptr(draft_lse),
            _ptr(target_logits), _ptr(uniforms), float(temperature), draft.shape[0],
            _ptr(out_tokens), _ptr(n_accepted), _ptr(n_emitted), _ptr(ws), ws.numel(),
            _stream()))

    def test_force_timeout(self, enable: bool):
        _check(self.lib.dflash_test_force_timeout(self.h, int(bool(enable))))

    def device_error(self, clear=True) -> int:
        code = ctypes.c_int32()
        _check(self.lib.dflash_get_device_error(self.h, ctypes.byref(code), int(clear)))
        return code.value
