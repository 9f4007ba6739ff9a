"""C-ABI library: builds for sm_103a, loads without a GPU, exports every declared entry
point, and rejects bad host arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


@pytest.fixture(scope="module")
def lib():
    from block_diffusion_drafter_concat_gb300 import build, load
    build.build()
    return load()


def declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"DFLASH_API\s+[\w\s\*]+?\b(dflash_\w+)\s*\(", src)))


def test_header_declares_the_path_entry_points():
    names = declared()
    for n in ("dflash_fuse_features", "dflash_inject_kv", "dflash_draft_block",
              "dflash_lm_head_argmax", "dflash_verify_greedy", "dflash_verify_sample"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    import block_diffusion_drafter_concat_gb300 as pkg
    assert sorted(pkg.API) == declared()


def test_null_arguments_are_rejected_on_the_host(lib):
    import block_diffusion_drafter_concat_gb300 as pkg
    assert lib.dflash_create(None, None, None) == pkg.EINVAL
    assert lib.dflash_fuse_features(None, None, 1, None, None, 0, None) == pkg.EINVAL
    assert lib.dflash_verify_greedy(None, None, None, 1, None, None, None, None, 0, None) == pkg.EINVAL
    assert b"null" in lib.dflash_last_error()
    assert lib.dflash_destroy(None) == pkg.EINVAL
    n = ctypes.c_size_t()
    assert lib.dflash_workspace_size(None, 1, 1, 1, ctypes.byref(n)) == pkg.EINVAL


def test_config_validation_happens_before_any_device_call(lib):
    import block_diffusion_drafter_concat_gb300 as pkg
    from block_diffusion_drafter_concat_gb300.runner import drafter_config
    from workload import configs
    cfg = drafter_config(configs.QWEN3_8B_B1)
    w = pkg.Weights()
    h = ctypes.c_void_p()
    bad = dict(cfg, page_size=8)
    c = pkg.Config(**{k: bad[k] for k, _ in pkg.Config._fields_})
    assert lib.dflash_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h)) == pkg.EUNSUPPORTED
    bad = dict(cfg, head_dim=96)
    c = pkg.Config(**{k: bad[k] for k, _ in pkg.Config._fields_})
    assert lib.dflash_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h)) == pkg.EUNSUPPORTED
    bad = dict(cfg, d_model=0)
    c = pkg.Config(**{k: bad[k] for k, _ in pkg.Config._fields_})
    assert lib.dflash_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h)) == pkg.EINVAL
    # a valid shape with null weight arrays is rejected before any CUDA call
    c = pkg.Config(**{k: cfg[k] for k, _ in pkg.Config._fields_})
    assert lib.dflash_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(h)) == pkg.EINVAL
    assert not h.value


def test_missing_library_fails_loudly(tmp_path):
    import block_diffusion_drafter_concat_gb300 as pkg
    with pytest.raises(RuntimeError):
        pkg._lib_saved = pkg._lib
        pkg._lib = None
        try:
            pkg.load(str(tmp_path / "nope.so"))
        finally:
            pkg._lib = pkg._lib_saved
