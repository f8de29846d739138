"""Host-side checks of the C ABI (no GPU needed): the library builds, loads,
exports every symbol include/bsattn.h declares, and rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bsattn.h")


@pytest.fixture(scope="module")
def lib():
    from block_sparse_flash_attn_gb300 import _build
    _build.build()
    import block_sparse_flash_attn_gb300 as bs
    return bs.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsattn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ["bsattn_plan", "bsattn_plan_csr", "bsattn_fwd", "bsattn_plan_free",
              "bsattn_status_string"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    import block_sparse_flash_attn_gb300 as bs
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) == set(bs.EXPORTS)


def test_status_strings_and_version(lib):
    import block_sparse_flash_attn_gb300 as bs
    assert lib.bsattn_version() == 100
    for s in range(7):
        assert bs.status_string(s)
    assert bs.status_string(99) == "unknown status"


def test_plan_rejects_bad_arguments_without_a_device(lib):
    import block_sparse_flash_attn_gb300 as bs
    vp = ctypes.c_void_p
    out = vp()
    fake = vp(0x10000)
    assert lib.bsattn_plan(vp(0), 1, 1, 128, 0, vp(0), ctypes.byref(out)) == bs.ERR_INVALID_ARG
    assert lib.bsattn_plan(fake, 1, 1, 128, 0, vp(0), None) == bs.ERR_INVALID_ARG
    assert lib.bsattn_plan(fake, 1, 1, 100, 0, vp(0), ctypes.byref(out)) == bs.ERR_INVALID_ARG
    assert lib.bsattn_plan(fake, 0, 1, 128, 0, vp(0), ctypes.byref(out)) == bs.ERR_INVALID_ARG
    assert lib.bsattn_plan(fake, 1, -2, 128, 0, vp(0), ctypes.byref(out)) == bs.ERR_INVALID_ARG
    assert lib.bsattn_plan(fake, 1, 1, 128, 16, vp(0), ctypes.byref(out)) == bs.ERR_INVALID_ARG
    assert lib.bsattn_plan(fake, 1, 1, 128 * 4097, 0, vp(0), ctypes.byref(out)) == bs.ERR_UNSUPPORTED
    assert lib.bsattn_plan(fake, 1024, 1024, 4096, 0, vp(0), ctypes.byref(out)) == bs.ERR_UNSUPPORTED
    assert out.value is None


def test_fwd_and_status_reject_missing_plan(lib):
    import block_sparse_flash_attn_gb300 as bs
    vp = ctypes.c_void_p
    fake = vp(0x10000)
    assert lib.bsattn_fwd(fake, fake, fake, vp(0), fake, fake, 1, 1, 128, 128,
                          ctypes.c_float(0.1), vp(0)) == bs.ERR_INVALID_ARG
    assert lib.bsattn_plan_status(vp(0), vp(0)) == bs.ERR_INVALID_ARG
    rp, ci, n = vp(), vp(), ctypes.c_int64()
    assert lib.bsattn_plan_csr(vp(0), ctypes.byref(rp), ctypes.byref(ci), ctypes.byref(n)) == \
        bs.ERR_INVALID_ARG
    v16, nbytes = vp(), ctypes.c_size_t()
    assert lib.bsattn_plan_v16(vp(0), ctypes.byref(v16), ctypes.byref(nbytes)) == \
        bs.ERR_INVALID_ARG
    lib.bsattn_plan_free(vp(0))  # ignored
    assert lib.bsattn_selftest_wait_timeout(10, vp(0)) == bs.ERR_INVALID_ARG
    assert lib.bsattn_selftest_wait_timeout(10 ** 10, vp(0)) == bs.ERR_INVALID_ARG


def test_binding_fails_loudly_without_the_library(monkeypatch):
    import block_sparse_flash_attn_gb300 as bs
    from block_sparse_flash_attn_gb300 import _build
    monkeypatch.setattr(_build, "LIB", os.path.join(ROOT, "does-not-exist", "libbsattn.so"))
    monkeypatch.setattr(bs, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        bs.load()


def test_kernel_source_is_tcgen05_tma():
    """The forward kernel is written with tcgen05 + TMA inline PTX for sm_103a."""
    src = open(os.path.join(ROOT, "block_sparse_flash_attn_gb300", "csrc", "ptx.cuh")).read()
    for needle in ["tcgen05.mma.cta_group::1.kind::f16", "tcgen05.alloc", "tcgen05.ld",
                   "tcgen05.st", "cp.async.bulk.tensor.2d", "mbarrier.try_wait"]:
        assert needle in src
    from block_sparse_flash_attn_gb300 import _build
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.ARCH)


def test_backward_and_gqa_reject_missing_plan(lib):
    """The entry points added for the backward pass and grouped-query attention
    check the plan handle before anything else."""
    import block_sparse_flash_attn_gb300 as bs
    vp = ctypes.c_void_p
    fake = vp(0x10000)
    f = ctypes.c_float(0.1)
    assert lib.bsattn_bwd(fake, fake, fake, fake, fake, fake, vp(0), fake, fake, fake,
                          1, 1, 128, 128, f, vp(0)) == bs.ERR_INVALID_ARG
    assert lib.bsattn_bwd_gqa(fake, fake, fake, fake, fake, fake, vp(0), fake, fake, fake,
                              1, 4, 2, 128, 128, f, vp(0)) == bs.ERR_INVALID_ARG
    assert lib.bsattn_fwd_gqa(fake, fake, fake, vp(0), fake, fake, 1, 4, 2, 128, 128, f,
                              vp(0)) == bs.ERR_INVALID_ARG
    cp, ri, n = vp(), vp(), ctypes.c_int64()
    assert lib.bsattn_plan_csc(vp(0), ctypes.byref(cp), ctypes.byref(ri), ctypes.byref(n)) == \
        bs.ERR_INVALID_ARG
    # the shared-mask flag is accepted by the argument check; an unknown bit is not
    out = vp()
    assert lib.bsattn_plan(vp(0), 1, 4, 128, bs.MASK_SHARED_HEADS, vp(0), ctypes.byref(out)) == \
        bs.ERR_INVALID_ARG  # (null mask)
    assert lib.bsattn_plan(fake, 1, 4, 128, 32, vp(0), ctypes.byref(out)) == bs.ERR_INVALID_ARG


def test_noalloc_wrapper_rejects_bad_tensors_before_any_call(monkeypatch):
    """The allocation-free wrapper checks every tensor itself (the C entry point
    sees raw pointers only): a host mask, a K of another shape, a mask of the
    wrong block shape and a non-contiguous Q are rejected before the library is
    even loaded."""
    import torch

    import block_sparse_flash_attn_gb300 as bs

    def no_load():
        raise AssertionError("the library must not be reached")

    monkeypatch.setattr(bs, "load", no_load)
    B, H, S, D = 1, 2, 256, 64
    q = torch.zeros((B, H, S, D), dtype=torch.bfloat16)
    mask = torch.ones((B, H, 2, 2), dtype=torch.uint8)
    with pytest.raises(ValueError, match="one shape"):
        bs.fwd_noalloc(q, q[:, :1].contiguous(), q, mask)
    with pytest.raises(ValueError, match="mask"):
        bs.fwd_noalloc(q, q, q, torch.ones((B, H, 3, 3), dtype=torch.uint8))
    with pytest.raises(TypeError, match="mask"):
        bs.fwd_noalloc(q, q, q, mask.float())
    with pytest.raises(ValueError, match="contiguous"):
        bs.fwd_noalloc(q.transpose(2, 3), q, q, mask)
    with pytest.raises(ValueError, match="lse"):
        bs.fwd_noalloc(q, q, q, mask, lse=torch.zeros((B, H, S + 1)))
    # right shapes and dtypes, but host tensors (a host mask among them)
    with pytest.raises(TypeError, match="CUDA device"):
        bs.fwd_noalloc(q, q, q, mask)


def test_header_states_the_v_copy_thresholds():
    """bsattn_fwd's documentation gives the sizes at which the call converts V
    to an fp16 copy before the launch; they are the library's constants."""
    internal = open(os.path.join(ROOT, "block_sparse_flash_attn_gb300", "csrc",
                                 "internal.h")).read()
    rows = int(re.search(r"kV16MinRows = (\d+);", internal).group(1))
    reuse = int(re.search(r"kV16MinReuse = (\d+);", internal).group(1))
    header = " ".join(open(HEADER).read().split())
    assert f"at least {rows} rows" in header
    assert f"at least {reuse} live blocks per key block of V" in header
