"""Block-sparse flash-attention forward for NVIDIA GB300 (sm_103a).

Thin Python binding over the C ABI in ``include/bsattn.h`` (``libbsattn.so``,
built in-tree by ``_build.build()``).  This module only marshals arguments:
every step of the attention runs in the library's CUDA kernels.  PyTorch is
used for device memory and streams.  There is no CPU fallback: if the library
is missing, every call raises.

    plan = bsattn.plan(mask_u8_cuda, causal=False)   # once per mask
    o, lse = bsattn.fwd(q, k, v, plan, scale)        # q/k/v bf16 [B,H,S,D] on cuda

The operation: "Writing Pallas Kernels for JAX: Stepping Outside the XLA
Safety Net" (sections "Designing the Block Specification" and "Writing the
Kernel Logic: Load, Compute, Store"), computed exactly across key blocks as in
"Pallas-Triton kernels and kernel auto-tuning" (section "Flash Attention").
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from . import _build

BLOCK = 128

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_OOM, ERR_TIMEOUT, ERR_INTERNAL = range(7)
ERR_SCRATCH_LIMIT = 7
ERR_RANGE = 8
CAUSAL, OUT_F32, MASK_SHARED_HEADS, KEY_BLOCK_64 = 1, 2, 4, 8

EXPORTS = ["bsattn_plan", "bsattn_plan_csr", "bsattn_plan_schedule", "bsattn_fwd",
           "bsattn_plan_status", "bsattn_plan_free", "bsattn_status_string", "bsattn_version",
           "bsattn_selftest_wait_timeout", "bsattn_fwd_noalloc", "bsattn_pipeline_create",
           "bsattn_pipeline_run", "bsattn_pipeline_status", "bsattn_pipeline_free",
           "bsattn_plan_csc", "bsattn_bwd", "bsattn_fwd_gqa", "bsattn_bwd_gqa",
           "bsattn_fwd_fp8", "bsattn_plan_v16"]


class BsattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None


def lib_path() -> str:
    """The library this process loads: _build.LIB, or the build named by the
    BSATTN_LIBRARY environment variable (the tuner's per-setting builds)."""
    return os.environ.get("BSATTN_LIBRARY") or _build.LIB


def load():
    """Load libbsattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run block_sparse_flash_attn_gb300._build.build()"
                           " (or __graft_entry__.build()) first -- there is no fallback path")
    lib = ctypes.CDLL(path)
    vp, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint
    lib.bsattn_plan.argtypes = [vp, i32, i32, i32, u32, vp, ctypes.POINTER(vp)]
    lib.bsattn_plan.restype = i32
    lib.bsattn_plan_csr.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i64)]
    lib.bsattn_plan_csr.restype = i32
    lib.bsattn_plan_schedule.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(i64),
                                         ctypes.POINTER(vp), ctypes.POINTER(i64)]
    lib.bsattn_plan_schedule.restype = i32
    lib.bsattn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_float, vp]
    lib.bsattn_fwd.restype = i32
    lib.bsattn_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float,
                                   vp]
    lib.bsattn_fwd_gqa.restype = i32
    lib.bsattn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_float,
                                   ctypes.c_float, vp]
    lib.bsattn_fwd_fp8.restype = i32
    lib.bsattn_plan_csc.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i64)]
    lib.bsattn_plan_csc.restype = i32
    lib.bsattn_plan_v16.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(ctypes.c_size_t)]
    lib.bsattn_plan_v16.restype = i32
    lib.bsattn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                               ctypes.c_float, vp]
    lib.bsattn_bwd.restype = i32
    lib.bsattn_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                   ctypes.c_float, vp]
    lib.bsattn_bwd_gqa.restype = i32
    lib.bsattn_plan_status.argtypes = [vp, vp]
    lib.bsattn_plan_status.restype = i32
    lib.bsattn_plan_free.argtypes = [vp]
    lib.bsattn_plan_free.restype = None
    lib.bsattn_status_string.argtypes = [i32]
    lib.bsattn_status_string.restype = ctypes.c_char_p
    lib.bsattn_version.argtypes = []
    lib.bsattn_version.restype = i32
    lib.bsattn_selftest_wait_timeout.argtypes = [i64, vp]
    lib.bsattn_selftest_wait_timeout.restype = i32
    lib.bsattn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_float,
                                       u32, vp]
    lib.bsattn_fwd_noalloc.restype = i32
    lib.bsattn_pipeline_create.argtypes = [vp, i32, i32, i32, i32, u32, i32, vp, ctypes.POINTER(vp)]
    lib.bsattn_pipeline_create.restype = i32
    lib.bsattn_pipeline_run.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, vp]
    lib.bsattn_pipeline_run.restype = i32
    lib.bsattn_pipeline_status.argtypes = [vp]
    lib.bsattn_pipeline_status.restype = i32
    lib.bsattn_pipeline_free.argtypes = [vp]
    lib.bsattn_pipeline_free.restype = None
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().bsattn_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise BsattnError(status, what)


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class _DeviceView:
    """Zero-copy int32 view of library-owned device memory (for torch.as_tensor)."""

    def __init__(self, ptr: int, n: int):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i4", "data": (ptr, False),
                                         "version": 3, "strides": None}


def _view_i32(ptr, n: int) -> torch.Tensor:
    if n == 0:
        return torch.empty(0, dtype=torch.int32, device="cuda")
    return torch.as_tensor(_DeviceView(int(ptr), int(n)), device="cuda").clone()


class Plan:
    """Handle to a device-side plan (CSR of live key blocks + tile schedule)."""

    def __init__(self, handle: int, B: int, H: int, S: int, causal: bool, out_f32: bool,
                 key_block: int = BLOCK):
        self._h = ctypes.c_void_p(handle)
        self.B, self.H, self.S = B, H, S
        self.causal, self.out_f32 = causal, out_f32
        self.key_block = key_block

    @property
    def handle(self) -> ctypes.c_void_p:
        if not self._h:
            raise ValueError("plan was freed")
        return self._h

    def close(self) -> None:
        if self._h:
            load().bsattn_plan_free(self._h)
            self._h = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass


def plan(mask: torch.Tensor, causal: bool = False, out_f32: bool = False, stream=None,
         heads: int | None = None, key_block: int = BLOCK) -> Plan:
    """Build the plan for a uint8 block mask [B, H, S/128, S/128] on the GPU.

    With heads=H and a mask of shape [B, 1, S/128, S/128], the one mask of
    each batch entry applies to all its H heads.  With key_block=64 the mask
    is [B, H, S/128, S/64]: one entry per 128-query x 64-key block (forward
    pass only)."""
    if not (isinstance(mask, torch.Tensor) and mask.is_cuda and mask.dtype == torch.uint8):
        raise TypeError("mask must be a CUDA uint8 tensor")
    if key_block not in (BLOCK, 64):
        raise ValueError("key_block must be 128 or 64")
    kdiv = BLOCK // key_block
    if mask.dim() != 4 or mask.shape[3] != kdiv * mask.shape[2]:
        raise ValueError(f"mask must be [B, H, nb, {kdiv} * nb]")
    mask = mask.contiguous()
    B, H, nb, _ = mask.shape
    flags = (CAUSAL if causal else 0) | (OUT_F32 if out_f32 else 0) | \
        (KEY_BLOCK_64 if key_block == 64 else 0)
    if heads is not None and heads != H:
        if H != 1:
            raise ValueError("a mask shared by the heads must have shape [B, 1, nb, nb]")
        H = int(heads)
        flags |= MASK_SHARED_HEADS
    h = ctypes.c_void_p()
    with torch.cuda.device(mask.device):
        _check(load().bsattn_plan(ctypes.c_void_p(mask.data_ptr()), B, H, nb * BLOCK, flags,
                                  _stream_handle(stream), ctypes.byref(h)), "bsattn_plan")
    return Plan(h.value, B, H, nb * BLOCK, causal, out_f32, key_block)


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, p: Plan, scale: float | None = None,
        out: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """O, LSE = block-sparse attention.  q: CUDA bf16 [B, H, S, D]; k, v: [B, Hkv, S, D]
    with H % Hkv == 0 (Hkv < H: grouped-query attention); all contiguous."""
    for t in (q, k, v):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16):
            raise TypeError("q, k, v must be CUDA bf16 tensors")
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    if q.dim() != 4 or k.shape != v.shape or k.dim() != 4 or k.shape[0] != q.shape[0] \
            or k.shape[2:] != q.shape[2:] or q.shape[1] % k.shape[1] != 0:
        raise ValueError("q must be [B, H, S, D] and k, v [B, Hkv, S, D] with H % Hkv == 0")
    B, H, S, D = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    odt = torch.float32 if p.out_f32 else torch.bfloat16
    if out is None:
        out = torch.empty((B, H, S, D), dtype=odt, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    if out.dtype != odt or out.shape != (B, H, S, D) or not out.is_contiguous():
        raise ValueError("out has the wrong dtype/shape/layout for this plan")
    if lse.dtype != torch.float32 or lse.shape != (B, H, S) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B, H, S]")
    vp = ctypes.c_void_p
    with torch.cuda.device(q.device):
        if Hkv == H:
            _check(load().bsattn_fwd(vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()),
                                     p.handle, vp(out.data_ptr()), vp(lse.data_ptr()), B, H, S, D,
                                     float(scale), _stream_handle(stream)), "bsattn_fwd")
        else:
            _check(load().bsattn_fwd_gqa(vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()),
                                         p.handle, vp(out.data_ptr()), vp(lse.data_ptr()), B, H,
                                         Hkv, S, D, float(scale), _stream_handle(stream)),
                   "bsattn_fwd_gqa")
    return out, lse


def fwd_fp8(q8: torch.Tensor, k8: torch.Tensor, v8: torch.Tensor, p: Plan,
            scale: float | None = None, v_scale: float = 1.0, out: torch.Tensor | None = None,
            lse: torch.Tensor | None = None, stream=None):
    """O, LSE of block-sparse attention on e4m3 inputs: q8, k8, v8 CUDA
    [B, H, S, 128] of torch.float8_e4m3fn (or uint8 holding e4m3 bits),
    contiguous.  scale multiplies q.k (include the Q and K scales in it);
    v_scale multiplies O."""
    for t in (q8, k8, v8):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or \
                t.dtype not in (torch.uint8, torch.float8_e4m3fn):
            raise TypeError("q8, k8, v8 must be CUDA float8_e4m3fn (or uint8) tensors")
        if not t.is_contiguous():
            raise ValueError("q8, k8, v8 must be contiguous")
    if q8.dim() != 4 or k8.shape != q8.shape or v8.shape != q8.shape:
        raise ValueError("q8, k8, v8 must share one shape [B, H, S, D]")
    B, H, S, D = q8.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    odt = torch.float32 if p.out_f32 else torch.bfloat16
    if out is None:
        out = torch.empty((B, H, S, D), dtype=odt, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q8.device)
    if out.dtype != odt or out.shape != (B, H, S, D) or not out.is_contiguous():
        raise ValueError("out has the wrong dtype/shape/layout for this plan")
    if lse.dtype != torch.float32 or lse.shape != (B, H, S) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B, H, S]")
    vp = ctypes.c_void_p
    with torch.cuda.device(q8.device):
        _check(load().bsattn_fwd_fp8(vp(q8.data_ptr()), vp(k8.data_ptr()), vp(v8.data_ptr()),
                                     p.handle, vp(out.data_ptr()), vp(lse.data_ptr()), B, H, S, D,
                                     float(scale), float(v_scale), _stream_handle(stream)),
               "bsattn_fwd_fp8")
    return out, lse


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
        dout: torch.Tensor, p: Plan, scale: float | None = None, dq: torch.Tensor | None = None,
        dk: torch.Tensor | None = None, dv: torch.Tensor | None = None, stream=None):
    """dQ [B, H, S, D], dK and dV [B, Hkv, S, D] (CUDA fp32) of block-sparse attention.

    q/dout: CUDA bf16 [B, H, S, D], k/v: [B, Hkv, S, D] (H % Hkv == 0; Hkv < H:
    grouped-query attention), contiguous; o, lse: the forward's outputs for
    plan p; scale: the forward's scale."""
    for t in (q, k, v, dout):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16):
            raise TypeError("q, k, v, dout must be CUDA bf16 tensors")
        if not t.is_contiguous():
            raise ValueError("q, k, v, dout must be contiguous")
    if q.dim() != 4 or dout.shape != q.shape or k.dim() != 4 or v.shape != k.shape \
            or k.shape[0] != q.shape[0] or k.shape[2:] != q.shape[2:] or q.shape[1] % k.shape[1]:
        raise ValueError("q, dout must be [B, H, S, D] and k, v [B, Hkv, S, D] with H % Hkv == 0")
    B, H, S, D = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    odt = torch.float32 if p.out_f32 else torch.bfloat16
    if o.dtype != odt or o.shape != q.shape or not o.is_contiguous():
        raise ValueError("o has the wrong dtype/shape/layout for this plan")
    if lse.dtype != torch.float32 or lse.shape != (B, H, S) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B, H, S]")
    grads = []
    for g, shape in ((dq, q.shape), (dk, k.shape), (dv, k.shape)):
        if g is None:
            g = torch.empty(shape, dtype=torch.float32, device=q.device)
        if g.dtype != torch.float32 or g.shape != shape or not g.is_contiguous():
            raise ValueError("dq must be contiguous fp32 like q, dk and dv like k")
        grads.append(g)
    vp = ctypes.c_void_p
    with torch.cuda.device(q.device):
        _check(load().bsattn_bwd_gqa(vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()),
                                     vp(o.data_ptr()), vp(lse.data_ptr()), vp(dout.data_ptr()),
                                     p.handle, vp(grads[0].data_ptr()), vp(grads[1].data_ptr()),
                                     vp(grads[2].data_ptr()), B, H, Hkv, S, D, float(scale),
                                     _stream_handle(stream)), "bsattn_bwd_gqa")
    return tuple(grads)


def plan_status(p: Plan, stream=None) -> None:
    """Wait for the stream; raise if a kernel reported a timeout or internal error."""
    _check(load().bsattn_plan_status(p.handle, _stream_handle(stream)), "device status")


def plan_csr(p: Plan):
    """(row_ptr, col_idx) as fresh CUDA int32 tensors."""
    rp, ci, nnz = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_int64()
    _check(load().bsattn_plan_csr(p.handle, ctypes.byref(rp), ctypes.byref(ci), ctypes.byref(nnz)),
           "bsattn_plan_csr")
    rows = p.B * p.H * (p.S // BLOCK)
    return _view_i32(rp.value, rows + 1), _view_i32(ci.value, nnz.value)


def plan_csc(p: Plan):
    """(col_ptr, row_idx) of the transposed plan as fresh CUDA int32 tensors."""
    cp, ri, nnz = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_int64()
    _check(load().bsattn_plan_csc(p.handle, ctypes.byref(cp), ctypes.byref(ri), ctypes.byref(nnz)),
           "bsattn_plan_csc")
    cols = p.B * p.H * (p.S // BLOCK)
    return _view_i32(cp.value, cols + 1), _view_i32(ri.value, nnz.value)


def plan_schedule(p: Plan):
    """(tile_order, empty_tiles) as fresh CUDA int32 tensors."""
    to, et = ctypes.c_void_p(), ctypes.c_void_p()
    nl, ne = ctypes.c_int64(), ctypes.c_int64()
    _check(load().bsattn_plan_schedule(p.handle, ctypes.byref(to), ctypes.byref(nl),
                                       ctypes.byref(et), ctypes.byref(ne)), "bsattn_plan_schedule")
    return _view_i32(to.value, nl.value), _view_i32(et.value, ne.value)


def plan_v16_bytes(p: Plan) -> int:
    """Size in bytes of the plan's fp16 copy of V (head_dim 64), 0 while none exists."""
    ptr, nbytes = ctypes.c_void_p(), ctypes.c_size_t()
    _check(load().bsattn_plan_v16(p.handle, ctypes.byref(ptr), ctypes.byref(nbytes)),
           "bsattn_plan_v16")
    return int(nbytes.value)


def selftest_wait_timeout(timeout_ns: int = 1_000_000, stream=None) -> int:
    """Run the bounded-wait self test; returns the status (ERR_TIMEOUT is the expected one)."""
    return int(load().bsattn_selftest_wait_timeout(int(timeout_ns), _stream_handle(stream)))


def fwd_noalloc(q, k, v, mask, causal: bool = False, scale: float | None = None,
                out_f32: bool = False, out=None, lse=None, stream=None):
    """Forward pass that allocates no device memory inside the library.

    For callers that cannot call cudaMalloc: the plan and the kernel's scratch
    live in the library's fixed 16 MiB device array (see bsattn_fwd_noalloc in
    include/bsattn.h for the limit and the sharing rules).  Output tensors are
    allocated here by torch only when not passed in.

    Every tensor is checked before the call (the C entry point sees only raw
    pointers and cannot tell a host tensor or a short buffer from a good one):
    q, k, v contiguous bf16 [B, H, S, D] of one shape; mask contiguous uint8
    [B, H, S/128, S/128]; out and lse of the output dtype and shape; all on
    one CUDA device.
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be a bf16 tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one shape [B, H, S, D]")
    B, H, S, D = q.shape
    if S % BLOCK:
        raise ValueError("S must be a multiple of 128")
    nb = S // BLOCK
    if not isinstance(mask, torch.Tensor) or mask.dtype != torch.uint8:
        raise TypeError("mask must be a uint8 tensor")
    if tuple(mask.shape) != (B, H, nb, nb) or not mask.is_contiguous():
        raise ValueError(f"mask must be contiguous [B, H, S/128, S/128] = {(B, H, nb, nb)}")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    odt = torch.float32 if out_f32 else torch.bfloat16
    if out is not None and (out.dtype != odt or tuple(out.shape) != (B, H, S, D)
                            or not out.is_contiguous()):
        raise ValueError("out must be contiguous [B, H, S, D] of the output dtype")
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, S)
                            or not lse.is_contiguous()):
        raise ValueError("lse must be contiguous fp32 [B, H, S]")
    for name, t in (("q", q), ("k", k), ("v", v), ("mask", mask), ("out", out), ("lse", lse)):
        if t is not None and (not t.is_cuda or t.device != q.device):
            raise TypeError(f"{name} must be on q's CUDA device")
    if out is None:
        out = torch.empty((B, H, S, D), dtype=odt, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    flags = (CAUSAL if causal else 0) | (OUT_F32 if out_f32 else 0)
    with torch.cuda.device(q.device):
        _check(load().bsattn_fwd_noalloc(
            ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(mask.data_ptr()),
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), B, H, S, D,
            float(scale), flags, _stream_handle(stream)), "bsattn_fwd_noalloc")
    return out, lse


class HostPipeline:
    """Forward passes on host-resident (pinned) tensors, transfers overlapped.

    Wraps bsattn_pipeline_*: the library cuts the flattened (batch, head)
    range into `chunks` parts (a plan each, built here once) and, on every
    run, overlaps one part's upload, another's kernel and a third's download
    on three streams.  Every run copies all of its inputs in and all of its
    results out; results equal fwd()'s.
    """

    def __init__(self, mask: torch.Tensor, D: int, causal: bool = False, out_f32: bool = False,
                 chunks: int = 4, stream=None):
        if not (isinstance(mask, torch.Tensor) and mask.is_cuda and mask.dtype == torch.uint8):
            raise TypeError("mask must be a CUDA uint8 tensor")
        if mask.dim() != 4 or mask.shape[2] != mask.shape[3]:
            raise ValueError("mask must be [B, H, nb, nb]")
        mask = mask.contiguous()
        B, H, nb, _ = mask.shape
        self.B, self.H, self.S, self.D = B, H, nb * BLOCK, int(D)
        self.out_dtype = torch.float32 if out_f32 else torch.bfloat16
        flags = (CAUSAL if causal else 0) | (OUT_F32 if out_f32 else 0)
        h = ctypes.c_void_p()
        with torch.cuda.device(mask.device):
            _check(load().bsattn_pipeline_create(ctypes.c_void_p(mask.data_ptr()), B, H, self.S,
                                                 self.D, flags, int(chunks),
                                                 _stream_handle(stream), ctypes.byref(h)),
                   "bsattn_pipeline_create")
        self._h = h.value
        self.device = mask.device

    def run(self, hq: torch.Tensor, hk: torch.Tensor, hv: torch.Tensor, ho: torch.Tensor,
            hlse: torch.Tensor, scale: float | None = None, stream=None) -> None:
        """Enqueue one forward pass: pinned host [B, H, S, D] bf16 in, pinned host O
        [B, H, S, D] and LSE [B, H, S] out.  `stream` (default: the current one)
        is made to wait for the results; synchronise it before reading them."""
        shp = (self.B, self.H, self.S, self.D)
        for t in (hq, hk, hv):
            if t.is_cuda or t.dtype != torch.bfloat16 or tuple(t.shape) != shp or \
                    not t.is_contiguous():
                raise ValueError("hq, hk, hv must be contiguous host bf16 [B, H, S, D]")
        if ho.is_cuda or ho.dtype != self.out_dtype or tuple(ho.shape) != shp or \
                not ho.is_contiguous():
            raise ValueError("ho must be a contiguous host tensor [B, H, S, D] of the output dtype")
        if hlse.is_cuda or hlse.dtype != torch.float32 or tuple(hlse.shape) != shp[:3] or \
                not hlse.is_contiguous():
            raise ValueError("hlse must be a contiguous host fp32 tensor [B, H, S]")
        if scale is None:
            scale = 1.0 / math.sqrt(self.D)
        with torch.cuda.device(self.device):
            _check(load().bsattn_pipeline_run(
                ctypes.c_void_p(self._h), ctypes.c_void_p(hq.data_ptr()),
                ctypes.c_void_p(hk.data_ptr()), ctypes.c_void_p(hv.data_ptr()),
                ctypes.c_void_p(ho.data_ptr()), ctypes.c_void_p(hlse.data_ptr()), float(scale),
                _stream_handle(stream)), "bsattn_pipeline_run")

    def status(self) -> None:
        """Wait for the pipeline; raise if a kernel reported a timeout or internal error."""
        _check(load().bsattn_pipeline_status(ctypes.c_void_p(self._h)), "pipeline status")

    def close(self) -> None:
        if getattr(self, "_h", None):
            load().bsattn_pipeline_free(ctypes.c_void_p(self._h))
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown
            pass


def attention(q, k, v, mask, causal: bool = False, scale: float | None = None,
              out_f32: bool = False):
    """Convenience: plan + fwd for a one-off call."""
    p = plan(mask, causal=causal, out_f32=out_f32)
    try:
        return fwd(q, k, v, p, scale)
    finally:
        torch.cuda.current_stream().synchronize()
        p.close()
