"""ORACLE -- test infrastructure, not product code.

A plain fp64 CPU definition of block-sparse attention (and of its mask-to-CSR
plan), written in C (``oracle.c``) and loaded through ctypes.  Only the tests,
``__graft_entry__.smoke()`` and the bench's ``cpu_baseline`` / reference leg
may import this package.  It shares nothing with the CUDA path.

Definitions follow "Writing Pallas Kernels for JAX: Stepping Outside the XLA
Safety Net" (sections "Designing the Block Specification" and "Writing the
Kernel Logic: Load, Compute, Store") and "Pallas-Triton kernels and kernel
auto-tuning" (section "Flash Attention": exact attention); see oracle.c for
the formulas and the readings taken where the pages are silent.

Every function here is pinned by tests/test_oracle_pins.py (brute force,
library special cases, closed forms and invariants); none is "parity
unpinned".  The gradients and the transposed plan (``backward.py``, numpy
fp64) are pinned by tests/test_oracle_bwd_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")

BLOCK = 128

# Planted mistakes (test-only), see oracle.c.
MUTATIONS = {
    1: "scale dropped",
    2: "exp sign flipped",
    3: "block mask transposed",
    4: "causal made strict (j < i)",
    5: "LSE without the max term",
    6: "O not normalised by l",
    7: "scores use Q in place of K",
    8: "O sums the query row of V",
    9: "fully masked rows left as NaN",
    10: "last head_dim term dropped from the dot product",
    11: "LSE in log2 units",
    14: "causal flag ignored",
}


def build(force: bool = False) -> str:
    """Compile oracle.c into _lib/liboracle.so (plain C99, fp64, OpenMP)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
                               "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _get():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        lib.oracle_attn_rows.argtypes = [i32, vp, vp, vp, vp, i32, i32, i32, i32,
                                         ctypes.c_double, i32, vp, i64, vp, vp, i32]
        lib.oracle_attn_rows.restype = i32
        lib.oracle_csr.argtypes = [vp, i32, i32, i32, i32, vp, vp]
        lib.oracle_csr.restype = i64
        lib.oracle_set_mutation.argtypes = [i32]
        lib.oracle_set_mutation.restype = None
        lib.oracle_get_mutation.argtypes = []
        lib.oracle_get_mutation.restype = i32
        _lib = lib
    return _lib


def set_mutation(m: int) -> None:
    """Plant mistake number m (0 = none).  Tests only."""
    _get().oracle_set_mutation(int(m))


def attention(q, k, v, mask, scale: float, causal: bool = False, rows=None,
              nthreads: int = 0):
    """Exact block-sparse attention in fp64.

    q, k, v: [B][H][S][D] as uint16 bf16 bit patterns, or float64 arrays.
    mask: uint8 [B][H][S/128][S/128].  rows: flat row ids (b*H+h)*S+i, or
    None for every row.  Returns (O [n_rows][D] float64, LSE [n_rows] float64);
    with rows=None they are reshaped to [B][H][S][D] and [B][H][S].
    """
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    if q.dtype == np.uint16:
        kind = 0
    elif q.dtype == np.float64:
        kind = 1
    else:
        raise TypeError("q/k/v must be uint16 bf16 bit patterns or float64")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share a dtype")
    B, H, S, D = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v shapes differ")
    if S % BLOCK:
        raise ValueError("S must be a multiple of 128")
    nb = S // BLOCK
    if mask.shape != (B, H, nb, nb):
        raise ValueError(f"mask shape {mask.shape} != {(B, H, nb, nb)}")
    full = rows is None
    if full:
        rows = np.arange(B * H * S, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    O = np.empty((rows.size, D), dtype=np.float64)
    L = np.empty(rows.size, dtype=np.float64)
    rc = _get().oracle_attn_rows(kind, q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                 mask.ctypes.data, B, H, S, D, float(scale), int(bool(causal)),
                                 rows.ctypes.data, rows.size, O.ctypes.data, L.ctypes.data,
                                 int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_rows failed ({rc})")
    if full:
        return O.reshape(B, H, S, D), L.reshape(B, H, S)
    return O, L


def csr(mask, causal: bool = False):
    """Per query block, the ascending live key blocks: (row_ptr int32, col_idx int32)."""
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    B, H, nb, nb2 = mask.shape
    if nb != nb2:
        raise ValueError("mask must be [B][H][nb][nb]")
    row_ptr = np.empty(B * H * nb + 1, dtype=np.int32)
    lib = _get()
    nnz = lib.oracle_csr(mask.ctypes.data, B, H, nb, int(bool(causal)), row_ptr.ctypes.data, None)
    if nnz < 0:
        raise RuntimeError("oracle_csr failed")
    col_idx = np.empty(max(int(nnz), 1), dtype=np.int32)
    lib.oracle_csr(mask.ctypes.data, B, H, nb, int(bool(causal)), row_ptr.ctypes.data,
                   col_idx.ctypes.data)
    return row_ptr, col_idx[:nnz]


def attention_gqa(q, k, v, mask, scale: float, causal: bool = False, rows=None):
    """Grouped-query attention, fp64: q [B][H][S][D], k and v [B][Hkv][S][D]
    with H % Hkv == 0; query head h attends with K/V head h // (H // Hkv).
    mask [B][H][nb][nb], or [B][1][nb][nb] shared by the heads of a batch entry.

    Defined as the attention above on K and V with each head repeated
    H // Hkv times and the mask broadcast over the heads (the pages use one
    K/V head per query head; this is the plain extension of their shapes).
    Pinned by tests/test_oracle_pins.py against torch's float64
    scaled_dot_product_attention with enable_gqa.
    """
    q = np.asarray(q)
    B, H = q.shape[:2]
    Hkv = np.asarray(k).shape[1]
    if H % Hkv:
        raise ValueError("H must be a multiple of the K/V heads")
    g = H // Hkv
    k_rep = np.ascontiguousarray(np.repeat(np.asarray(k), g, axis=1))
    v_rep = np.ascontiguousarray(np.repeat(np.asarray(v), g, axis=1))
    mask = np.asarray(mask, dtype=np.uint8)
    if mask.shape[1] == 1 and H > 1:
        mask = np.ascontiguousarray(np.broadcast_to(mask, (B, H) + mask.shape[2:]))
    return attention(q, k_rep, v_rep, mask, scale, causal, rows=rows)

from .backward import BWD_MUTATIONS, attention_bwd, attention_bwd_gqa, csc, set_bwd_mutation  # noqa: E402,F401,E501
from .fp8 import attention_fp8, decode_e4m3  # noqa: E402,F401
from .keyblocks import attention_kb, csr_kb  # noqa: E402,F401
