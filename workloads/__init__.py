"""Seeded synthetic workloads for block-sparse attention (inputs only).

This module produces inputs -- Q/K/V bit patterns and block masks -- and
nothing else: no attention arithmetic lives here.  Both the CUDA path and the
CPU oracle consume what it produces.

Shapes follow the query/key/value layout of "Writing Pallas Kernels for JAX:
Stepping Outside the XLA Safety Net" (section "Designing the Block
Specification": tensors of shape (batch, seq_len, head_dim) processed in
128-token chunks), with a head axis added: every tensor is [B][H][S][D],
contiguous, bf16.  The block mask is uint8 [B][H][S/128][S/128], one entry per
(128-query-block, 128-key-block) pair, nonzero = live.

Recipes of the five workloads (seeds: data = 1000 + id, mask = 2000 + id):
  1  B1 H2  S512   D64   N(0,1)   off-diagonal blocks live iid p=0.5, diagonal live
  2  B4 H16 S4096  D128  N(0,1)   causal: lower-triangular blocks + element causal
  3  B2 H32 S16384 D128  N(0,1)   BigBird: |qb-kb|<=4, rows/cols 0..1 global,
                                  + 3 distinct random blocks per row drawn
                                  uniformly from that row's still-dead blocks
  4  B1 H32 S65536 D128  N(0,1)   iid p=0.1 per block per head, diagonal live
  5  B8 H16 S8192  D64   N(0,1)*2 all ones (dense, non-causal)
Random masks are independent per (batch, head).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libbsgen.so")
_SRC = os.path.join(_HERE, "gen.c")

BLOCK = 128

# stream ids inside one seed
STREAM_Q, STREAM_K, STREAM_V = 1, 2, 3
STREAM_DO = 4  # upstream gradient dO of the backward pass
STREAM_MASK_IID, STREAM_MASK_BIGBIRD = 10, 11


def build(force: bool = False) -> str:
    """Compile gen.c into _lib/libbsgen.so (plain C99 + OpenMP)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _get():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u64, i64 = ctypes.c_uint64, ctypes.c_int64
        lib.bsgen_u64.argtypes = [u64, u64, i64, i64, ctypes.c_void_p]
        lib.bsgen_uniform.argtypes = [u64, u64, i64, i64, ctypes.c_void_p]
        lib.bsgen_normal_bf16.argtypes = [u64, u64, i64, i64, ctypes.c_float, ctypes.c_void_p]
        lib.bsgen_normal_f64.argtypes = [u64, u64, i64, i64, ctypes.c_double, ctypes.c_void_p]
        lib.bsgen_splitmix64_raw.argtypes = [u64, i64, i64, ctypes.c_void_p]
        for f in (lib.bsgen_u64, lib.bsgen_uniform, lib.bsgen_normal_bf16, lib.bsgen_normal_f64,
                  lib.bsgen_splitmix64_raw):
            f.restype = None
        _lib = lib
    return _lib


def splitmix64_raw(key: int, count: int, start: int = 0) -> np.ndarray:
    out = np.empty(count, dtype=np.uint64)
    _get().bsgen_splitmix64_raw(key, start, count, out.ctypes.data)
    return out


def uniform(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    out = np.empty(count, dtype=np.float64)
    _get().bsgen_uniform(seed, stream, start, count, out.ctypes.data)
    return out


def normal_bf16(seed: int, stream: int, shape, mult: float = 1.0) -> np.ndarray:
    """N(0,1)*mult rounded to bf16; returns the uint16 bit patterns."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    _get().bsgen_normal_bf16(seed, stream, 0, n, float(mult), out.ctypes.data)
    return out.reshape(shape)


def normal_f64(seed: int, stream: int, shape, mult: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)
    _get().bsgen_normal_f64(seed, stream, 0, n, float(mult), out.ctypes.data)
    return out.reshape(shape)


# e4m3 (the OCP 8-bit format: sign, 4 exponent bits with bias 7, 3 mantissa
# bits, no infinities, 0x7F / 0xFF NaN): the 127 non-negative finite values,
# indexed by their code 0x00..0x7E, for rounding inputs to the format.
_E4M3_POS = np.array([(m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
                      for e in range(16) for m in range(8)][:127])


def e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round values to e4m3 (nearest, ties to the even code; beyond +-448
    saturates to +-448; NaN -> 0x7F); returns the uint8 bit patterns.

    A value a = |x| in [2^E, 2^(E+1)) (E >= -6) has e4m3 steps of 2^(E-3):
    q = rint(a / 2^(E-3)) in [8, 16] (16 carries into the next binade), code
    = (E + 7) * 8 + q - 8; below 2^-6 the steps are 2^-9 (subnormals)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(np.nan_to_num(x)), _E4M3_POS[-1])
    _, e = np.frexp(a)                      # a = f * 2^e, f in [0.5, 1)
    E = np.maximum(e.astype(np.int64) - 1, -6)
    q = np.rint(np.ldexp(a, -(E - 3))).astype(np.int64)   # ties to even, like the format
    code = np.where(a < 2.0 ** -6, q, (E + 7) * 8 + q - 8)
    code = np.minimum(code, 0x7E).astype(np.uint8)
    code = np.where(np.signbit(x) & (code != 0), code | 0x80, code)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def normal_e4m3(seed: int, stream: int, shape, mult: float = 1.0) -> np.ndarray:
    """N(0,1)*mult (the same draws as normal_f64) rounded to e4m3; uint8 bits."""
    return e4m3_bits(normal_f64(seed, stream, shape, mult))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for display/tests)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# masks
# ----------------------------------------------------------------------------

def mask_iid(seed: int, B: int, H: int, nb: int, p: float, diag: bool = True) -> np.ndarray:
    u = uniform(seed, STREAM_MASK_IID, B * H * nb * nb).reshape(B, H, nb, nb)
    m = (u < p).astype(np.uint8)
    if diag:
        idx = np.arange(nb)
        m[:, :, idx, idx] = 1
    return m


def mask_causal(B: int, H: int, nb: int) -> np.ndarray:
    tri = np.tril(np.ones((nb, nb), dtype=np.uint8))
    return np.broadcast_to(tri, (B, H, nb, nb)).copy()


def mask_bigbird(seed: int, B: int, H: int, nb: int, window: int = 4,
                 n_global: int = 2, n_random: int = 3) -> np.ndarray:
    qb = np.arange(nb)[:, None]
    kb = np.arange(nb)[None, :]
    base = ((np.abs(qb - kb) <= window) | (qb < n_global) | (kb < n_global)).astype(np.uint8)
    m = np.broadcast_to(base, (B, H, nb, nb)).copy()
    u = uniform(seed, STREAM_MASK_BIGBIRD, B * H * nb * n_random).reshape(B, H, nb, n_random)
    for b in range(B):
        for h in range(H):
            for r in range(nb):
                cand = list(np.flatnonzero(m[b, h, r] == 0))
                for t in range(n_random):
                    if not cand:
                        break
                    pick = cand.pop(int(u[b, h, r, t] * len(cand)))
                    m[b, h, r, pick] = 1
    return m


def mask_ones(B: int, H: int, nb: int) -> np.ndarray:
    return np.ones((B, H, nb, nb), dtype=np.uint8)


# ----------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    id: int
    name: str
    B: int
    H: int
    S: int
    D: int
    mask_kind: str      # "iid50", "causal", "bigbird", "iid10", "ones"
    causal: bool
    mult: float         # input standard deviation

    @property
    def nb(self) -> int:
        return self.S // BLOCK

    @property
    def scale(self) -> float:
        """1/sqrt(D) as the float32 value both sides receive."""
        return float(np.float32(1.0 / np.sqrt(self.D)))

    @property
    def data_seed(self) -> int:
        return 1000 + self.id

    @property
    def mask_seed(self) -> int:
        return 2000 + self.id

    def describe(self, in_dtype: str = "bf16") -> str:
        return (f"B={self.B} H={self.H} S={self.S} D={self.D} mask={self.mask_kind}"
                f"{' causal' if self.causal else ''} inputs=N(0,1)*{self.mult:g} {in_dtype}")


WORKLOADS = {
    1: Workload(1, "sparse-p50-s512-d64", 1, 2, 512, 64, "iid50", False, 1.0),
    2: Workload(2, "causal-s4096-d128", 4, 16, 4096, 128, "causal", True, 1.0),
    3: Workload(3, "bigbird-s16384-d128", 2, 32, 16384, 128, "bigbird", False, 1.0),
    4: Workload(4, "random10-s65536-d128", 1, 32, 65536, 128, "iid10", False, 1.0),
    5: Workload(5, "dense-s8192-d64-x2", 8, 16, 8192, 64, "ones", False, 2.0),
}


def make_mask(w: Workload, B: int | None = None, H: int | None = None) -> np.ndarray:
    B = w.B if B is None else B
    H = w.H if H is None else H
    nb = w.nb
    if w.mask_kind == "iid50":
        return mask_iid(w.mask_seed, B, H, nb, 0.5)
    if w.mask_kind == "iid10":
        return mask_iid(w.mask_seed, B, H, nb, 0.1)
    if w.mask_kind == "causal":
        return mask_causal(B, H, nb)
    if w.mask_kind == "bigbird":
        return mask_bigbird(w.mask_seed, B, H, nb)
    if w.mask_kind == "ones":
        return mask_ones(B, H, nb)
    raise ValueError(w.mask_kind)


STREAM_MASK_IID64 = 12


def make_mask_kb64(w: Workload, B: int | None = None, H: int | None = None) -> np.ndarray:
    """The workload's mask at 64-key granularity, uint8 [B][H][S/128][S/64]:
    the iid masks drawn afresh per (128-query, 64-key) block with the same
    density, the two 64-key halves of each diagonal block live; the
    structured masks (causal, BigBird, dense) with every 128-key entry
    repeated over its two halves (the same pattern, finer grid)."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    nb = w.nb
    if w.mask_kind in ("iid50", "iid10"):
        p = 0.5 if w.mask_kind == "iid50" else 0.1
        u = uniform(w.mask_seed, STREAM_MASK_IID64, B * H * nb * 2 * nb).reshape(B, H, nb, 2 * nb)
        m = (u < p).astype(np.uint8)
        idx = np.arange(nb)
        m[:, :, idx, 2 * idx] = 1
        m[:, :, idx, 2 * idx + 1] = 1
        return m
    return np.repeat(make_mask(w, B, H), 2, axis=3)


def make_qkv(w: Workload, B: int | None = None, H: int | None = None):
    """Q, K, V as bf16 bit patterns [B][H][S][D] (uint16)."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    shape = (B, H, w.S, w.D)
    return tuple(normal_bf16(w.data_seed, s, shape, w.mult) for s in (STREAM_Q, STREAM_K, STREAM_V))


def custom(seed: int, B: int, H: int, S: int, D: int, mult: float = 1.0):
    """Q, K, V bit patterns for an ad-hoc shape (edge-case tests)."""
    shape = (B, H, S, D)
    return tuple(normal_bf16(seed, s, shape, mult) for s in (STREAM_Q, STREAM_K, STREAM_V))


def upstream_grad(seed: int, B: int, H: int, S: int, D: int, mult: float = 1.0):
    """dO bit patterns (bf16, N(0,1) * mult) for the backward pass."""
    return normal_bf16(seed, STREAM_DO, (B, H, S, D), mult)
