"""ORACLE -- test infrastructure, not product code.

Block-sparse attention with a key granularity finer than the query one, in
fp64 (numpy): the mask has one entry per (128-query block, key_block-key
block) pair.  Only the tests and the bench's reference leg may use this
module; it shares nothing with the CUDA path.

"Pallas-Triton kernels and kernel auto-tuning" (section "Auto-tuning") tunes
the query and key block sizes of a flash-attention kernel separately; its
best setting has 128-row query blocks and 64-row key blocks.  In a
block-sparse kernel the key block is also the unit the mask switches on and
off ("Writing Pallas Kernels for JAX", section "Designing the Block
Specification": one mask entry per (query block, key block) pair).  The plain
reading of block_k = 64 taken here: the mask is [B][H][S/128][S/key_block],
and for query row i of head (b, h)

    allowed(j) = mask[b][h][i / 128][j / key_block] != 0  and  (not causal or j <= i)

after which the definition of ``oracle.attention`` applies unchanged: the
full length-S score row (-inf where not allowed), its max, exp, sum, the
weighted sum of V, LSE = m + ln l; O = 0 and LSE = -inf for a row with no
allowed key (with key blocks of 64 keys this can happen inside a query block
that has live entries, under causal).

Each row is written out with numpy (one matrix product per chunk of rows as
the only library primitive).  Pinned by tests/test_oracle_keyblocks_pins.py:
a key_block = 64 mask that repeats a 128-key mask reduces to the pinned
oracle.attention; brute force with math.exp/math.fsum on tiny shapes; torch
float64 SDPA with the expanded boolean mask.
"""
from __future__ import annotations

import numpy as np

QBLOCK = 128
_mutation = 0
KB_MUTATIONS = {1: "key blocks indexed at the query granularity",
                2: "causal limit taken at the block, not the element"}


def set_kb_mutation(m: int) -> None:
    """Plant mistake number m (0 = none).  Tests only."""
    global _mutation
    _mutation = int(m)


def _f64(x):
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if x.dtype == np.float64:
        return x
    raise TypeError("expected uint16 bf16 bit patterns or float64")


def allowed_rows(mask_bh, rows_i, S: int, key_block: int, causal: bool) -> np.ndarray:
    """allowed[i, j] for the given query rows of one (batch, head)."""
    j = np.arange(S)
    kb = j // (QBLOCK if _mutation == 1 else key_block)
    qb = rows_i // QBLOCK
    a = mask_bh[qb[:, None], kb[None, :]] != 0
    if causal:
        if _mutation == 2:
            a &= (kb[None, :] * key_block) <= (qb[:, None] * QBLOCK)
        else:
            a &= j[None, :] <= rows_i[:, None]
    return a


def attention_kb(q, k, v, mask, scale: float, causal: bool = False, key_block: int = 64,
                 rows=None, chunk: int = 256):
    """Exact block-sparse attention with key blocks of `key_block` keys.

    q, k, v: [B][H][S][D] bf16 bit patterns (uint16) or float64.  mask: uint8
    [B][H][S/128][S/key_block].  rows: flat row ids (b*H + h)*S + i, or None
    for every row.  Returns (O [n][D], LSE [n]) float64, reshaped to
    [B][H][S][D] / [B][H][S] when rows is None."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    mask = np.asarray(mask, dtype=np.uint8)
    B, H, S, D = q.shape
    if S % QBLOCK or S % key_block:
        raise ValueError("S must be a multiple of 128 and of key_block")
    if mask.shape != (B, H, S // QBLOCK, S // key_block):
        raise ValueError(f"mask shape {mask.shape} != {(B, H, S // QBLOCK, S // key_block)}")
    full = rows is None
    if full:
        rows = np.arange(B * H * S, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    O = np.empty((rows.size, D))
    L = np.empty(rows.size)
    bh_of = rows // S
    for bh in np.unique(bh_of):
        b, h = divmod(int(bh), H)
        sel = np.flatnonzero(bh_of == bh)
        for c0 in range(0, sel.size, chunk):
            idx = sel[c0:c0 + chunk]
            ri = rows[idx] - bh * S
            allowed = allowed_rows(mask[b, h], ri, S, key_block, causal)
            s = np.where(allowed, float(scale) * (q[b, h, ri] @ k[b, h].T), -np.inf)
            m = s.max(axis=1)
            live = np.isfinite(m)
            w = np.where(allowed, np.exp(s - np.where(live, m, 0.0)[:, None]), 0.0)
            l = w.sum(axis=1)
            O[idx] = np.where(live[:, None], (w @ v[b, h]) / np.where(live, l, 1.0)[:, None], 0.0)
            L[idx] = np.where(live, m + np.log(np.where(live, l, 1.0)), -np.inf)
    if full:
        return O.reshape(B, H, S, D), L.reshape(B, H, S)
    return O, L


def csr_kb(mask, causal: bool = False, key_block: int = 64):
    """Per query block, the ascending live key blocks (key_block keys each);
    under causal a key block is kept when its first key is <= the query
    block's last row.  (row_ptr int32, col_idx int32)."""
    mask = np.asarray(mask, dtype=np.uint8)
    B, H, nbq, nbk = mask.shape
    row_ptr = [0]
    cols = []
    for b in range(B):
        for h in range(H):
            for qb in range(nbq):
                for kb in range(nbk):
                    if mask[b, h, qb, kb] and (not causal or kb * key_block <= qb * QBLOCK + QBLOCK - 1):
                        cols.append(kb)
                row_ptr.append(len(cols))
    return np.asarray(row_ptr, dtype=np.int32), np.asarray(cols, dtype=np.int32)
