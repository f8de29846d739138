"""ORACLE -- test infrastructure, not product code.

Gradients of exact block-sparse attention, in fp64 (numpy), and the
transposed plan (per key block, the live query blocks).  Only the tests and
the bench's reference leg may use this module; it shares nothing with the
CUDA path.

"Writing Pallas Kernels for JAX: Stepping Outside the XLA Safety Net"
(section "The Empathy of the Void") notes that a hand-written attention
kernel needs hand-written gradient definitions.  The definition used here is
the derivative of the forward operation of the same article (sections
"Designing the Block Specification" and "Writing the Kernel Logic: Load,
Compute, Store"), made exact across key blocks as in "Pallas-Triton kernels
and kernel auto-tuning" (section "Flash Attention").  For one (batch, head),
with allowed(i, j) the block mask ANDed with the causal restriction:

    s_ij  = scale * q_i . k_j        (-inf where not allowed)
    P_ij  = exp(s_ij - max_j s_ij) / sum_j exp(...)   (0 where not allowed;
                                                       rows with no allowed key: P = 0)
    O_i   = sum_j P_ij v_j
    dP_ij = dO_i . v_j
    Dl_i  = sum_j P_ij dP_ij         (= dO_i . O_i)
    dS_ij = P_ij (dP_ij - Dl_i)
    dQ_i  = scale * sum_j dS_ij k_j
    dK_j  = scale * sum_i dS_ij q_i
    dV_j  = sum_i P_ij dO_i

Each step is written out with numpy matrix products as the only library
primitive; there is no blocking and no reordering beyond the formulas above.
Pinned by tests/test_oracle_bwd_pins.py (finite differences of the forward
oracle, torch float64 autograd, closed forms, invariants, planted mistakes).
"""
from __future__ import annotations

import numpy as np

BLOCK = 128

# Planted mistakes (test-only): each must make at least one pin fail.
BWD_MUTATIONS = {
    1: "Dl term dropped from dS",
    2: "dV uses P instead of its transpose",
    3: "scale missing from dQ",
    4: "dK built from dS without transposing",
    5: "dP uses K in place of V",
    6: "sign of dS flipped",
    7: "causal restriction ignored in the gradients",
}
_mutation = 0


def set_bwd_mutation(m: int) -> None:
    """Plant mistake number m (0 = none).  Tests only."""
    global _mutation
    _mutation = int(m)


def _as_f64(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) or float64 values -> float64."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if x.dtype == np.float64:
        return x
    raise TypeError("expected uint16 bf16 bit patterns or float64")


def allowed_matrix(mask_bh: np.ndarray, S: int, causal: bool) -> np.ndarray:
    """allowed[i, j] for one (batch, head): the block mask, ANDed with j <= i under causal."""
    nb = S // BLOCK
    assert mask_bh.shape == (nb, nb)
    allowed = np.repeat(np.repeat(mask_bh != 0, BLOCK, axis=0), BLOCK, axis=1)
    if causal and _mutation != 7:
        allowed &= np.tril(np.ones((S, S), dtype=bool))
    return allowed


def _head(q, k, v, do, allowed, scale, bounds, o_bf16=True, acc_mult=1):
    """One (batch, head): the formulas of the module docstring, in order."""
    s = scale * (q @ k.T)
    s = np.where(allowed, s, -np.inf)
    live = allowed.any(axis=1)
    m = np.where(live, s.max(axis=1, initial=-np.inf), 0.0)
    e = np.where(allowed, np.exp(s - m[:, None]), 0.0)
    l = e.sum(axis=1)
    P = np.where(live[:, None], e / np.where(live, l, 1.0)[:, None], 0.0)
    O = P @ v
    dP = do @ (k.T if _mutation == 5 else v.T)
    Dl = (P * dP).sum(axis=1)
    if _mutation == 1:
        dS = P * dP
    else:
        dS = P * (dP - Dl[:, None])
    if _mutation == 6:
        dS = -dS
    dq = (1.0 if _mutation == 3 else scale) * (dS @ k)
    dk = scale * ((dS if _mutation == 4 else dS.T) @ q)
    dv = (P if _mutation == 2 else P.T) @ do
    if not bounds:
        return dq, dk, dv, None
    return dq, dk, dv, _bounds(q, k, v, do, allowed, scale, s, P, O, dP, dS, m, l, o_bf16,
                               acc_mult)


# Error model of a kernel that computes the gradients this way (it is the
# arithmetic of the CUDA backward pass, stated here so the bound can be
# checked by reading):
#   * Q, K, V, dO are bf16 inputs, used exactly;
#   * S = Q K^T and dP = dO V^T come from the tensor core in fp32 (products
#     exact, D additions);
#   * P is recomputed as 2^(S scale log2 e - LSE log2 e) in fp32 with a
#     hardware exp2 approximation, from the given fp32 LSE;
#   * Dl = dO . O in fp32 over the given O (bf16 or fp32);
#   * dS = P (dP - Dl) in fp32;
#   * P and dS are rounded to bf16 (round to nearest) as tensor-core operands;
#   * dV = P^T dO, dK = dS^T Q, dQ = dS K accumulate in fp32 over every live
#     row (dV, dK) or key (dQ), then dK and dQ are multiplied by scale.
U_BF16 = 2.0 ** -8    # unit roundoff of bf16 (8 significant bits, round to nearest)
U_F32 = 2.0 ** -24    # unit roundoff of fp32
ADD_F32 = 2.0 ** -23  # one fp32 addition that may truncate instead of rounding
# Relative error of the hardware exp2 approximation: a deliberately loose
# bound (the approximation is accurate to a few fp32 ulps, ~2^-22); any value
# in between changes the bound by less than 1 %.
EXP2_REL = 2.0 ** -16
LOG2E = 1.0 / np.log(2.0)
# P below fp32's normal range is flushed to zero by the kernel's exp2; each
# such P is off by at most 2^-126, which this absolute term covers for any
# sum of up to 2^20 of them times |values| <= 2^6.
ABS_FLOOR = 2.0 ** -100


def _bounds(q, k, v, do, allowed, scale, s, P, O, dP, dS, m, l, o_bf16, acc_mult):
    """Per-element bounds on |kernel - exact| for (dQ, dK, dV) of one head,
    first order in the roundings of the error model above, times (1 + 2^-7)
    for the neglected products of two rounding errors."""
    D = q.shape[1]
    aq, ak, av, ado = np.abs(q), np.abs(k), np.abs(v), np.abs(do)
    sl = abs(scale) * LOG2E
    # error of the exponent x = S sl - LSE log2 e: the S product (D additions),
    # the fused multiply-add and the fp32 LSE (stored and converted)
    live = allowed.any(axis=1)
    lse2 = np.where(live, (m + np.log(np.where(live, l, 1.0))) * LOG2E, 0.0)
    x_abs = np.where(allowed, np.abs(s) * LOG2E, 0.0)
    dx = sl * D * ADD_F32 * (aq @ ak.T) + 4 * U_F32 * (x_abs + np.abs(lse2)[:, None])
    eps_p = np.where(allowed, np.log(2.0) * dx + EXP2_REL, 0.0)   # relative error of P
    # dP (D additions) and Dl (O's storage rounding and D additions)
    u_o = U_BF16 if o_bf16 else U_F32
    E = np.abs(do * O).sum(axis=1)
    ddp = D * ADD_F32 * (ado @ av.T)
    ddl = (u_o + D * ADD_F32) * E
    # dS before and after its bf16 rounding
    ads = np.abs(dS)
    dds = (U_BF16 + eps_p + 2 * U_F32) * ads + P * (ddp + ddl[:, None])
    # accumulation lengths: live rows per key (dV, dK), live keys per row (dQ)
    n_col = acc_mult * allowed.sum(axis=0).astype(np.float64)
    n_row = allowed.sum(axis=1).astype(np.float64)
    g_col = n_col * ADD_F32
    g_row = n_row * ADD_F32
    bv = (U_BF16 + g_col[:, None]) * (P.T @ ado) + (eps_p * P).T @ ado
    bk = abs(scale) * (dds.T @ aq + (g_col + U_F32)[:, None] * (ads.T @ aq))
    bq = abs(scale) * (dds @ ak + (g_row + U_F32)[:, None] * (ads @ ak))
    slack = 1.0 + 2.0 ** -7
    return tuple(slack * b + ABS_FLOOR for b in (bq, bk, bv))


def attention_bwd(q, k, v, do, mask, scale: float, causal: bool = False, heads=None,
                  bounds: bool = False, o_bf16: bool = True, acc_mult: int = 1):
    """Gradients (dQ, dK, dV) of exact block-sparse attention, fp64.

    q, k, v, do: [B][H][S][D] as bf16 bit patterns (uint16) or float64.
    mask: uint8 [B][H][S/128][S/128].  heads: iterable of (b, h) to compute,
    or None for all.  Returns float64 arrays [B][H][S][D] (heads not computed
    are NaN); with bounds=True also a tuple of per-element error bounds
    (same shapes) for a kernel computing with the error model of ``_bounds``
    (o_bf16: the O it is given was rounded to bf16, else to fp32;
    acc_mult: dK and dV rows accumulate over that many heads' live rows).
    """
    q, k, v, do = (_as_f64(x) for x in (q, k, v, do))
    mask = np.asarray(mask, dtype=np.uint8)
    B, H, S, D = q.shape
    for x in (k, v, do):
        if x.shape != q.shape:
            raise ValueError("q, k, v, do shapes differ")
    if S % BLOCK:
        raise ValueError("S must be a multiple of 128")
    if mask.shape != (B, H, S // BLOCK, S // BLOCK):
        raise ValueError("mask shape does not match")
    out = [np.full(q.shape, np.nan) for _ in range(3)]
    bnd = [np.full(q.shape, np.nan) for _ in range(3)] if bounds else None
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    for b, h in heads:
        allowed = allowed_matrix(mask[b, h], S, causal)
        dq, dk, dv, bb = _head(q[b, h], k[b, h], v[b, h], do[b, h], allowed, float(scale), bounds,
                               o_bf16=o_bf16, acc_mult=acc_mult)
        out[0][b, h], out[1][b, h], out[2][b, h] = dq, dk, dv
        if bounds:
            for t in range(3):
                bnd[t][b, h] = bb[t]
    if bounds:
        return tuple(out), tuple(bnd)
    return tuple(out)


def csc(mask, causal: bool = False):
    """Per key block, the ascending live query blocks: (col_ptr int32, row_idx int32).

    Entry (b, h, kb) lists qb with mask[b, h, qb, kb] != 0 (and qb >= kb under
    causal), in ascending qb; col_ptr has B*H*nb + 1 entries.
    """
    mask = np.asarray(mask, dtype=np.uint8)
    B, H, nb, nb2 = mask.shape
    if nb != nb2:
        raise ValueError("mask must be [B][H][nb][nb]")
    col_ptr = [0]
    rows = []
    for b in range(B):
        for h in range(H):
            for kb in range(nb):
                for qb in range(nb):
                    if mask[b, h, qb, kb] and (not causal or qb >= kb):
                        rows.append(qb)
                col_ptr.append(len(rows))
    return np.asarray(col_ptr, dtype=np.int32), np.asarray(rows, dtype=np.int32)


def attention_bwd_gqa(q, k, v, do, mask, scale: float, causal: bool = False,
                      bounds: bool = False, o_bf16: bool = True):
    """Gradients for grouped-query attention, fp64: q, do [B][H][S][D]; k, v
    [B][Hkv][S][D] (query head h attends with K/V head h // (H // Hkv)); mask
    [B][H][nb][nb] or [B][1][nb][nb] shared by the heads.

    The gradients of attention on K and V with each head repeated H // Hkv
    times (attention_bwd), with dK and dV of each K/V head summed over the
    query heads of its group (the chain rule through the repetition); with
    bounds=True the per-element bounds are summed the same way, each with the
    accumulation length of the whole group (the kernel adds all g heads' terms
    into one fp32 sum)."""
    q, k, v, do = (_as_f64(x) for x in (q, k, v, do))
    B, H, S, D = q.shape
    Hkv = k.shape[1]
    if H % Hkv:
        raise ValueError("H must be a multiple of the K/V heads")
    g = H // Hkv
    k_rep, v_rep = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    mask = np.asarray(mask, dtype=np.uint8)
    if mask.shape[1] == 1 and H > 1:
        mask = np.broadcast_to(mask, (B, H) + mask.shape[2:])
    res = attention_bwd(q, k_rep, v_rep, do, mask, scale, causal, bounds=bounds, o_bf16=o_bf16,
                        acc_mult=g)

    def fold(x):
        return x.reshape(B, Hkv, g, S, D).sum(axis=2)

    if bounds:
        (dq, dk, dv), (bq, bk, bv) = res
        return (dq, fold(dk), fold(dv)), (bq, fold(bk), fold(bv))
    dq, dk, dv = res
    return dq, fold(dk), fold(dv)
