"""Helpers shared by the GPU parity tests (comparison and data movement only)."""
from __future__ import annotations

import numpy as np

# Tolerances of the forward pass against the fp64 oracle (fp32 O):
# max |dO| <= 1e-2, mean |dO| <= 1e-3, |dLSE| <= 1e-3; -inf LSE rows and
# O = 0 rows must match exactly.
MAX_O, MEAN_O, MAX_LSE = 1e-2, 1e-3, 1e-3


def to_dev(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp at |x| (the extra error of rounding an exact O to bf16)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 8), 0.0)


def compare(o_gpu, lse_gpu, O_ref, L_ref, out_bf16: bool = False):
    """Returns (ok, report) for one comparison, element by element."""
    o = np.asarray(o_gpu, dtype=np.float64)
    l = np.asarray(lse_gpu, dtype=np.float64)
    rep = {}
    if not np.all(np.isfinite(o)):
        return False, {"nonfinite_O": int((~np.isfinite(o)).sum())}
    ninf_ref = np.isneginf(L_ref)
    ninf_gpu = np.isneginf(l)
    if not np.array_equal(ninf_ref, ninf_gpu):
        return False, {"lse_inf_mismatch": int((ninf_ref != ninf_gpu).sum())}
    dead = ninf_ref
    if dead.any() and not np.all(o[dead] == 0.0):
        return False, {"dead_rows_nonzero": int((o[dead] != 0).any(axis=-1).sum())}
    err = np.abs(o - O_ref)
    tol_max = MAX_O
    tol_mean = MEAN_O
    if out_bf16:
        hu = half_ulp_bf16(O_ref)
        tol_max_arr = MAX_O + hu
        rep["max_excess"] = float((err - tol_max_arr).max())
        ok_max = bool(np.all(err <= tol_max_arr))
        tol_mean = MEAN_O + float(hu.mean())
    else:
        ok_max = bool(err.max() <= tol_max)
    live = ~dead
    dl = np.abs(l[live] - L_ref[live]) if live.any() else np.zeros(1)
    rep.update(max_dO=float(err.max()), mean_dO=float(err.mean()), max_dLSE=float(dl.max()),
               rows=int(l.size), dead_rows=int(dead.sum()))
    ok = ok_max and err.mean() <= tol_mean and dl.max() <= MAX_LSE
    return bool(ok), rep
