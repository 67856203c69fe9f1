"""Helpers shared by the GPU parity tests (no GPU work at import time)."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances: max-abs error over the compared elements divided by max |reference|.
TOL_F32 = 1e-4
TOL_BF16_O = 2e-2
TOL_BF16_S = 1e-2


def rel_err(got, ref) -> float:
    got = got.detach().to("cpu", torch.float64).numpy() if hasattr(got, "detach") else got
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    scale = np.abs(ref).max()
    if scale == 0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / scale)


def tol_o(dtype):
    return TOL_F32 if dtype == torch.float32 else TOL_BF16_O


def tol_s(dtype):
    return TOL_F32 if dtype == torch.float32 else TOL_BF16_S


def oracle_on_heads(prob, heads):
    """Run the fp64 oracle on a subset of heads of a Problem (any device).

    Returns (o [.., len(heads), dv], S_T [N, len(heads), dv, dk]) as float64.
    """
    idx = torch.tensor(heads, device=prob.q.device)
    q = prob.q.index_select(-2, idx)
    k = prob.k.index_select(-2, idx)
    v = prob.v.index_select(-2, idx)
    g = prob.log_alpha.index_select(-2, idx)
    b = prob.beta.index_select(-1, idx)
    S0 = None if prob.S0 is None else prob.S0.index_select(1, idx)
    cu = None if prob.cu_seqlens is None else prob.cu_seqlens.cpu().numpy()
    return oracle.fwd(q, k, v, g, b, S0, cu)


_ORACLE_CACHE = {}


def cached_oracle(key, prob, heads):
    """The oracle's (o, S_T) on `heads` of a workload, computed once per test
    session: every engine and every test of the same seeded workload compares
    against the same fp64 run."""
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE[key] = oracle_on_heads(prob, heads)
    return _ORACLE_CACHE[key]
