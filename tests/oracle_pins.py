"""Pins for the fp64 KDA oracle: facts fixed by the pages and by mathematics.

Each pin takes an implementation ``impl(q, k, v, log_alpha, beta, S0, erase)``
for ONE head (q, k, log_alpha [T, dk]; v [T, dv]; beta [T]; S0 in the memory
layout [dv, dk] or None) returning ``(o [T, dv], S_T [dv, dk] or None)`` and
returns a relative error.  A pin holds when its error is below ``TOL``.

The pins are chosen so that a plausible slip anywhere in the recurrence (a
dropped decay, the erase applied before the decay, a flipped sign, a read of the
pre-update state, a transposed state index, the gate on the wrong axis, beta in
the wrong place, the gate of the wrong token) breaks at least one of them;
``test_oracle_pins.py::test_planted_mistakes_are_caught`` checks exactly that.
"""
from __future__ import annotations

import numpy as np

import oracle

TOL = 1e-11


def unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def relerr(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(np.abs(b).max(), 1e-300)
    return float(np.abs(a - b).max() / scale)


def random_head(rng, T, dk, dv, la=(-0.7, -0.01), beta_range=(0.05, 0.95), s0=0.3):
    q = unit(rng.standard_normal((T, dk)))
    k = unit(rng.standard_normal((T, dk)))
    v = rng.standard_normal((T, dv))
    g = rng.uniform(la[0], la[1], (T, dk))
    b = rng.uniform(beta_range[0], beta_range[1], T)
    S0 = None if s0 is None else s0 * rng.standard_normal((dv, dk))
    return q, k, v, g, b, S0


def orthonormal_rows(rng, n, d):
    """n <= d orthonormal vectors of length d (rows of a random orthogonal matrix)."""
    m, _ = np.linalg.qr(rng.standard_normal((d, d)))
    return m.T[:n].copy()


# ---------------------------------------------------------------- adapters

def c_oracle(plant=0):
    """Adapter: the C oracle for one head, optionally with a planted mistake."""
    def impl(q, k, v, g, b, S0, erase=True):
        T, dk = q.shape
        dv = v.shape[1]
        o, ST = oracle.fwd(q.reshape(T, 1, dk), k.reshape(T, 1, dk), v.reshape(T, 1, dv),
                           g.reshape(T, 1, dk), b.reshape(T, 1),
                           None if S0 is None else S0.reshape(1, 1, dv, dk),
                           cu_seqlens=np.array([0, T]), erase=erase, plant=plant)
        return o[:, 0, :], ST[0, 0]
    return impl


def bruteforce_impl(q, k, v, g, b, S0, erase=True):
    if not erase:
        raise NotImplementedError
    o, S = oracle.bruteforce(q, k, v, g, b, None if S0 is None else S0.T)
    return o, S.T


def expanded_impl(q, k, v, g, b, S0, erase=True):
    if not erase:
        raise NotImplementedError
    return oracle.expanded_outputs(q, k, v, g, b, None if S0 is None else S0.T), None


# ---------------------------------------------------------------- pins

def pin_identity_transition(impl, seed=1):
    """alpha = 1 and beta = 0: the state passes through unchanged and every
    output reads the initial state, o_t = S_0^T q_t ("完全拆解": beta = 0 means
    forget only, no write; alpha = 1 means no forgetting)."""
    rng = np.random.default_rng(seed)
    q, k, v, _, _, S0 = random_head(rng, 9, 6, 5)
    g = np.zeros_like(q)
    b = np.zeros(q.shape[0])
    o, ST = impl(q, k, v, g, b, S0)
    err = relerr(o, q @ S0.T)          # S0 memory is [dv, dk]: o = mem @ q
    if ST is not None:
        err = max(err, relerr(ST, S0))
    return err


def pin_unit_key_recall(impl, seed=2):
    """||k_t|| = 1 and beta_t = 1: after the update S_t^T k_t = v_t exactly, for
    any gate ("完全拆解": with a unit key and beta = 1 the old projection along
    k_t is removed completely and the new value written)."""
    rng = np.random.default_rng(seed)
    q, k, v, g, _, S0 = random_head(rng, 6, 8, 7)
    b = np.ones(q.shape[0])
    err = 0.0
    for t in range(1, q.shape[0] + 1):
        _, ST = impl(q[:t], k[:t], v[:t], g[:t], b[:t], S0)
        if ST is None:
            return 0.0
        err = max(err, relerr(ST @ k[t - 1], v[t - 1]))
    return err


def pin_orthonormal_keys_linear_attention(impl, seed=3):
    """alpha = 1, beta = 1, S_0 = 0 and mutually orthonormal keys: the erase
    term vanishes (the decayed state has no component along a new orthogonal
    key) and KDA reduces to linear attention, o_t = sum_{i<=t} (q_t.k_i) v_i
    ("Kimi K3 的 KDA" section 2; "完全拆解", linear attention)."""
    rng = np.random.default_rng(seed)
    T, d = 7, 8
    k = orthonormal_rows(rng, T, d)
    q = unit(rng.standard_normal((T, d)))
    v = rng.standard_normal((T, 6))
    o, _ = impl(q, k, v, np.zeros((T, d)), np.ones(T), None)
    ref = np.tril(q @ k.T) @ v
    return relerr(o, ref)


def pin_no_erase_linear_attention(impl, seed=4):
    """No-erase mode, alpha = 1, beta = 1: o_t = sum_{i<=t} (q_t.k_i) v_i for
    arbitrary keys (the linear-attention closed form)."""
    rng = np.random.default_rng(seed)
    q, k, v, _, _, _ = random_head(rng, 9, 6, 5)
    T, d = q.shape
    o, _ = impl(q, k, v, np.zeros((T, d)), np.ones(T), None, erase=False)
    return relerr(o, np.tril(q @ k.T) @ v)


def pin_worked_two_token_example(impl, seed=5):
    """The two-token example of "Kimi K3 的 KDA" section 5 (no erase):
    S_2 = a_2 a_1 S_in + a_2 k_1 v_1^T + k_2 v_2^T, with the per-channel gates
    acting as Diag(a) on the key axis; also o_2 = S_2^T q_2."""
    rng = np.random.default_rng(seed)
    q, k, v, g, _, S0 = random_head(rng, 2, 5, 5)
    a1, a2 = np.exp(g[0]), np.exp(g[1])
    Sin = S0.T                                     # logical [dk, dv]
    S2 = (a2 * a1)[:, None] * Sin + a2[:, None] * np.outer(k[0], v[0]) + np.outer(k[1], v[1])
    o, ST = impl(q, k, v, g, np.ones(2), S0, erase=False)
    err = relerr(o[1], S2.T @ q[1])
    if ST is not None:
        err = max(err, relerr(ST, S2.T))
    return err


def pin_worked_example_with_erase(impl, seed=6):
    """Same example with the erase active: when the gate is a scalar per token,
    k_1, k_2 are orthonormal and S_in lives on the orthogonal complement of
    both, the erase removes nothing and the no-erase formula still holds."""
    rng = np.random.default_rng(seed)
    d, dv = 6, 4
    basis = orthonormal_rows(rng, d, d)
    k = basis[:2]
    Sin = sum(np.outer(basis[m], rng.standard_normal(dv)) for m in range(2, d))
    v = rng.standard_normal((2, dv))
    q = unit(rng.standard_normal((2, d)))
    s = rng.uniform(-0.6, -0.05, 2)
    g = np.repeat(s[:, None], d, axis=1)
    a1, a2 = np.exp(s)
    S2 = a2 * a1 * Sin + a2 * np.outer(k[0], v[0]) + np.outer(k[1], v[1])
    o, ST = impl(q, k, v, g, np.ones(2), Sin.T)
    err = relerr(o[1], S2.T @ q[1])
    if ST is not None:
        err = max(err, relerr(ST, S2.T))
    return err


def pin_sgd_step(impl, seed=7, eps=1e-6):
    """The delta rule is one gradient step of size beta on
    L(S) = 1/2 ||S^T k - v||^2 taken from the decayed state ("完全拆解", the
    DeltaNet loss and its gradient step; KDA applies it to Diag(alpha) S).
    The gradient here is a central finite difference -- no formula."""
    rng = np.random.default_rng(seed)
    dk, dv = 5, 5
    q, k, v, g, b, S0 = random_head(rng, 1, dk, dv)
    Sbar = np.exp(g[0])[:, None] * S0.T             # logical [dk, dv]

    def loss(S):
        r = S.T @ k[0] - v[0]
        return 0.5 * float(r @ r)

    grad = np.zeros_like(Sbar)
    for i in range(dk):
        for j in range(dv):
            e = np.zeros_like(Sbar)
            e[i, j] = eps
            grad[i, j] = (loss(Sbar + e) - loss(Sbar - e)) / (2 * eps)
    S1 = Sbar - b[0] * grad
    o, ST = impl(q, k, v, g, b, S0)
    err = relerr(o[0], S1.T @ q[0])
    if ST is not None:
        err = max(err, relerr(ST, S1.T))
    return err


def pin_norm_nonincreasing(impl, seed=8):
    """v = 0, ||k|| = 1, beta in [0, 1], alpha <= 1: each transition has
    eigenvalues in [1 - beta, 1] after the decay, so ||S_t||_F never grows.
    Returns 0 when it holds, else the largest relative growth."""
    rng = np.random.default_rng(seed)
    q, k, _, g, b, S0 = random_head(rng, 10, 6, 6, beta_range=(0.0, 1.0))
    v = np.zeros((10, 6))
    prev = np.linalg.norm(S0)
    worst = 0.0
    for t in range(1, 11):
        _, ST = impl(q[:t], k[:t], v[:t], g[:t], b[:t], S0)
        if ST is None:
            return 0.0
        cur = np.linalg.norm(ST)
        worst = max(worst, (cur - prev) / prev)
        prev = cur
    return max(worst, 0.0)


def pin_bruteforce(impl, seed=9, dk=6, dv=6, T=7):
    """T <= 8: agreement with explicit products of the d_k x d_k transition
    matrices and with the fully expanded output sum."""
    rng = np.random.default_rng(seed)
    q, k, v, g, b, S0 = random_head(rng, T, dk, dv)
    o, ST = impl(q, k, v, g, b, S0)
    ob, Sb = oracle.bruteforce(q, k, v, g, b, S0.T)
    oe = oracle.expanded_outputs(q, k, v, g, b, S0.T)
    err = max(relerr(o, ob), relerr(o, oe))
    if ST is not None:
        err = max(err, relerr(ST, Sb.T))
    return err


# Central differences of a quadratic are exact up to rounding (~1e-16 / eps).
TOLS = {pin_sgd_step: 1e-7}


def tol(pin):
    return TOLS.get(pin, TOL)


# Pins that come from the pages or from mathematics (not self-consistency).
INDEPENDENT_PINS = [
    pin_identity_transition,
    pin_unit_key_recall,
    pin_orthonormal_keys_linear_attention,
    pin_no_erase_linear_attention,
    pin_worked_two_token_example,
    pin_worked_example_with_erase,
    pin_sgd_step,
    pin_norm_nonincreasing,
    pin_bruteforce,
]
