"""KDA oracle -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct CPU implementations of the Kimi Delta Attention
(KDA) operator, used to check the GPU library.  Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  It shares no code with the GPU library and never imports it.

Contents
--------
``fwd`` / ``decode_step``
    ctypes front end of ``kda_oracle.c``: the token-by-token fp64 recurrence
    (decay -> old = Sbar^T k -> erase + write -> read the updated state), as
    written in "Kimi K3 的 KDA" sections 3-4, "Kimi K3" (gentlecold) section 3.2
    and "Kimi Delta Attention 完全拆解" (KDA equations and the decode-order listing).
``bruteforce``
    For tiny T: builds each d_k x d_k transition matrix
    A_t = (I - beta_t k_t k_t^T) Diag(alpha_t) explicitly and iterates
    S_t = A_t S_{t-1} + beta_t k_t v_t^T ("完全拆解", the state-space form in the
    section on why a plain prefix scan is not used).  numpy, independent code.
``expanded_outputs``
    For tiny T: the fully expanded output
    o_t = (A_t...A_1 S_0)^T q_t + sum_{i<=t} beta_i [q_t^T A_t...A_{i+1} k_i] v_i
    ("完全拆解", the expansion in the comparison with GDN; the page's display drops
    beta_i and the S_0 term; both are restored here, since unrolling the
    recurrence S_t = A_t S_{t-1} + beta_t k_t v_t^T produces them).

``gated_rmsnorm``
    The output epilogue of a KDA layer, per (token, head): a head-wise RMSNorm
    over the value channels times a per-channel weight, then the sigmoid output
    gate, y = sigmoid(g) * w * o / sqrt(mean_v(o^2) + eps) ("Kimi K3 模型结构（1）",
    output section: per-head RMSNorm over the 128 channels, sigmoid gate on each
    normalised channel; "Kimi K3" (gentlecold) section 3.2, y = W_o[Sigmoid(W_g x)
    . RMSNorm(o~)]; "完全拆解", the KDA layer's output).  numpy, the definition
    written out.

``short_conv`` / ``prologue``
    The input prologue of a KDA layer: a depthwise causal convolution of
    kernel 4 along the sequence (ShortConv), Swish, and for q and k an L2
    normalisation over the d channels of one (token, head)
    ("Kimi K3 模型结构（1）", parameterisation section: depthwise causal, kernel
    size 4, each token mixed with the previous 3, and the last 3 projected inputs
    of q, k, v cached for decode; "Kimi Delta Attention 完全拆解", the KDA
    layer's forward: q, k = L2Norm(Swish(ShortConv(W x))), v =
    Swish(ShortConv(W_v x)); "Kimi K3" (gentlecold) section 3.3).  numpy,
    token by token, the definition written out.

``verify_tokens`` / ``commit_tokens``
    Speculative-decode verification and commit over K cached draft tokens
    ("Kimi K3 深度拆解" section 9.2), written out as K (or n_accept[n]) calls of
    ``decode_step``; no arithmetic of their own.

Parity status of every function is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "libkda_oracle.so")
# test-only build of the same file with the planted mistakes compiled in
_SO_PLANTS = os.path.join(_BUILD_DIR, "libkda_oracle_plants.so")
_lock = threading.Lock()
_handles = {}

# Planted-mistake codes understood by the test-only build (mutation check).
PLANTS = {
    "no_decay": 1,
    "erase_then_decay": 2,
    "erase_sign": 3,
    "read_before_write": 4,
    "transposed_old": 5,
    "decay_value_axis": 6,
    "beta_on_erase_only": 7,
    "stale_gate": 8,
}


def build(force: bool = False, plants: bool = False) -> str:
    """Compile kda_oracle.c into a shared library with gcc (-O2, OpenMP).  With
    plants=True: the test-only build with the planted mistakes."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    so = _SO_PLANTS if plants else _SO
    if (not force and os.path.exists(so)
            and os.path.getmtime(so) >= os.path.getmtime(_SRC)):
        return so
    tmp = so + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-o", tmp, _SRC, "-lm"] + (["-DKDA_ORACLE_PLANTS"] if plants else [])
    subprocess.run(cmd, check=True)
    os.replace(tmp, so)
    return so


def _lib(plants: bool = False):
    with _lock:
        if plants not in _handles:
            path = build(plants=plants)
            lib = ctypes.CDLL(path)
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_int64)
            ci = ctypes.c_int
            lib.kda_oracle_fwd.restype = ci
            lib.kda_oracle_fwd.argtypes = [dp, dp, dp, dp, dp, dp, lp, ci, ci, ci, ci,
                                           ci, ci, dp, dp]
            lib.kda_oracle_decode_step.restype = ci
            lib.kda_oracle_decode_step.argtypes = [dp, dp, dp, dp, dp, dp, ci, ci, ci, ci, dp]
            lib.kda_oracle_max_threads.restype = ci
            lib.kda_oracle_max_threads.argtypes = []
            _handles[plants] = lib
    return _handles[plants]


def _f64(x) -> np.ndarray:
    """Exact upcast to a contiguous float64 numpy array (accepts torch tensors)."""
    if hasattr(x, "detach"):  # torch tensor: upcast exactly on the CPU
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    """Number of OpenMP threads the oracle runs with."""
    return int(_lib().kda_oracle_max_threads())


def fwd(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, erase: bool = True,
        plant: int = 0):
    """Token-by-token fp64 KDA forward.

    Shapes (either a fixed-length batch or a packed varlen batch):
      q, k, log_alpha : [B, T, H, dk] or [Ttot, H, dk]
      v               : [B, T, H, dv] or [Ttot, H, dv]
      beta            : [B, T, H]     or [Ttot, H]
      S0              : [N, H, dv, dk] (memory layout mem[v][c] = S[c][v]) or None
      cu_seqlens      : [N+1] int offsets into the packed token axis, or None
                        (then N = B and sequence b is tokens b*T..(b+1)*T-1)
    Returns (o, S_T) as float64 arrays, o shaped like v, S_T [N, H, dv, dk].
    """
    q, k, v, g, b = (_f64(x) for x in (q, k, v, log_alpha, beta))
    lead = v.shape[:-2]
    H, dk = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    Ttot = int(np.prod(lead)) if len(lead) else 0
    if cu_seqlens is None:
        if q.ndim == 4:
            Bsz, T = q.shape[0], q.shape[1]
        else:
            Bsz, T = 1, q.shape[0]
        cu = np.arange(Bsz + 1, dtype=np.int64) * T
    else:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
    N = cu.shape[0] - 1
    if int(cu[-1]) != Ttot:
        raise ValueError("cu_seqlens[-1] must equal the number of packed tokens")
    s0 = None if S0 is None else _f64(S0).reshape(N, H, dv, dk)
    o = np.zeros(lead + (H, dv), dtype=np.float64)
    ST = np.zeros((N, H, dv, dk), dtype=np.float64)
    rc = _lib(plants=bool(plant)).kda_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(s0),
                               cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                               N, H, dk, dv, int(bool(erase)), int(plant), _ptr(o), _ptr(ST))
    if rc != 0:
        raise ValueError("kda_oracle_fwd rejected its arguments")
    return o, ST


def decode_step(q, k, v, log_alpha, beta, S):
    """One fp64 decode step for every (session, head).

    q, k, log_alpha [N, H, dk]; v [N, H, dv]; beta [N, H]; S [N, H, dv, dk].
    Returns (o [N, H, dv], S_new); the inputs are not modified.
    """
    q, k, v, g, b = (_f64(x) for x in (q, k, v, log_alpha, beta))
    S = _f64(S).copy()
    N, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((N, H, dv), dtype=np.float64)
    rc = _lib().kda_oracle_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(S),
                                       N, H, dk, dv, _ptr(o))
    if rc != 0:
        raise ValueError("kda_oracle_decode_step rejected its arguments")
    return o, S


def gated_rmsnorm(o, g, weight=None, eps=0.0):
    """y = sigmoid(g) * weight * o / sqrt(mean over the last axis of o^2 + eps).

    o, g: [..., dv] (any leading shape: tokens, heads); weight: [dv] or None
    (ones); eps >= 0.  The mean runs over the value channels of one (token,
    head) only.  Returns float64 of o's shape."""
    o, g = _f64(o), _f64(g)
    w = np.ones(o.shape[-1]) if weight is None else _f64(weight)
    ms = np.mean(o * o, axis=-1, keepdims=True)          # mean square per (token, head)
    with np.errstate(over="ignore"):
        gate = 1.0 / (1.0 + np.exp(-g))                  # sigmoid
    return o / np.sqrt(ms + eps) * w * gate


def short_conv(x, w, conv0=None, cu_seqlens=None, l2norm=False, eps=0.0):
    """ShortConv(4) + Swish (+ L2Norm) of one stream, token by token.

    x: [B, T, H, d] (fixed length) or [Ttot, H, d] with cu_seqlens [N+1];
    w: [H, d, 4] depthwise taps, tap 3 on the current token and taps 0-2 on the
    three before it, oldest first; conv0: [N, 3, H, d] the three inputs before
    each sequence, oldest first, or None (zeros).  Per sequence and channel:
      c_t = sum_{i=0..3} w[i] x_{t-3+i}   (x_{-3..-1} from conv0)
      y_t = c_t * sigmoid(c_t)            (Swish)
    and with l2norm, y_t / sqrt(sum_d y_t^2 + eps) over the d channels of one
    (token, head) (zero where that sum is zero).  Returns (y float64 of x's
    shape, conv_T [N, 3, H, d]: the last three inputs of each sequence, oldest
    first -- with conv0's tail where the sequence has fewer than three)."""
    x, w = _f64(x), _f64(w)
    packed = cu_seqlens is not None
    xs = x if packed else x.reshape((-1,) + x.shape[2:])
    if packed:
        cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
    else:
        T = x.shape[1]
        cu = [b * T for b in range(x.shape[0] + 1)]
    N = len(cu) - 1
    H, d = xs.shape[1], xs.shape[2]
    hist0 = np.zeros((N, 3, H, d)) if conv0 is None else _f64(conv0)
    y = np.zeros(xs.shape, dtype=np.float64)
    conv_T = np.zeros((N, 3, H, d), dtype=np.float64)
    for n in range(N):
        win = [hist0[n, 0], hist0[n, 1], hist0[n, 2]]   # the three inputs before token t
        for t in range(cu[n], cu[n + 1]):
            cur = xs[t]
            c = w[:, :, 0] * win[0] + w[:, :, 1] * win[1] + w[:, :, 2] * win[2] + w[:, :, 3] * cur
            with np.errstate(over="ignore"):
                yt = c / (1.0 + np.exp(-c))              # c * sigmoid(c)
            if l2norm:
                ss = np.sum(yt * yt, axis=-1, keepdims=True) + eps
                yt = np.where(ss > 0, yt / np.sqrt(np.where(ss > 0, ss, 1.0)), 0.0)
            y[t] = yt
            win = [win[1], win[2], cur]
        conv_T[n] = np.stack(win)
    return (y if packed else y.reshape(x.shape)), conv_T


def prologue(xq, xk, xv, wq, wk, wv, conv0=None, cu_seqlens=None, eps=0.0):
    """The input prologue of a KDA layer for the three streams: q and k through
    ShortConv(4), Swish and L2Norm, v through ShortConv(4) and Swish (see
    short_conv).  conv0: [N, 3, 3, H, d] (stream q, k, v; three inputs, oldest
    first) or None.  Returns (q, k, v, conv_T [N, 3, 3, H, d])."""
    outs, states = [], []
    for i, (x, w, norm) in enumerate(((xq, wq, True), (xk, wk, True), (xv, wv, False))):
        y, st = short_conv(x, w, None if conv0 is None else _f64(conv0)[:, i], cu_seqlens,
                           l2norm=norm, eps=eps)
        outs.append(y)
        states.append(st)
    return outs[0], outs[1], outs[2], np.stack(states, axis=1)


def verify_tokens(q, k, v, log_alpha, beta, S):
    """Speculative-decode verification ("Kimi K3 深度拆解" section 9.2): the
    outputs of K draft tokens per session run in order from S, which is not
    changed.  q, k, log_alpha [N, K, H, dk]; v [N, K, H, dv]; beta [N, K, H];
    S [N, H, dv, dk].  The definition written out: K decode steps on a copy of
    S.  Returns o [N, K, H, dv]."""
    q, k, v, g, b = (_f64(x) for x in (q, k, v, log_alpha, beta))
    St = _f64(S)
    N, K = q.shape[:2]
    o = np.zeros(v.shape, dtype=np.float64)
    for t in range(K):
        o[:, t], St = decode_step(q[:, t], k[:, t], v[:, t], g[:, t], b[:, t], St)
    return o


def commit_tokens(q, k, v, log_alpha, beta, S, n_accept=None):
    """The first n_accept[n] draft tokens of session n applied to S (all K when
    n_accept is None): that many decode steps, session by session.  Returns
    the new state [N, H, dv, dk]; the inputs are not modified."""
    q, k, v, g, b = (_f64(x) for x in (q, k, v, log_alpha, beta))
    S = _f64(S).copy()
    N, K = q.shape[:2]
    acc = [K] * N if n_accept is None else \
        [min(max(int(a), 0), K) for a in np.asarray(_f64(n_accept)).reshape(-1)]
    for n in range(N):
        for t in range(acc[n]):
            _, S[n:n + 1] = decode_step(q[n:n + 1, t], k[n:n + 1, t], v[n:n + 1, t],
                                        g[n:n + 1, t], b[n:n + 1, t], S[n:n + 1])
    return S


def bruteforce(q, k, v, log_alpha, beta, S0=None):
    """Single head, tiny T: explicit d_k x d_k transitions.

    q, k, log_alpha [T, dk]; v [T, dv]; beta [T]; S0 logical [dk, dv] or None.
    Returns (o [T, dv], S_T logical [dk, dv]).
    """
    q, k, v, g, b = (_f64(x) for x in (q, k, v, log_alpha, beta))
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else _f64(S0).copy()
    eye = np.eye(dk)
    o = np.zeros((T, dv))
    for t in range(T):
        A = (eye - b[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(g[t]))
        S = A @ S + b[t] * np.outer(k[t], v[t])
        o[t] = S.T @ q[t]
    return o, S


def expanded_outputs(q, k, v, log_alpha, beta, S0=None):
    """Single head, tiny T: o_t from the fully expanded sum over earlier writes.

    o_t = (P_{t,0} S_0)^T q_t + sum_{i<=t} beta_i (q_t^T P_{t,i} k_i) v_i,
    with P_{t,i} = A_t A_{t-1} ... A_{i+1} (identity when i = t) and
    A_j = (I - beta_j k_j k_j^T) Diag(alpha_j).
    """
    q, k, v, g, b = (_f64(x) for x in (q, k, v, log_alpha, beta))
    T, dk = q.shape
    dv = v.shape[1]
    S0 = np.zeros((dk, dv)) if S0 is None else _f64(S0)
    eye = np.eye(dk)
    A = [(eye - b[j] * np.outer(k[j], k[j])) @ np.diag(np.exp(g[j])) for j in range(T)]
    o = np.zeros((T, dv))
    for t in range(T):
        P = eye.copy()          # P_{t,t}
        acc = np.zeros(dv)
        for i in range(t, -1, -1):
            acc += b[i] * (q[t] @ P @ k[i]) * v[i]
            P = P @ A[i]        # becomes P_{t,i-1} = A_t ... A_i
        acc += (P @ S0).T @ q[t]  # P is now A_t ... A_1 (all transitions)
        o[t] = acc
    return o
