"""The fp64 oracle against what the pages and mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as P


@pytest.mark.parametrize("pin", P.INDEPENDENT_PINS, ids=lambda f: f.__name__)
def test_c_oracle_pins(pin):
    assert pin(P.c_oracle()) < P.tol(pin)


# The numpy brute force and the expanded sum are pinned by the same closed forms
# (the pins that need no-erase mode or the final state skip themselves there).
@pytest.mark.parametrize("pin", [P.pin_identity_transition, P.pin_unit_key_recall,
                                 P.pin_orthonormal_keys_linear_attention,
                                 P.pin_worked_example_with_erase, P.pin_sgd_step,
                                 P.pin_norm_nonincreasing],
                         ids=lambda f: f.__name__)
@pytest.mark.parametrize("impl", [P.bruteforce_impl, P.expanded_impl],
                         ids=["bruteforce", "expanded"])
def test_tiny_restatements_pins(pin, impl):
    assert pin(impl) < P.tol(pin)


@pytest.mark.parametrize("name,code", sorted(oracle.PLANTS.items()))
def test_planted_mistakes_are_caught(name, code):
    """Every planted slip in the C oracle breaks at least one independent pin."""
    impl = P.c_oracle(plant=code)
    failures = []
    for pin in P.INDEPENDENT_PINS:
        try:
            err = pin(impl)
        except ValueError:
            continue  # this mistake needs dk == dv; the pin uses other sizes
        if not err < P.tol(pin):
            failures.append(pin.__name__)
    assert failures, f"planted mistake '{name}' passed every pin"


def _rand_packed(rng, lengths, H, dk, dv, s0=True):
    T = int(sum(lengths))
    q = P.unit(rng.standard_normal((T, H, dk)))
    k = P.unit(rng.standard_normal((T, H, dk)))
    v = rng.standard_normal((T, H, dv))
    g = rng.uniform(-0.5, -0.001, (T, H, dk))
    b = 1 / (1 + np.exp(-rng.standard_normal((T, H))))
    S0 = 0.1 * rng.standard_normal((len(lengths), H, dv, dk)) if s0 else None
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return q, k, v, g, b, S0, cu


def test_segment_split_equals_whole():
    """Running T1 tokens, then T2 tokens from the returned state, equals one run
    over T1 + T2 ("完全拆解", validation advice: two segments with a nonzero
    initial state against the whole).  The oracle is sequential: bit-identical."""
    rng = np.random.default_rng(11)
    q, k, v, g, b, S0, _ = _rand_packed(rng, [50], 3, 8, 6)
    o, ST = oracle.fwd(q, k, v, g, b, S0, np.array([0, 50]))
    o1, S1 = oracle.fwd(q[:20], k[:20], v[:20], g[:20], b[:20], S0, np.array([0, 20]))
    o2, S2 = oracle.fwd(q[20:], k[20:], v[20:], g[20:], b[20:], S1, np.array([0, 30]))
    assert np.array_equal(np.concatenate([o1, o2]), o)
    assert np.array_equal(S2, ST)


def test_varlen_isolation():
    """Packing other sequences next to a sequence, or reordering them, leaves
    its output and final state bit-identical ("完全拆解", validation advice on
    varlen batches)."""
    rng = np.random.default_rng(12)
    lengths = [5, 17, 1, 9]
    q, k, v, g, b, S0, cu = _rand_packed(rng, lengths, 2, 6, 6)
    o, ST = oracle.fwd(q, k, v, g, b, S0, cu)
    for i, L in enumerate(lengths):
        sl = slice(cu[i], cu[i + 1])
        oi, Si = oracle.fwd(q[sl], k[sl], v[sl], g[sl], b[sl], S0[i:i + 1], np.array([0, L]))
        assert np.array_equal(oi, o[sl])
        assert np.array_equal(Si[0], ST[i])
    perm = [2, 0, 3, 1]
    parts = [slice(cu[i], cu[i + 1]) for i in perm]
    cat = lambda x: np.concatenate([x[s] for s in parts])
    cu_p = np.concatenate([[0], np.cumsum([lengths[i] for i in perm])])
    op, Sp = oracle.fwd(cat(q), cat(k), cat(v), cat(g), cat(b), S0[perm], cu_p)
    assert np.array_equal(Sp, ST[perm])
    assert np.array_equal(op, cat(o))


def test_empty_sequences():
    """Zero-length sequences return their initial state and produce no output."""
    rng = np.random.default_rng(13)
    q, k, v, g, b, S0, cu = _rand_packed(rng, [0, 4, 0], 2, 4, 4)
    o, ST = oracle.fwd(q, k, v, g, b, S0, cu)
    assert np.array_equal(ST[0], S0[0]) and np.array_equal(ST[2], S0[2])
    assert o.shape == (4, 2, 4)


def test_prefill_equals_decode_steps():
    """The prefill path and T single-token decode steps give the same outputs
    and state: the output of a token reads the state after its own write in
    both ("完全拆解": the parallel and recurrent paths must share the causal
    mask)."""
    rng = np.random.default_rng(14)
    q, k, v, g, b, S0, _ = _rand_packed(rng, [12], 3, 8, 8)
    o, ST = oracle.fwd(q, k, v, g, b, S0, np.array([0, 12]))
    S = S0.copy()
    for t in range(12):
        ot, S = oracle.decode_step(q[t][None], k[t][None], v[t][None], g[t][None],
                                   b[t][None], S)
        np.testing.assert_allclose(ot[0], o[t], rtol=0, atol=1e-13)
    np.testing.assert_allclose(S, ST, rtol=0, atol=1e-13)


def test_scalar_gate_is_gated_deltanet():
    """All channels of alpha_t equal: KDA reduces to Gated DeltaNet,
    S_t = a_t (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T ("完全拆解", GDN and
    the degenerate cases of KDA).  GDN is written here as its own loop."""
    rng = np.random.default_rng(15)
    T, d, dv = 9, 6, 5
    q, k, v, _, b, S0 = P.random_head(rng, T, d, dv)
    s = rng.uniform(-0.5, -0.01, T)
    g = np.repeat(s[:, None], d, axis=1)
    S = S0.T.copy()
    ref = np.zeros((T, dv))
    for t in range(T):
        S = np.exp(s[t]) * (S - b[t] * np.outer(k[t], k[t] @ S)) + b[t] * np.outer(k[t], v[t])
        ref[t] = S.T @ q[t]
    o, ST = P.c_oracle()(q, k, v, g, b, S0)
    assert P.relerr(o, ref) < P.TOL and P.relerr(ST, S.T) < P.TOL


def test_unit_gate_is_deltanet():
    """alpha = 1: KDA reduces to DeltaNet, S_t = S_{t-1} - b_t k_t (S_{t-1}^T k_t - v_t)^T
    ("完全拆解", the DeltaNet update written as a gradient step)."""
    rng = np.random.default_rng(16)
    T, d, dv = 9, 7, 4
    q, k, v, _, b, S0 = P.random_head(rng, T, d, dv)
    S = S0.T.copy()
    ref = np.zeros((T, dv))
    for t in range(T):
        S = S - b[t] * np.outer(k[t], S.T @ k[t] - v[t])
        ref[t] = S.T @ q[t]
    o, ST = P.c_oracle()(q, k, v, np.zeros((T, d)), b, S0)
    assert P.relerr(o, ref) < P.TOL and P.relerr(ST, S.T) < P.TOL


def test_segment_map_is_affine_and_composes():
    """For a fixed segment the map S_in -> S_out is affine, S_out = M S_in + S~
    (M and S~ depending only on the segment's tokens), and two segment maps
    compose as (M2, b2) o (M1, b1) = (M2 M1, M2 b1 + b2) ("Kimi K3" (gentlecold)
    section 3.6, KDA context parallelism)."""
    rng = np.random.default_rng(17)
    d = 5
    q, k, v, g, b, _ = P.random_head(rng, 14, d, d)

    def seg(lo, hi, S_in_logical):
        _, ST = P.c_oracle()(q[lo:hi], k[lo:hi], v[lo:hi], g[lo:hi], b[lo:hi],
                             S_in_logical.T)
        return ST.T

    def affine(lo, hi):
        b0 = seg(lo, hi, np.zeros((d, d)))
        # the linear part acts on the key axis: column j of S_in maps
        # independently, so M is recovered from unit inputs e_i e_j^T.
        M = np.zeros((d, d))
        for i in range(d):
            E = np.zeros((d, d))
            E[i, 0] = 1.0
            M[:, i] = (seg(lo, hi, E) - b0)[:, 0]
        return M, b0

    X = rng.standard_normal((d, d))
    M1, b1 = affine(0, 6)
    M2, b2 = affine(6, 14)
    assert P.relerr(seg(0, 6, X), M1 @ X + b1) < 1e-12
    M12, b12 = M2 @ M1, M2 @ b1 + b2
    whole = seg(0, 14, X)
    assert P.relerr(whole, M12 @ X + b12) < 1e-12
    Mw, bw = affine(0, 14)
    assert P.relerr(Mw, M12) < 1e-12 and P.relerr(bw, b12) < 1e-12


def test_rejects_bad_arguments():
    rng = np.random.default_rng(18)
    q, k, v, g, b, S0, cu = _rand_packed(rng, [3, 3], 1, 4, 4)
    with pytest.raises(ValueError):
        oracle.fwd(q, k, v, g, b, S0, np.array([0, 7, 6]))      # decreasing offsets
    with pytest.raises(ValueError):
        oracle.fwd(q, k, v, g, b, S0, np.array([0, 3, 5]))      # does not cover all tokens


def test_verify_and_commit_compose_like_a_prefill():
    """The draft-token verify/commit helpers against the prefill recurrence on
    the same tokens: verify's outputs are the prefill outputs of the K tokens
    from S, commit(all) is the prefill's final state, commit(0) leaves S, and
    committing a tokens equals a prefill over those a tokens."""
    rng = np.random.default_rng(11)
    N, K, H, d = 3, 5, 2, 8
    q = rng.standard_normal((N, K, H, d)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((N, K, H, d)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((N, K, H, d))
    g = rng.uniform(-0.5, -0.01, (N, K, H, d))
    b = rng.uniform(0.1, 0.9, (N, K, H))
    S = rng.standard_normal((N, H, d, d)) * 0.1
    o = oracle.verify_tokens(q, k, v, g, b, S)
    o_ref, S_ref = oracle.fwd(q, k, v, g, b, S)          # [B=N, T=K, H, d] prefill form
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.commit_tokens(q, k, v, g, b, S), S_ref, rtol=1e-12,
                               atol=1e-12)
    np.testing.assert_array_equal(oracle.commit_tokens(q, k, v, g, b, S, [0, 0, 0]), S)
    acc = [2, 0, 5]
    Sc = oracle.commit_tokens(q, k, v, g, b, S, acc)
    for n, a in enumerate(acc):
        if a:
            _, Sa = oracle.fwd(q[n:n + 1, :a], k[n:n + 1, :a], v[n:n + 1, :a], g[n:n + 1, :a],
                               b[n:n + 1, :a], S[n:n + 1])
            np.testing.assert_allclose(Sc[n:n + 1], Sa, rtol=1e-12, atol=1e-12)
        else:
            np.testing.assert_array_equal(Sc[n], S[n])


# ---------------------------------------------------------------- output epilogue
# y = sigmoid(g) * w * o / sqrt(mean_v(o^2) + eps), per (token, head) ("Kimi K3 模型
# 结构（1）", output section: head-wise RMSNorm over the value channels and a sigmoid
# gate on each normalised channel).  Each pin below is fixed by the definition
# or by arithmetic done by hand, not by the oracle's own formula.

def test_gated_rmsnorm_worked_example():
    """o = (3, 4), g = (0, ln 3), w = (1, 2), eps = 1/2, worked by hand: the
    mean square is (9 + 16) / 2 = 12.5, plus eps is 13; sigmoid(0) = 1/2 and
    sigmoid(ln 3) = 3 / 4; so y = (3 * 1 * 1/2, 4 * 2 * 3/4) / sqrt(13)."""
    y = oracle.gated_rmsnorm(np.array([3.0, 4.0]), np.array([0.0, np.log(3.0)]),
                             np.array([1.0, 2.0]), eps=0.5)
    assert np.allclose(y, np.array([1.5, 6.0]) / np.sqrt(13.0), rtol=1e-15, atol=0)


def test_gated_rmsnorm_saturated_gate_gives_unit_rms_per_head():
    """A gate far above zero passes everything (sigmoid = 1 in fp64), and with
    w = 1, eps = 0 every (token, head) row then has mean square exactly 1 --
    per head, even when the heads' scales differ by orders of magnitude (a norm
    over the wrong axis fails this)."""
    rng = np.random.default_rng(31)
    o = rng.standard_normal((5, 3, 16)) * np.array([1e-3, 1.0, 1e3])[None, :, None]
    y = oracle.gated_rmsnorm(o, np.full(o.shape, 60.0), None, eps=0.0)
    assert np.allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-13, atol=0)
    assert np.allclose(np.sign(y), np.sign(o))


def test_gated_rmsnorm_scale_invariant_without_eps():
    """With eps = 0 the output does not depend on the scale of o (the RMS norm
    divides it out); with eps > 0 a tiny o is no longer blown up to unit RMS."""
    rng = np.random.default_rng(32)
    o = rng.standard_normal((4, 2, 8))
    g = rng.standard_normal((4, 2, 8))
    w = rng.uniform(0.5, 2.0, 8)
    y1 = oracle.gated_rmsnorm(o, g, w, eps=0.0)
    y2 = oracle.gated_rmsnorm(7.25 * o, g, w, eps=0.0)
    assert np.allclose(y1, y2, rtol=1e-13, atol=0)
    y3 = oracle.gated_rmsnorm(1e-6 * o, g, w, eps=1.0)
    assert np.abs(y3).max() < 1e-5


def test_gated_rmsnorm_gate_is_the_logistic_function():
    """Dividing out the normalised value leaves exactly the gate, which must be
    the logistic function of g (scipy's expit, an independent routine); g = 0
    halves the plain RMS norm."""
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(33)
    o = rng.standard_normal((6, 2, 8)) + 3.0            # no zero entries
    g = rng.uniform(-8.0, 8.0, o.shape)
    w = rng.uniform(0.5, 2.0, 8)
    y = oracle.gated_rmsnorm(o, g, w, eps=0.25)
    plain = oracle.gated_rmsnorm(o, np.full(o.shape, 60.0), w, eps=0.25)
    assert np.allclose(y / plain, special.expit(g), rtol=1e-13, atol=0)
    half = oracle.gated_rmsnorm(o, np.zeros(o.shape), w, eps=0.25)
    assert np.allclose(half, 0.5 * plain, rtol=1e-15, atol=0)


# ------------------------------------------------------- input prologue (ShortConv(4), Swish, L2Norm)

def _swish_expit(c):
    special = pytest.importorskip("scipy.special")
    return c * special.expit(c)


def test_short_conv_identity_taps_give_swish():
    """Taps (0, 0, 0, 1) put the whole weight on the current token: the output
    is Swish(x) = x * sigmoid(x) (scipy's expit), whatever the history."""
    rng = np.random.default_rng(41)
    x = rng.standard_normal((2, 9, 3, 8)) * 3
    w = np.zeros((3, 8, 4))
    w[:, :, 3] = 1.0
    conv0 = rng.standard_normal((2, 3, 3, 8))
    y, _ = oracle.short_conv(x, w, conv0)
    assert np.allclose(y, _swish_expit(x), rtol=1e-14, atol=1e-15)


def test_short_conv_delay_tap_is_causal_three_steps_back():
    """Taps (1, 0, 0, 0) read the input three tokens back: zeros (no history)
    for the first three tokens, then Swish(x_{t-3}); changing a later token
    never changes an earlier output (causality)."""
    rng = np.random.default_rng(42)
    x = rng.standard_normal((1, 10, 2, 4))
    w = np.zeros((2, 4, 4))
    w[:, :, 0] = 1.0
    y, _ = oracle.short_conv(x, w)
    assert np.all(y[:, :3] == 0.0)
    assert np.allclose(y[:, 3:], _swish_expit(x[:, :-3]), rtol=1e-14, atol=1e-15)
    x2 = x.copy()
    x2[:, 6:] += 5.0
    y2, _ = oracle.short_conv(x2, w)
    assert np.array_equal(y2[:, :9], y[:, :9])   # token 6 reaches outputs 9 on


def test_short_conv_matches_numpy_convolution_with_history():
    """General taps and a nonzero history against numpy's convolve (an
    independent routine): the valid part of history ++ x convolved with the
    reversed taps is the pre-Swish sum c_t = sum_i w_i x_{t-3+i}."""
    rng = np.random.default_rng(43)
    T, H, d = 12, 2, 5
    x = rng.standard_normal((1, T, H, d))
    w = rng.standard_normal((H, d, 4))
    conv0 = rng.standard_normal((1, 3, H, d))
    y, _ = oracle.short_conv(x, w, conv0)
    c = np.zeros((T, H, d))
    for h in range(H):
        for ch in range(d):
            seq = np.concatenate([conv0[0, :, h, ch], x[0, :, h, ch]])
            c[:, h, ch] = np.convolve(seq, w[h, ch, ::-1], mode="valid")
    assert np.allclose(y[0], _swish_expit(c), rtol=1e-12, atol=1e-14)


def test_prologue_l2norm_unit_rows_for_q_and_k_only():
    """With eps = 0, every (token, head) row of q and k has norm 1 (a norm over
    the wrong axis fails this with heads of very different scales); v is not
    normalised."""
    rng = np.random.default_rng(44)
    scale = np.array([1e-2, 1.0, 1e2])[None, None, :, None]
    xq, xk, xv = (rng.standard_normal((2, 7, 3, 16)) * scale for _ in range(3))
    wq, wk, wv = (rng.standard_normal((3, 16, 4)) for _ in range(3))
    q, k, v, _ = oracle.prologue(xq, xk, xv, wq, wk, wv, eps=0.0)
    assert np.allclose(np.linalg.norm(q, axis=-1), 1.0, rtol=1e-13)
    assert np.allclose(np.linalg.norm(k, axis=-1), 1.0, rtol=1e-13)
    v_plain, _ = oracle.short_conv(xv, wv)
    assert np.array_equal(v, v_plain)


def test_prologue_state_hand_off_and_varlen_isolation():
    """Running a sequence in two pieces, the second from the first's final conv
    state, equals one run (pieces of 2 tokens, shorter than the window,
    included); packed sequences equal their runs alone; the final state is the
    last three inputs of each stream."""
    rng = np.random.default_rng(45)
    H, d = 2, 6
    lengths = [2, 7, 0, 1, 5]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    Tt = int(cu[-1])
    xs = [rng.standard_normal((Tt, H, d)) for _ in range(3)]
    ws = [rng.standard_normal((H, d, 4)) for _ in range(3)]
    conv0 = rng.standard_normal((len(lengths), 3, 3, H, d))
    q, k, v, st = oracle.prologue(*xs, *ws, conv0, cu, eps=1e-6)
    for n, L in enumerate(lengths):
        a, b = int(cu[n]), int(cu[n + 1])
        one = [x[a:b][None] for x in xs]
        q1, k1, v1, st1 = oracle.prologue(*one, *ws, conv0[n:n + 1], eps=1e-6)
        assert np.array_equal(q1[0], q[a:b]) and np.array_equal(v1[0], v[a:b])
        assert np.array_equal(st1[0], st[n])
        hist = np.concatenate([conv0[n, 0], xs[0][a:b]])     # stream q: history ++ inputs
        assert np.array_equal(st[n, 0], hist[-3:])
        for cut in range(0, L + 1):
            p1 = [x[:, :cut] for x in one]
            p2 = [x[:, cut:] for x in one]
            qa, ka, va, sa = oracle.prologue(*p1, *ws, conv0[n:n + 1], eps=1e-6)
            qb, kb, vb, sb = oracle.prologue(*p2, *ws, sa, eps=1e-6)
            assert np.allclose(np.concatenate([qa, qb], 1), q1, rtol=0, atol=0)
            assert np.array_equal(sb, st1)
