"""GPU parity: libkda against the fp64 oracle on the same seeded inputs.

Small cases span several 64-token chunks and a ragged tail.  The workload
cases run the full problem sizes on the GPU: the prefill workload on every
head, the decode workload on every (session, head) pair at chosen steps plus
a 1000-step trace of sampled pairs, the varlen batch on 24 seeded heads of
every sequence, and the long workload on 4 seeded heads.
Tolerances (max-abs error / max |reference|): fp32 inputs 1e-4 on o and S;
bf16 inputs 2e-2 on o and 1e-2 on the final state.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrence_chunkwise_gb300 import build as kbuild
from linear_attention_recurrence_chunkwise_gb300 import inputs as I
from tests.gpu_util import cached_oracle, oracle_on_heads, rel_err, tol_o, tol_s

pytestmark = pytest.mark.gpu
DEV = "cuda"
ENGINES = ["cudacore", "tensorcore"]


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    kbuild.build()
    from linear_attention_recurrence_chunkwise_gb300 import kda as mod
    mod.load()
    return mod


def engine_ok(engine, dtype, d):
    """The tensor-core engine takes bf16 at d = 128 and fp32 or bf16 at d = 64;
    its variant with the blocked path for wide gates only bf16 at d = 128."""
    if engine == "tensorcore_wide":
        return dtype == "bf16" and d == 128
    if engine == "tensorcore":
        return d == 64 or dtype == "bf16"
    return True


def assert_engine_rejects(kda, call):
    """The tensor-core engine asked for a dtype or head size it does not take:
    the call returns KDA_ERR_UNSUPPORTED before any launch."""
    with pytest.raises(kda.KdaError) as e:
        call()
    assert e.value.status == kda.KDA_ERR_UNSUPPORTED


def run_fwd(kda, prob, engine, **kw):
    o, ST = kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0,
                        prob.cu_seqlens, engine=engine, **kw)
    torch.cuda.synchronize()
    return o, ST


# --------------------------------------------------------------- prefill, small

@pytest.mark.parametrize("engine", ENGINES + ["tensorcore_wide"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200, 333])
def test_prefill_small(kda, engine, dtype, d, T):
    prob = I.prefill_problem(2, T, 3, d, d, dtype, (-0.5, -0.001), 0.05, seed=T + d,
                             device=DEV)
    if not engine_ok(engine, dtype, d):
        return assert_engine_rejects(kda, lambda: run_fwd(kda, prob, engine))
    o, ST = run_fwd(kda, prob, engine)
    o_ref, S_ref = oracle_on_heads(prob, [0, 1, 2])
    dt = prob.q.dtype
    assert rel_err(o, o_ref) < tol_o(dt)
    assert rel_err(ST, S_ref) < tol_s(dt)


@pytest.mark.parametrize("engine", ENGINES)
def test_prefill_varlen_small(kda, engine):
    lengths = [0, 1, 64, 130, 7, 0, 257, 63]
    prob = I.prefill_problem(1, 0, 4, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=3,
                             device=DEV, lengths=lengths)
    o, ST = run_fwd(kda, prob, engine)
    o_ref, S_ref = oracle_on_heads(prob, [0, 1, 2, 3])
    assert rel_err(o, o_ref) < 2e-2
    assert rel_err(ST, S_ref) < 1e-2
    # empty sequences hand their initial state straight through
    for i, L in enumerate(lengths):
        if L == 0:
            assert torch.equal(ST[i], prob.S0[i])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefill_d64_tensorcore_varlen_in_place(kda, dtype):
    """d = 64 on the tensor cores: packed sequences with empty, one-token and
    ragged ones, S_T written over S0, one head with gates past the chunk form's
    range (recomputed token by token); fp32 inputs at the fp32 tolerance."""
    lengths = [0, 1, 64, 130, 7, 0, 257, 63]
    prob = I.prefill_problem(1, 0, 3, 64, 64, dtype, (-0.5, -0.001), 0.05, seed=41,
                             device=DEV, lengths=lengths)
    la = prob.log_alpha.cpu()
    la[266:266 + 100, 1] = -3.0                # head 1 of the 257-token sequence: wide
    prob.log_alpha.copy_(la.to(DEV))
    o_ref, S_ref = oracle_on_heads(prob, [0, 1, 2])
    S = prob.S0.clone()
    ws = torch.zeros(kda.kda_fwd_workspace_bytes(len(lengths)), dtype=torch.uint8, device=DEV)
    o, _ = kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, S, prob.cu_seqlens,
                       S_T=S, workspace=ws, engine="tensorcore")
    torch.cuda.synchronize()
    assert kda.kda_read_device_status(ws) == kda.KDA_OK
    dt = prob.q.dtype
    assert rel_err(o, o_ref) < tol_o(dt)
    assert rel_err(S, S_ref) < tol_s(dt)
    for i, L in enumerate(lengths):
        if L == 0:
            assert torch.equal(S[i], prob.S0[i])


@pytest.mark.parametrize("engine", ENGINES)
def test_varlen_isolation_bit_identical(kda, engine):
    """Reordering the packed sequences leaves each one's o and S_T bit-identical."""
    lengths = [100, 5, 64, 300]
    prob = I.prefill_problem(1, 0, 2, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=4,
                             device=DEV, lengths=lengths)
    o, ST = run_fwd(kda, prob, engine)
    cu = prob.cu_seqlens.cpu().tolist()
    perm = [3, 1, 0, 2]
    cat = lambda t: torch.cat([t[cu[i]:cu[i + 1]] for i in perm])
    cu_p = torch.tensor([0] + list(np.cumsum([lengths[i] for i in perm])), dtype=torch.int32,
                        device=DEV)
    prob_p = I.Problem(cat(prob.q), cat(prob.k), cat(prob.v), cat(prob.log_alpha),
                       cat(prob.beta), prob.S0[perm].contiguous(), cu_p)
    o_p, ST_p = run_fwd(kda, prob_p, engine)
    assert torch.equal(ST_p, ST[perm])
    assert torch.equal(o_p, cat(o))


@pytest.mark.parametrize("engine", ENGINES)
def test_split_run_matches_whole(kda, engine):
    """fwd(T1) then fwd(T2, S0 = S_T1) agrees with fwd(T1 + T2)."""
    prob = I.prefill_problem(1, 500, 3, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=5,
                             device=DEV)
    o, ST = run_fwd(kda, prob, engine)
    a = I.Problem(prob.q[:, :170].contiguous(), prob.k[:, :170].contiguous(),
                  prob.v[:, :170].contiguous(), prob.log_alpha[:, :170].contiguous(),
                  prob.beta[:, :170].contiguous(), prob.S0, None)
    o1, S1 = run_fwd(kda, a, engine)
    b = I.Problem(prob.q[:, 170:].contiguous(), prob.k[:, 170:].contiguous(),
                  prob.v[:, 170:].contiguous(), prob.log_alpha[:, 170:].contiguous(),
                  prob.beta[:, 170:].contiguous(), S1, None)
    o2, S2 = run_fwd(kda, b, engine)
    assert rel_err(torch.cat([o1, o2], 1), o.double().cpu().numpy()) < 2e-2
    assert rel_err(S2, ST.double().cpu().numpy()) < 1e-2


@pytest.mark.parametrize("engine", ENGINES)
def test_state_in_place_and_optional_outputs(kda, engine):
    prob = I.prefill_problem(2, 150, 2, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=6,
                             device=DEV)
    o, ST = run_fwd(kda, prob, engine)
    S = prob.S0.clone()
    o2, S_ret = kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, S, None,
                            S_T=S, engine=engine)        # S_T aliases S0
    torch.cuda.synchronize()
    assert S_ret.data_ptr() == S.data_ptr()
    assert torch.equal(S, ST) and torch.equal(o2, o)
    o3, none = kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0, None,
                           return_state=False, engine=engine)
    torch.cuda.synchronize()
    assert none is None and torch.equal(o3, o)
    zero = I.Problem(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, None, None)
    oz, Sz = run_fwd(kda, zero, engine)
    zref = I.Problem(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta,
                     torch.zeros_like(prob.S0), None)
    oz2, Sz2 = run_fwd(kda, zref, engine)
    assert torch.equal(oz, oz2) and torch.equal(Sz, Sz2)


def test_prefill_equals_decode_steps(kda):
    """The chunkwise prefill and T single-token decode steps agree (same causal
    semantics: a token reads the state after its own write)."""
    prob = I.prefill_problem(1, 96, 2, 128, 128, "f32", (-0.5, -0.001), 0.05, seed=7,
                             device=DEV)
    o, ST = run_fwd(kda, prob, "cudacore")
    S = prob.S0.clone()
    outs = []
    for t in range(96):
        outs.append(kda.kda_decode_step(prob.q[:, t].contiguous(), prob.k[:, t].contiguous(),
                                        prob.v[:, t].contiguous(),
                                        prob.log_alpha[:, t].contiguous(),
                                        prob.beta[:, t].contiguous(), S))
    torch.cuda.synchronize()
    assert rel_err(torch.stack(outs, 1), o.double().cpu().numpy()) < 1e-4
    assert rel_err(S, ST.double().cpu().numpy()) < 1e-4


def test_zero_sizes(kda):
    e = torch.empty(0, 2, 64, device=DEV)
    o, ST = kda.kda_fwd(e, e, e, e, torch.empty(0, 2, device=DEV), None,
                        torch.zeros(1, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert o.numel() == 0 and ST.shape == (0, 2, 64, 64)


@pytest.mark.parametrize("engine", ENGINES + ["tensorcore_wide"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T", [1, 65, 200])
def test_wide_gate_domain(kda, engine, dtype, d, T):
    """Per-token log-decay down to -5 (the K3 bound: -320 over a 64-token chunk,
    far outside the chunk form's +-80) is exact: such chunks take the blocked
    path (tensorcore_wide) or are taken token by token, and the status word
    stays clear."""
    prob = I.prefill_problem(2, T, 3, d, d, dtype, (-5.0, -0.5), 0.05, seed=T + d + 11,
                             device=DEV)
    ws = torch.zeros(kda.kda_fwd_workspace_bytes(2), dtype=torch.uint8, device=DEV)
    if not engine_ok(engine, dtype, d):
        return assert_engine_rejects(kda, lambda: run_fwd(kda, prob, engine, workspace=ws))
    o, ST = run_fwd(kda, prob, engine, workspace=ws)
    assert kda.kda_read_device_status(ws) == kda.KDA_OK
    o_ref, S_ref = oracle_on_heads(prob, [0, 1, 2])
    dt = prob.q.dtype
    assert rel_err(o, o_ref) < tol_o(dt)
    assert rel_err(ST, S_ref) < tol_s(dt)


@pytest.mark.parametrize("engine", ENGINES + ["tensorcore_wide"])
def test_wide_gate_mixed_chunks_varlen_in_place(kda, engine):
    """Strong and mild gates mixed across heads and across the chunks of one
    sequence, packed varlen with empty and ragged sequences, S_T written over
    S0: the wide chunks take the blocked path (tensorcore_wide; a head with ten
    tokens of near-total forgetting, beyond any 16-token block's range, still
    goes token by token) or the token-serial path, the rest the chunk form."""
    lengths = [130, 0, 64, 257, 1]
    prob = I.prefill_problem(1, 0, 4, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=21,
                             device=DEV, lengths=lengths)
    g = torch.Generator().manual_seed(22)
    la = prob.log_alpha.cpu()
    strong = -(torch.rand(la.shape, generator=g) * 4.5 + 0.5)     # U(-5, -0.5)
    la[:, 0] = strong[:, 0]                  # head 0: every chunk wide
    la[64:128, 2] = strong[64:128, 2]         # head 2: the second chunk of sequence 0
    la[194 + 100:194 + 110, 3] = -60.0        # head 3: ten tokens of near-total forgetting
    prob.log_alpha.copy_(la.to(DEV))
    o_ref, S_ref = oracle_on_heads(prob, [0, 1, 2, 3])
    S = prob.S0.clone()
    ws = torch.zeros(kda.kda_fwd_workspace_bytes(len(lengths)), dtype=torch.uint8, device=DEV)
    o, _ = kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, S, prob.cu_seqlens,
                       S_T=S, workspace=ws, engine=engine)
    torch.cuda.synchronize()
    assert kda.kda_read_device_status(ws) == kda.KDA_OK
    assert rel_err(o, o_ref) < 2e-2
    assert rel_err(S, S_ref) < 1e-2
    assert torch.equal(S[1], prob.S0[1])      # the empty sequence passes its state through


def test_bad_device_offsets_write_nothing(kda):
    prob = I.prefill_problem(1, 0, 2, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=9,
                             device=DEV, lengths=[50, 50])
    bad = torch.tensor([0, 70, 60], dtype=torch.int32, device=DEV)   # decreasing
    o = torch.full_like(prob.v, 7.0)
    ST = torch.full_like(prob.S0, 7.0)
    ws = torch.zeros(kda.kda_fwd_workspace_bytes(2), dtype=torch.uint8, device=DEV)
    kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0, bad, o=o, S_T=ST,
                workspace=ws)
    assert kda.kda_read_device_status(ws) == kda.KDA_ERR_INVALID_ARGUMENT
    assert bool((o == 7.0).all()) and bool((ST == 7.0).all())
    short = torch.tensor([0, 50, 90], dtype=torch.int32, device=DEV)  # does not end at Ttot
    kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0, short, o=o,
                S_T=ST, workspace=ws)
    assert kda.kda_read_device_status(ws) == kda.KDA_ERR_INVALID_ARGUMENT


# --------------------------------------------------------------- decode, small

@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("N", [8192, 8500])
def test_many_short_sequences(kda, engine, N):
    """N packed sequences of 0-130 tokens: 8192 is the largest count that gets
    the longest-first launch order, 8500 runs in the given order.  Every
    sequence of one head follows the oracle."""
    pattern = [0, 1, 2, 7, 63, 64, 65, 130]
    lengths = [pattern[(i * 5 + i // 8) % len(pattern)] for i in range(N)]
    prob = I.prefill_problem(1, 0, 2, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=N,
                             device=DEV, lengths=lengths)
    ws = torch.zeros(kda.kda_fwd_workspace_bytes(N), dtype=torch.uint8, device=DEV)
    o, ST = run_fwd(kda, prob, engine, workspace=ws)
    assert kda.kda_read_device_status(ws) == kda.KDA_OK
    o_ref, S_ref = oracle_on_heads(prob, [1])
    idx = torch.tensor([1], device=DEV)
    assert rel_err(o.index_select(1, idx), o_ref) < 2e-2
    assert rel_err(ST.index_select(1, idx), S_ref) < 1e-2


@pytest.mark.parametrize("engine", ENGINES)
def test_bounds_checked_build(kda, engine):
    """The bounds-checked build (every computed global index checked against its
    tensor's extent, KDA_ERR_BOUNDS on a miss) runs fixed-length, ragged and
    empty sequences without a report and with results that match the oracle."""
    lib = kda.load_library(kbuild.build(bounds_check=True))
    cases = [I.prefill_problem(2, T, 2, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=T,
                               device=DEV) for T in (1, 65, 333)]
    cases.append(I.prefill_problem(1, 0, 2, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=5,
                                   device=DEV, lengths=[0, 130, 1, 64, 0, 7]))
    for prob in cases:
        n = prob.S0.shape[0]
        ws = torch.zeros(int(lib.kda_fwd_workspace_bytes(n)), dtype=torch.uint8, device=DEV)
        o, ST = kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0,
                            prob.cu_seqlens, workspace=ws, engine=engine, lib=lib)
        assert kda.kda_read_device_status(ws, lib=lib) == kda.KDA_OK
        o_ref, S_ref = oracle_on_heads(prob, [0, 1])
        assert rel_err(o, o_ref) < 2e-2
        assert rel_err(ST, S_ref) < 1e-2


def test_bounds_checked_build_d64_tensorcore(kda):
    """The bounds-checked build through the d = 64 tensor-core engine: fp32
    fixed-length and ragged packed sequences with empty ones, a wide-gate head
    (token-serial pass), and kda_fwd_cp's task tables -- no report, results
    against the oracle at the fp32 tolerance."""
    lib = kda.load_library(kbuild.build(bounds_check=True))
    cases = [I.prefill_problem(2, 65, 2, 64, 64, "f32", (-0.5, -0.001), 0.05, seed=12,
                               device=DEV),
             I.prefill_problem(1, 0, 2, 64, 64, "f32", (-0.5, -0.001), 0.05, seed=13,
                               device=DEV, lengths=[0, 130, 1, 64, 0, 7]),
             I.prefill_problem(1, 0, 2, 64, 64, "f32", (-5.0, -0.5), 0.05, seed=14,
                               device=DEV, lengths=[70, 0, 3])]
    for prob in cases:
        n = prob.S0.shape[0]
        ws = torch.zeros(int(lib.kda_fwd_cp_workspace_bytes(n, 2, 64, 64, 3)),
                         dtype=torch.uint8, device=DEV)
        o_ref, S_ref = oracle_on_heads(prob, [0, 1])
        for call in (kda.kda_fwd, lambda *a, **k: kda.kda_fwd_cp(*a, segments=3, **k)):
            o, ST = call(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0,
                         prob.cu_seqlens, workspace=ws, engine="tensorcore", lib=lib)
            assert kda.kda_read_device_status(ws, lib=lib) == kda.KDA_OK
            assert rel_err(o, o_ref) < 1e-4
            assert rel_err(ST, S_ref) < 1e-4


def test_cuda_graph_capture(kda):
    """kda_fwd, kda_fwd_cp and kda_decode_step enqueue kernels only (no
    allocation, no synchronisation), so each can be captured in a CUDA graph;
    replays reproduce the eager results bit for bit (three replays of the
    decode step = three in-place steps)."""
    prob = I.prefill_problem(1, 300, 4, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=71,
                             device=DEV)
    o_e, S_e = run_fwd(kda, prob, "auto")
    oc_e, Sc_e = run_cp(kda, prob, "auto", 3)
    N, H, d = 6, 4, 128
    S_dec0 = I.decode_state(N, H, d, d, 0.02, seed=72, device=DEV)
    x = I.decode_token(N, H, d, d, "bf16", seed=72, step=0, device=DEV)
    S_eager = S_dec0.clone()
    for _ in range(3):
        od_e = kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S_eager)
    torch.cuda.synchronize()

    o, ST = torch.empty_like(o_e), torch.empty_like(S_e)
    oc, STc = torch.empty_like(o_e), torch.empty_like(S_e)
    ws = torch.zeros(kda.kda_fwd_workspace_bytes(1), dtype=torch.uint8, device=DEV)
    wsc = torch.zeros(kda.kda_fwd_cp_workspace_bytes(1, 4, 128, 128, 3), dtype=torch.uint8,
                      device=DEV)
    S_dec, od = S_dec0.clone(), torch.empty_like(od_e)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # first calls outside capture (one-time host set-up)
        kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0, o=o, S_T=ST,
                    workspace=ws)
        kda.kda_fwd_cp(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0, segments=3,
                       o=oc, S_T=STc, workspace=wsc)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g_fwd, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_fwd):
        kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0, o=o, S_T=ST,
                    workspace=ws)
        kda.kda_fwd_cp(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0, segments=3,
                       o=oc, S_T=STc, workspace=wsc)
    with torch.cuda.graph(g_dec):
        kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S_dec, o=od)
    o.zero_(), ST.zero_(), oc.zero_(), STc.zero_()
    torch.cuda.synchronize()
    g_fwd.replay()
    for _ in range(3):
        g_dec.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_e) and torch.equal(ST, S_e)
    assert torch.equal(oc, oc_e) and torch.equal(STc, Sc_e)
    assert torch.equal(S_dec, S_eager) and torch.equal(od, od_e)


@pytest.mark.parametrize("engine", ENGINES)
def test_bounds_checked_build_segment_parallel(kda, engine):
    """The bounds-checked build through kda_fwd_cp: task-table addressing of
    token ranges and state blocks, empty segments, the zero-v tile, wide-gate
    chunks on the token-serial path -- no report, results match the oracle."""
    lib = kda.load_library(kbuild.build(bounds_check=True))
    cases = [(I.prefill_problem(1, 0, 2, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=6,
                                device=DEV, lengths=[0, 130, 1, 64, 300]), 4),
             (I.prefill_problem(2, 200, 2, 128, 128, "bf16", (-5.0, -0.5), 0.05, seed=7,
                                device=DEV), 3)]
    for prob, P in cases:
        n = prob.S0.shape[0]
        ws = torch.zeros(int(lib.kda_fwd_cp_workspace_bytes(n, 2, 128, 128, P)),
                         dtype=torch.uint8, device=DEV)
        o, ST = kda.kda_fwd_cp(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0,
                               prob.cu_seqlens, segments=P, workspace=ws, engine=engine,
                               lib=lib)
        assert kda.kda_read_device_status(ws, lib=lib) == kda.KDA_OK
        o_ref, S_ref = oracle_on_heads(prob, [0, 1])
        assert rel_err(o, o_ref) < 2e-2
        assert rel_err(ST, S_ref) < 1e-2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("K", [1, 4, 8, 11, 16])
def test_verify_and_commit_draft_tokens(kda, dtype, d, K):
    """Speculative-decode verify / commit over K cached draft tokens: outputs
    and states against the oracle, S untouched by verify, per-session accepted
    counts (clamped to [0, K]), and agreement with K single-token steps to fp32
    rounding."""
    N, H = 5, 3
    x = I.draft_tokens(N, K, H, d, d, dtype, seed=K, device=DEV)
    q, k, v, la, b = (x[key] for key in ("q", "k", "v", "log_alpha", "beta"))
    S = I.decode_state(N, H, d, d, 0.02, seed=K, device=DEV)
    S0 = S.clone()
    o = kda.kda_verify_tokens(q, k, v, la, b, S)
    torch.cuda.synchronize()
    assert torch.equal(S, S0)
    assert rel_err(o, oracle.verify_tokens(q, k, v, la, b, S0)) < tol_o(q.dtype)
    Sd, od = S0.clone(), []
    for t in range(K):
        od.append(kda.kda_decode_step(q[:, t].contiguous(), k[:, t].contiguous(),
                                      v[:, t].contiguous(), la[:, t].contiguous(),
                                      b[:, t].contiguous(), Sd))
    torch.cuda.synchronize()
    # the draft kernel sums in another order than the one-token kernel: fp32
    # rounding apart (one bf16 rounding step on a bf16 o)
    near = 1e-5 if dtype == "f32" else 8e-3
    assert rel_err(o, torch.stack(od, dim=1).double().cpu()) < near
    acc = torch.tensor([0, K, 1, K // 2, K + 3], dtype=torch.int32, device=DEV)
    kda.kda_commit_tokens(q, k, v, la, b, S, n_accept=acc)
    torch.cuda.synchronize()
    S_ref = oracle.commit_tokens(q, k, v, la, b, S0, acc.cpu().numpy())
    assert rel_err(S, S_ref) < (1e-4 if dtype == "f32" else 1e-2)
    assert torch.equal(S[0], S0[0])
    S_all = S0.clone()
    kda.kda_commit_tokens(q, k, v, la, b, S_all)
    torch.cuda.synchronize()
    assert rel_err(S_all, Sd.double().cpu()) < 1e-5


@pytest.mark.parametrize("la", [(-40.0, -5.0), (-1e-6, 0.0)])
def test_draft_tokens_extreme_decay(kda, la):
    """Gates far past exp underflow over a 16-token draft (the decay products
    go to zero, never overflow) and gates of exactly or nearly 1."""
    N, K, H, d = 3, 16, 4, 128
    x = I.draft_tokens(N, K, H, d, d, "f32", la, seed=7, device=DEV)
    ins = tuple(x[key] for key in ("q", "k", "v", "log_alpha", "beta"))
    S = I.decode_state(N, H, d, d, 0.5, seed=7, device=DEV)
    S0 = S.clone()
    o = kda.kda_verify_tokens(*ins, S)
    kda.kda_commit_tokens(*ins, S)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(S).all())
    assert rel_err(o, oracle.verify_tokens(*ins, S0)) < 1e-4
    assert rel_err(S, oracle.commit_tokens(*ins, S0)) < 1e-4


def _padded(shape, dtype, pad, fill):
    """A contiguous view of `shape` inside a buffer with `pad` canary elements
    on each side (pad keeps the view 16-byte aligned)."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * pad,), fill, dtype=dtype, device=DEV)
    return buf, buf[pad:pad + n].view(shape)


def _canaries_intact(buf, pad, fill):
    head, tail = buf[:pad], buf[-pad:]
    return bool((head == fill).all()) and bool((tail == fill).all())


@pytest.mark.parametrize("engine", ENGINES)
def test_no_writes_outside_outputs(kda, engine):
    """Ragged varlen tails, a single-token sequence and an empty one: o and S_T
    live inside canary-filled buffers, which must come back untouched, and the
    results must still match the oracle."""
    lengths = [1, 0, 65, 130, 7, 200]
    prob = I.prefill_problem(1, 0, 2, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=31,
                             device=DEV, lengths=lengths)
    pad, fill = 1024, -768.0  # exact in bf16 and fp32
    obuf, o = _padded(tuple(prob.v.shape), prob.v.dtype, pad, fill)
    sbuf, ST = _padded(tuple(prob.S0.shape), torch.float32, pad, fill)
    kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0, prob.cu_seqlens,
                o=o, S_T=ST, engine=engine)
    torch.cuda.synchronize()
    assert _canaries_intact(obuf, pad, fill) and _canaries_intact(sbuf, pad, fill)
    o_ref, S_ref = oracle_on_heads(prob, [0, 1])
    assert rel_err(o, o_ref) < 2e-2
    assert rel_err(ST, S_ref) < 1e-2
    # decode on the returned states, in place, with a canary-padded output
    x = I.decode_token(len(lengths), 2, 128, 128, "bf16", (-0.1, -0.0005), seed=3, step=0,
                       device=DEV)
    dbuf, od = _padded((len(lengths), 2, 128), torch.bfloat16, pad, fill)
    kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], ST, o=od)
    torch.cuda.synchronize()
    assert _canaries_intact(dbuf, pad, fill) and _canaries_intact(sbuf, pad, fill)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_small(kda, dtype, d):
    N, H, steps = 3, 5, 20
    S = I.decode_state(N, H, d, d, 0.05, seed=d, device=DEV)
    S_ref = S.double().cpu().numpy()
    for s in range(steps):
        x = I.decode_token(N, H, d, d, dtype, (-0.1, -0.0005), seed=d, step=s, device=DEV)
        o = kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S)
        o_ref, S_ref = oracle.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                          S_ref)
        torch.cuda.synchronize()
        assert rel_err(o, o_ref) < tol_o(x["q"].dtype)
    assert rel_err(S, S_ref) < (1e-4 if dtype == "f32" else 1e-2)


# --------------------------------------------------------------- workload sizes

@pytest.mark.parametrize("engine", ENGINES)
def test_workload_tiny_fp32(kda, engine):
    """B=1, H=2, T=256, d=64, fp32: every element against the oracle at 1e-4."""
    prob = I.preset_problem("tiny", seed=0, device=DEV)
    if not engine_ok(engine, "f32", 64):
        return assert_engine_rejects(kda, lambda: run_fwd(kda, prob, engine))
    o, ST = run_fwd(kda, prob, engine)
    o_ref, S_ref = oracle_on_heads(prob, [0, 1])
    eo, es = rel_err(o, o_ref), rel_err(ST, S_ref)
    print(f"[parity] tiny {engine}: o {eo:.2e} S {es:.2e}")
    assert eo < 1e-4
    assert es < 1e-4


@pytest.mark.parametrize("engine", ENGINES)
def test_workload_prefill_all_heads(kda, engine):
    """B=1, H=96, T=8192, d=128, bf16: o and S_T of every head against the oracle."""
    prob = I.preset_problem("prefill", seed=0, device=DEV)
    o, ST = run_fwd(kda, prob, engine)
    o_ref, S_ref = cached_oracle("prefill", prob, list(range(96)))
    eo, es = rel_err(o, o_ref), rel_err(ST, S_ref)
    print(f"[parity] prefill {engine}, all 96 heads: o {eo:.2e} S {es:.2e}")
    assert eo < 2e-2
    assert es < 1e-2


@pytest.mark.parametrize("engine", ENGINES)
def test_workload_long_sampled_heads(kda, engine):
    """B=1, H=96, T=131072, nonzero S0, long-memory gates: 4 sampled heads."""
    prob = I.preset_problem("long", seed=0, device=DEV)
    o, ST = run_fwd(kda, prob, engine)
    heads = I.sampled_heads(96, 4, seed=0)
    o_ref, S_ref = oracle_on_heads(prob, heads)
    idx = torch.tensor(heads, device=DEV)
    eo, es = rel_err(o.index_select(2, idx), o_ref), rel_err(ST.index_select(1, idx), S_ref)
    print(f"[parity] long {engine}: o {eo:.2e} S {es:.2e}")
    assert eo < 2e-2
    assert es < 1e-2
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(ST).all())


@pytest.mark.parametrize("engine", ["tensorcore_wide", "tensorcore"])
def test_workload_wide_gates_all_heads(kda, engine):
    """B=1, H=96, T=8192, d=128, bf16 with K3-strength gates, log alpha in
    U(-5, -0.5): every chunk leaves the chunk form's range; o and S_T of every
    head against the oracle."""
    prob = I.prefill_problem(1, 8192, 96, 128, 128, "bf16", (-5.0, -0.5), None, seed=0,
                             device=DEV)
    ws = torch.zeros(kda.kda_fwd_workspace_bytes(1), dtype=torch.uint8, device=DEV)
    o, ST = run_fwd(kda, prob, engine, workspace=ws)
    assert kda.kda_read_device_status(ws) == kda.KDA_OK
    o_ref, S_ref = cached_oracle("wide_gates", prob, list(range(96)))
    eo, es = rel_err(o, o_ref), rel_err(ST, S_ref)
    print(f"[parity] wide gates {engine}, all 96 heads: o {eo:.2e} S {es:.2e}")
    assert eo < 2e-2
    assert es < 1e-2


def test_bounds_checked_build_blocked_path(kda):
    """The bounds-checked build through the blocked path: wide chunks, ragged
    and empty sequences, no report, results against the oracle."""
    lib = kda.load_library(kbuild.build(bounds_check=True))
    prob = I.prefill_problem(1, 0, 2, 128, 128, "bf16", (-5.0, -0.5), 0.05, seed=8,
                             device=DEV, lengths=[0, 130, 1, 64, 200])
    ws = torch.zeros(int(lib.kda_fwd_workspace_bytes(5)), dtype=torch.uint8, device=DEV)
    o, ST = kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0,
                        prob.cu_seqlens, workspace=ws, engine="tensorcore_wide", lib=lib)
    assert kda.kda_read_device_status(ws, lib=lib) == kda.KDA_OK
    o_ref, S_ref = oracle_on_heads(prob, [0, 1])
    assert rel_err(o, o_ref) < 2e-2
    assert rel_err(ST, S_ref) < 1e-2


# ------------------------------------------------ segment-parallel forward

def run_cp(kda, prob, engine, segments, **kw):
    o, ST = kda.kda_fwd_cp(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0,
                           prob.cu_seqlens, segments=segments, engine=engine, **kw)
    torch.cuda.synchronize()
    return o, ST


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("segments", [2, 3, 5])
def test_cp_matches_oracle(kda, engine, dtype, d, segments):
    """kda_fwd_cp over 2, 3 and 5 segments per sequence (ragged T, nonzero S0,
    two sequences) against the oracle, at kda_fwd's tolerances."""
    prob = I.prefill_problem(2, 333, 3, d, d, dtype, (-0.5, -0.001), 0.05, seed=segments + d,
                             device=DEV)
    ws = torch.zeros(kda.kda_fwd_cp_workspace_bytes(2, 3, d, d, segments), dtype=torch.uint8,
                     device=DEV)
    if not engine_ok(engine, dtype, d):
        return assert_engine_rejects(kda, lambda: run_cp(kda, prob, engine, segments,
                                                         workspace=ws))
    o, ST = run_cp(kda, prob, engine, segments, workspace=ws)
    assert kda.kda_read_device_status(ws) == kda.KDA_OK
    o_ref, S_ref = oracle_on_heads(prob, [0, 1, 2])
    dt = prob.q.dtype
    assert rel_err(o, o_ref) < tol_o(dt)
    assert rel_err(ST, S_ref) < tol_s(dt)


@pytest.mark.parametrize("engine", ENGINES)
def test_cp_varlen_short_empty_in_place(kda, engine):
    """Packed sequences shorter than the segment count (empty segments act as
    identity maps), an empty sequence, a ragged tail, S_T written over S0."""
    lengths = [0, 1, 64, 130, 700, 65]
    prob = I.prefill_problem(1, 0, 4, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=31,
                             device=DEV, lengths=lengths)
    o_ref, S_ref = oracle_on_heads(prob, [0, 1, 2, 3])
    S = prob.S0.clone()
    o, _ = kda.kda_fwd_cp(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, S,
                          prob.cu_seqlens, segments=4, S_T=S, engine=engine)
    torch.cuda.synchronize()
    assert rel_err(o, o_ref) < 2e-2
    assert rel_err(S, S_ref) < 1e-2
    assert torch.equal(S[0], prob.S0[0])      # the empty sequence passes its state through


def test_cp_edge_sizes(kda):
    """kda_fwd_cp on degenerate sizes: no sequences, sequences of zero tokens,
    and more segments than chunks (every sequence shorter than the split)."""
    e = torch.empty(0, 2, 64, device=DEV)
    o, ST = kda.kda_fwd_cp(e, e, e, e, torch.empty(0, 2, device=DEV), None,
                           torch.zeros(1, dtype=torch.int32, device=DEV), segments=3)
    torch.cuda.synchronize()
    assert o.numel() == 0 and ST.shape == (0, 2, 64, 64)
    prob = I.prefill_problem(1, 0, 2, 64, 64, "f32", (-0.5, -0.001), 0.05, seed=81,
                             device=DEV, lengths=[0, 0, 3])
    o, ST = run_cp(kda, prob, "cudacore", 7)
    o_ref, S_ref = oracle_on_heads(prob, [0, 1])
    assert rel_err(o, o_ref) < 1e-4 and rel_err(ST, S_ref) < 1e-4
    assert torch.equal(ST[:2], prob.S0[:2])
    prob = I.prefill_problem(2, 100, 2, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=82,
                             device=DEV)
    o, ST = run_cp(kda, prob, "tensorcore", 16)     # 2 chunks per sequence, 16 segments
    o_ref, S_ref = oracle_on_heads(prob, [0, 1])
    assert rel_err(o, o_ref) < 2e-2 and rel_err(ST, S_ref) < 1e-2


@pytest.mark.parametrize("engine", ENGINES)
def test_cp_wide_gates(kda, engine):
    """Gates past the chunk form's range inside segment-parallel runs: the
    token-serial path honours the zero-v, identity-start and state-only tasks."""
    prob = I.prefill_problem(1, 400, 3, 128, 128, "bf16", (-5.0, -0.5), 0.05, seed=41,
                             device=DEV)
    o, ST = run_cp(kda, prob, engine, 3)
    o_ref, S_ref = oracle_on_heads(prob, [0, 1, 2])
    assert rel_err(o, o_ref) < 2e-2
    assert rel_err(ST, S_ref) < 1e-2


@pytest.mark.parametrize("engine", ENGINES)
def test_cp_slow_gates_compose(kda, engine):
    """Slow gates (log alpha in U(-0.01, -0.0001)) over 128-token segments keep
    each segment's map M far from zero, so the start states come from the scan's
    composition M S_in + S~ and not from forgetting: 8 segments against the
    oracle (bf16 on both engines)."""
    prob = I.prefill_problem(1, 1024, 3, 128, 128, "bf16", (-0.01, -0.0001), 0.05, seed=61,
                             device=DEV)
    o, ST = run_cp(kda, prob, engine, 8)
    o_ref, S_ref = oracle_on_heads(prob, [0, 1, 2])
    eo, es = rel_err(o, o_ref), rel_err(ST, S_ref)
    print(f"[parity] cp slow gates {engine}: o {eo:.2e} S {es:.2e}")
    assert eo < 2e-2
    assert es < 1e-2


def test_cp_fp32_agrees_with_plain(kda):
    """On the fp32 CUDA-core engine every step of the segment maps and the scan
    is fp32, so kda_fwd_cp and kda_fwd agree to fp32 rounding; slow gates keep
    the maps far from zero."""
    prob = I.prefill_problem(1, 1000, 2, 64, 64, "f32", (-0.01, -0.0001), 0.05, seed=51,
                             device=DEV)
    o1, S1 = run_fwd(kda, prob, "cudacore")
    o2, S2 = run_cp(kda, prob, "cudacore", 6)
    assert rel_err(o2, o1.double().cpu().numpy()) < 1e-5
    assert rel_err(S2, S1.double().cpu().numpy()) < 1e-5


def test_workload_long_tp8_segment_parallel(kda):
    """The segment-parallel workload at full size (B=1, H=12, T=131072, nonzero
    S0, long-memory gates) with the suggested segment count: 3 sampled heads
    against the oracle."""
    prob = I.preset_problem("long_tp8", seed=0, device=DEV)
    P = kda.kda_fwd_cp_segments(1, 12, 131072)
    assert P > 1
    o, ST = run_cp(kda, prob, "auto", P)
    heads = I.sampled_heads(12, 3, seed=0)
    o_ref, S_ref = oracle_on_heads(prob, heads)
    idx = torch.tensor(heads, device=DEV)
    eo, es = rel_err(o.index_select(2, idx), o_ref), rel_err(ST.index_select(1, idx), S_ref)
    print(f"[parity] long_tp8 segments={P}: o {eo:.2e} S {es:.2e}")
    assert eo < 2e-2
    assert es < 1e-2


def test_workload_decode_sampled_sessions(kda):
    """64 sessions x 96 heads, fp32 state, 1000 in-place steps: 12 sampled
    (session, head) pairs follow the oracle step by step; every one of the 6,144
    pairs follows it over steps 0 and 1 (same start state), and takes step 999
    as the oracle does from the state the GPU reached after step 998."""
    p = I.PRESETS["decode"]
    N, H, d = p["N"], p["H"], p["d"]
    S = I.decode_state(N, H, d, d, p["s0_std"], seed=0, device=DEV)
    S_all = S.double().cpu().numpy()
    g = torch.Generator().manual_seed(1)
    pairs = [(int(n), int(h)) for n, h in zip(torch.randint(0, N, (12,), generator=g),
                                              torch.randint(0, H, (12,), generator=g))]
    ns = torch.tensor([a for a, _ in pairs], device=DEV)
    hs = torch.tensor([b for _, b in pairs], device=DEV)
    S_ref = S[ns, hs].double().cpu().numpy()[:, None]          # [12, 1, d, d]
    worst = 0.0
    steps = p["steps"]
    for s in range(steps):
        x = I.decode_token(N, H, d, d, p["dtype"], p["la"], seed=0, step=s, device=DEV)
        if s == steps - 1:   # every pair: one oracle step from the GPU's own state
            torch.cuda.synchronize()
            S_all = S.double().cpu().numpy()
        o = kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S)
        pick = lambda t: t[ns, hs][:, None]
        o_ref, S_ref = oracle.decode_step(pick(x["q"]), pick(x["k"]), pick(x["v"]),
                                          pick(x["log_alpha"]), pick(x["beta"]), S_ref)
        worst = max(worst, rel_err(o[ns, hs], o_ref[:, 0]))
        if s in (0, 1, steps - 1):
            o_all, S_all = oracle.decode_step(x["q"], x["k"], x["v"], x["log_alpha"],
                                              x["beta"], S_all)
            torch.cuda.synchronize()
            eo, es = rel_err(o, o_all), rel_err(S, S_all)
            print(f"[parity] decode step {s}, all {N * H} pairs: o {eo:.2e} S {es:.2e}")
            assert eo < 2e-2
            assert es < 1e-2
    torch.cuda.synchronize()
    es = rel_err(S[ns, hs], S_ref[:, 0])
    print(f"[parity] decode: worst o {worst:.2e} S after 1000 steps {es:.2e}")
    assert worst < 2e-2
    assert es < 1e-2
    assert bool(torch.isfinite(S).all())


def test_workload_draft_sampled_sessions(kda):
    """Speculative decode at the benchmark's size (64 sessions x 96 heads, 8
    draft tokens, fp32 state): 20 rounds of verify then commit with seeded
    accepted counts in [0, 9] (9 clamps to 8); 12 sampled (session, head) pairs
    follow the oracle round by round."""
    p = I.PRESETS["draft"]
    N, K, H, d = p["N"], p["K"], p["H"], p["d"]
    S = I.decode_state(N, H, d, d, p["s0_std"], seed=3, device=DEV)
    g = torch.Generator().manual_seed(4)
    pairs = [(int(n), int(h)) for n, h in zip(torch.randint(0, N, (12,), generator=g),
                                              torch.randint(0, H, (12,), generator=g))]
    ns = torch.tensor([a for a, _ in pairs], device=DEV)
    hs = torch.tensor([b for _, b in pairs], device=DEV)
    S_ref = S[ns, hs].double().cpu().numpy()[:, None]          # [12, 1, d, d]
    worst = 0.0
    for r in range(20):
        x = I.draft_tokens(N, K, H, d, d, p["dtype"], p["la"], seed=100 + r, device=DEV)
        ins = tuple(x[key] for key in ("q", "k", "v", "log_alpha", "beta"))
        acc = torch.randint(0, K + 2, (N,), generator=g, dtype=torch.int32).to(DEV)
        o = kda.kda_verify_tokens(*ins, S)
        kda.kda_commit_tokens(*ins, S, n_accept=acc)
        pick = [t[ns, :, hs].unsqueeze(2) for t in ins]
        o_ref = oracle.verify_tokens(*pick, S_ref)
        S_ref = oracle.commit_tokens(*pick, S_ref, acc[ns].cpu().numpy())
        worst = max(worst, rel_err(o[ns, :, hs], o_ref[:, :, 0]))
    torch.cuda.synchronize()
    es = rel_err(S[ns, hs], S_ref[:, 0])
    print(f"[parity] draft: worst o {worst:.2e} S after 20 rounds {es:.2e}")
    assert worst < 2e-2
    assert es < 1e-2
    assert bool(torch.isfinite(S).all())


@pytest.mark.parametrize("engine", ENGINES)
def test_workload_varlen_then_decode(kda, engine):
    """16 packed sequences (lengths log-uniform in [1024, 65536]), H=96, bf16,
    per-sequence S0; then 256 decode steps per sequence from the returned
    states.  24 seeded heads of every sequence follow the oracle through the
    prefill (o of every token, S_T) and every decode step."""
    p = I.PRESETS["varlen"]
    prob = I.preset_problem("varlen", seed=0, device=DEV)
    o, ST = run_fwd(kda, prob, engine)
    heads = I.sampled_heads(p["H"], 24, seed=0)
    o_ref, S_ref = cached_oracle("varlen", prob, heads)
    idx = torch.tensor(heads, device=DEV)
    eo, es = rel_err(o.index_select(1, idx), o_ref), rel_err(ST.index_select(1, idx), S_ref)
    print(f"[parity] varlen {engine}, 24 heads x 16 sequences: o {eo:.2e} S {es:.2e}")
    assert eo < 2e-2
    assert es < 1e-2
    # each sequence on its own, so that no sequence hides behind another's scale
    cu = prob.cu_seqlens.cpu().tolist()
    o_sel = o.index_select(1, idx)
    for i in range(len(cu) - 1):
        assert rel_err(o_sel[cu[i]:cu[i + 1]], o_ref[cu[i]:cu[i + 1]]) < 2e-2
        assert rel_err(ST[i].index_select(0, idx), S_ref[i]) < 1e-2
    N, H, d = p["n_seq"], p["H"], p["d"]
    S = ST.clone()
    S_o = S_ref
    worst = 0.0
    for s in range(p["decode_steps"]):
        x = I.decode_token(N, H, d, d, p["dtype"], p["la"], seed=1, step=s, device=DEV)
        od = kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S)
        pick = lambda t: t.index_select(1, idx)
        od_ref, S_o = oracle.decode_step(pick(x["q"]), pick(x["k"]), pick(x["v"]),
                                         pick(x["log_alpha"]), pick(x["beta"]), S_o)
        worst = max(worst, rel_err(od.index_select(1, idx), od_ref))
    torch.cuda.synchronize()
    es = rel_err(S.index_select(1, idx), S_o)
    print(f"[parity] varlen decode {engine}: worst o {worst:.2e} S after 256 steps {es:.2e}")
    assert worst < 2e-2
    assert es < 1e-2


# ------------------------- closed form at full size: every token of every head
#
# With q_t = k_t and beta_t = 1 the output reads back the token's own value,
# for any gates and any initial state: after the decay, r = S~^T k_t, and
# S_t^T k_t = r + (v_t - r)(k_t^T k_t) = v_t when |k_t| = 1 ("Kimi Delta
# Attention 完全拆解", section 从线性注意力到 Delta Rule: with a unit key and
# beta = 1 the erase removes the state's whole component along k_t before the
# write).  The keys are
# unit vectors rounded to the input dtype, so o_t = v_t up to that rounding
# times |v_t - r| and the kernels' own rounding.  Unlike the oracle
# comparisons, which sample heads, these check every output of a full-size call.

def read_back_err(o, v):
    o, v = o.float(), v.float()
    return ((o - v).abs().max() / v.abs().max()).item()


def unit_beta(prob):
    prob.q = prob.k.clone()
    prob.beta = torch.ones_like(prob.beta)
    return prob


@pytest.mark.parametrize("engine,dtype", [("tensorcore", "bf16"), ("cudacore", "bf16"),
                                          ("cudacore", "f32")])
def test_workload_prefill_every_output_reads_back_v(kda, engine, dtype):
    """B=1, H=96, T=8192, d=128, nonzero S0: o_t = v_t on all 786,432 token-heads;
    S_T of every head against the oracle (o = v does not see the state that
    the chunks hand on, S_T does)."""
    p = I.PRESETS["prefill"]
    prob = unit_beta(I.prefill_problem(1, p["T"], p["H"], p["d"], p["d"], dtype, p["la"], 0.02,
                                       seed=7, device=DEV))
    o, ST = run_fwd(kda, prob, engine)
    err = read_back_err(o, prob.v)
    _, S_ref = cached_oracle(("read_back", dtype), prob, list(range(p["H"])))
    es = rel_err(ST, S_ref)
    print(f"[closed form] prefill {engine} {dtype}: max |o - v| / max |v| = {err:.2e}, "
          f"S_T vs oracle {es:.2e}")
    assert err < tol_o(prob.q.dtype)
    assert es < tol_s(prob.q.dtype)


def test_workload_long_tp8_segment_parallel_reads_back_v(kda):
    """B=1, H=12, T=131072 through kda_fwd_cp (the automatic segment count):
    o_t = v_t on every token, across every segment boundary the scan composes;
    S_T of all 12 heads against the oracle."""
    prob = unit_beta(I.preset_problem("long_tp8", seed=8, device=DEV))
    o, ST = run_cp(kda, prob, "auto", None)
    err = read_back_err(o, prob.v)
    _, S_ref = oracle_on_heads(prob, list(range(12)))
    es = rel_err(ST, S_ref)
    print(f"[closed form] segment-parallel long_tp8: {err:.2e}, S_T vs oracle {es:.2e}")
    assert err < 2e-2
    assert es < 1e-2


def test_workload_decode_and_draft_read_back_v(kda):
    """64 sessions x 96 heads, fp32 state: three decode steps, then a verify of
    8 draft tokens and their commit, all with q = k and beta = 1: every output
    of every session and head is its own v.  The state of all 6,144 pairs
    follows the oracle through the same steps (o = v does not see it)."""
    p = I.PRESETS["decode"]
    N, H, d = p["N"], p["H"], p["d"]
    S = I.decode_state(N, H, d, d, p["s0_std"], seed=9, device=DEV)
    S_ref = S.double().cpu().numpy()
    for s in range(3):
        x = I.decode_token(N, H, d, d, p["dtype"], p["la"], seed=9, step=s, device=DEV)
        ones = torch.ones_like(x["beta"])
        o = kda.kda_decode_step(x["k"], x["k"], x["v"], x["log_alpha"], ones, S)
        _, S_ref = oracle.decode_step(x["k"], x["k"], x["v"], x["log_alpha"], ones, S_ref)
        torch.cuda.synchronize()
        err = read_back_err(o, x["v"])
        print(f"[closed form] decode step {s}: {err:.2e}")
        assert err < 2e-2
    K = I.PRESETS["draft"]["K"]
    x = I.draft_tokens(N, K, H, d, d, p["dtype"], p["la"], seed=10, device=DEV)
    ins = (x["k"], x["k"], x["v"], x["log_alpha"], torch.ones_like(x["beta"]))
    o = kda.kda_verify_tokens(*ins, S)
    kda.kda_commit_tokens(*ins, S)
    S_ref = oracle.commit_tokens(*ins, S_ref)
    torch.cuda.synchronize()
    err = read_back_err(o, x["v"])
    es = rel_err(S, S_ref)
    print(f"[closed form] verify of {K} draft tokens: {err:.2e}; state of every pair after "
          f"the commit vs oracle {es:.2e}")
    assert err < 2e-2
    assert es < 1e-2
    # after the commit, one more step reads back too (the committed state is a
    # valid state; any state gives the property)
    y = I.decode_token(N, H, d, d, p["dtype"], p["la"], seed=11, step=0, device=DEV)
    o = kda.kda_decode_step(y["k"], y["k"], y["v"], y["log_alpha"], torch.ones_like(y["beta"]), S)
    torch.cuda.synchronize()
    assert read_back_err(o, y["v"]) < 2e-2
    assert bool(torch.isfinite(S).all())


def test_binding_rejects_mis_shaped_buffers(kda):
    """The C ABI takes bare pointers, so the binding checks every buffer's shape
    before the call: a wrong-sized o, S_T, S0 or decode / draft operand raises
    ValueError and nothing is launched (the caller's buffers stay untouched)."""
    prob = I.prefill_problem(1, 100, 2, 64, 64, "f32", (-0.5, -0.001), 0.05, seed=1, device=DEV)
    args = (prob.q, prob.k, prob.v, prob.log_alpha, prob.beta)
    o_bad = torch.full((1, 99, 2, 64), 7.0, device=DEV)
    with pytest.raises(ValueError):
        kda.kda_fwd(*args, prob.S0, o=o_bad)
    assert bool((o_bad == 7.0).all())
    with pytest.raises(ValueError):
        kda.kda_fwd(*args, prob.S0, S_T=torch.empty(1, 2, 64, 32, device=DEV))
    with pytest.raises(ValueError):
        kda.kda_fwd(*args, prob.S0[:, :1].contiguous())
    with pytest.raises(ValueError):
        kda.kda_fwd_cp(*args, prob.S0, segments=2, o=o_bad)
    with pytest.raises(ValueError):
        kda.kda_fwd_noalloc(*args, torch.zeros(2, 2, 64, 64, device=DEV))
    x = I.decode_token(2, 2, 64, 64, "f32", seed=1, device=DEV)
    S = torch.zeros(2, 2, 64, 64, device=DEV)
    with pytest.raises(ValueError):
        kda.kda_decode_step(x["q"], x["k"][:1].contiguous(), x["v"], x["log_alpha"], x["beta"], S)
    with pytest.raises(ValueError):
        kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S,
                            o=torch.empty(2, 2, 32, device=DEV))
    y = I.draft_tokens(2, 3, 2, 64, 64, "f32", seed=1, device=DEV)
    with pytest.raises(ValueError):
        kda.kda_verify_tokens(y["q"], y["k"], y["v"], y["log_alpha"], y["beta"], S,
                              o=torch.empty(2, 3, 2, 32, device=DEV))
    torch.cuda.synchronize()
    assert bool((S == 0).all())


@pytest.mark.parametrize("H", [70, 152])
def test_full_grid_variant_matches_oracle(kda, H):
    """A grid that keeps (nearly) every SM busy runs the tensor-core kernel's
    full-grid variant (the bf16 diagonal blocks of T' written by other warps):
    2 x H blocks here, ragged T and nonzero S0, sampled heads against the oracle."""
    prob = I.prefill_problem(2, 333, H, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=H,
                             device=DEV)
    o, ST = run_fwd(kda, prob, "tensorcore")
    heads = I.sampled_heads(H, 4, seed=1)
    o_ref, S_ref = oracle_on_heads(prob, heads)
    idx = torch.tensor(heads, device=DEV)
    assert rel_err(o.index_select(2, idx), o_ref) < 2e-2
    assert rel_err(ST.index_select(1, idx), S_ref) < 1e-2
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(ST).all())
