"""GPU parity of the input prologue (ShortConv(4), Swish, L2Norm of q and k)
against the fp64 oracle: whole sequences (fixed length and packed, with and
without an initial conv state, the final state written over the initial one),
decode steps chained through the state, pieces chained through the state, the
full prefill shape on every head, the bounds-checked build, and the decode
layer step that fuses the prologue, the recurrence and the output epilogue.
Tolerances (max-abs error / max |oracle|): fp32 1e-5, bf16 outputs 1e-2 (one
bf16 rounding of the result); conv states are copies of inputs and compare
exactly."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrence_chunkwise_gb300 import build as kbuild
from linear_attention_recurrence_chunkwise_gb300 import inputs as I
from tests.gpu_util import rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    kbuild.build()
    from linear_attention_recurrence_chunkwise_gb300 import kda as mod
    mod.load()
    return mod


def tol(dtype):
    return 1e-5 if dtype == "f32" else 1e-2


def make(lead, H, d, dtype, seed, with_state, N):
    """Projected inputs ~ N(0, 1), taps ~ N(0, 0.5), initial states ~ N(0, 1)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    xs = [torch.randn(lead + (H, d), generator=g).to(DT[dtype]).to(DEV) for _ in range(3)]
    ws = [(0.5 * torch.randn((H, d, 4), generator=g)).to(DEV) for _ in range(3)]
    c0 = torch.randn((N, 3, 3, H, d), generator=g).to(DEV) if with_state else None
    return xs, ws, c0


def check(got, ref, dtype):
    q, k, v, st = got
    rq, rk, rv, rst = ref
    for a, b in ((q, rq), (k, rk), (v, rv)):
        assert rel_err(a, b) < tol(dtype)
    assert np.array_equal(st.double().cpu().numpy(), rst)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("with_state", [False, True])
def test_short_conv_fixed_length(kda, dtype, d, with_state):
    """B = 2 sequences of 200 tokens (runs of 64 tokens end mid-sequence and
    one crosses between the sequences), H = 3."""
    xs, ws, c0 = make((2, 200), 3, d, dtype, seed=d + with_state, with_state=with_state, N=2)
    got = kda.kda_short_conv(*xs, *ws, c0, eps=1e-6)
    torch.cuda.synchronize()
    check(got, oracle.prologue(*xs, *ws, c0, eps=1e-6), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_short_conv_varlen_state_in_place(kda, dtype):
    """Packed sequences with empty, one- and two-token ones (shorter than the
    window: their final state keeps part of the initial one) and runs that
    cross several sequences; the final state written over the initial one."""
    lengths = [0, 1, 2, 64, 130, 0, 7, 300, 3]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=DEV)
    xs, ws, c0 = make((int(sum(lengths)),), 4, 128, dtype, seed=7, with_state=True,
                      N=len(lengths))
    ref = oracle.prologue(*xs, *ws, c0, cu.cpu().numpy(), eps=1e-6)
    state = c0.clone()
    q, k, v, _ = kda.kda_short_conv(*xs, *ws, state, cu, eps=1e-6, conv_T=state)
    torch.cuda.synchronize()
    check((q, k, v, state), ref, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_short_conv_pieces_and_steps_equal_one_run(kda, dtype):
    """A sequence run in pieces (of 1, 2, 61 and 96 tokens), each from the
    previous piece's final state, and then token by token with
    kda_short_conv_step, gives the one-run outputs bit for bit."""
    N, T, H, d = 3, 180, 2, 64
    xs, ws, c0 = make((N, T), H, d, dtype, seed=11, with_state=True, N=N)
    q1, k1, v1, s1 = kda.kda_short_conv(*xs, *ws, c0, eps=1e-6)
    cuts = [0, 1, 3, 64, 160]
    state = c0.clone()
    outs = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        piece = [x[:, a:b].contiguous() for x in xs]
        outs.append(kda.kda_short_conv(*piece, *ws, state, eps=1e-6, conv_T=state)[:3])
    for t in range(cuts[-1], T):
        tok = [x[:, t].contiguous() for x in xs]
        outs.append(tuple(o.unsqueeze(1) for o in
                          kda.kda_short_conv_step(*tok, *ws, state, eps=1e-6)))
    torch.cuda.synchronize()
    for i, ref in enumerate((q1, k1, v1)):
        assert torch.equal(torch.cat([o[i] for o in outs], 1), ref)
    assert torch.equal(state, s1)
    check((q1, k1, v1, s1), oracle.prologue(*xs, *ws, c0, eps=1e-6), dtype)


def test_short_conv_workload_all_heads(kda):
    """The prefill shape (B = 1, T = 8192, H = 96, d = 128, bf16) on every
    head against the oracle."""
    xs, ws, c0 = make((1, 8192), 96, 128, "bf16", seed=3, with_state=True, N=1)
    got = kda.kda_short_conv(*xs, *ws, c0, eps=1e-6)
    torch.cuda.synchronize()
    ref = oracle.prologue(*xs, *ws, c0, eps=1e-6)
    errs = [rel_err(a, b) for a, b in zip(got[:3], ref[:3])]
    print(f"[parity] prologue B=1 T=8192 H=96 d=128 bf16: q {errs[0]:.2e} k {errs[1]:.2e} "
          f"v {errs[2]:.2e}")
    check(got, ref, "bf16")


def test_short_conv_unit_rows(kda):
    """q and k come out with unit norm per (token, head) (eps = 0), v does not."""
    xs, ws, _ = make((2, 70), 5, 128, "f32", seed=5, with_state=False, N=2)
    q, k, v, _ = kda.kda_short_conv(*xs, *ws, eps=0.0)
    torch.cuda.synchronize()
    for t in (q, k):
        assert torch.allclose(t.norm(dim=-1), torch.ones(t.shape[:-1], device=DEV), atol=1e-5)
    assert not torch.allclose(v.norm(dim=-1), torch.ones(v.shape[:-1], device=DEV), atol=1e-2)


def test_short_conv_bad_offsets_write_nothing(kda):
    """A device-side cu_seqlens that decreases is reported through the status
    word and nothing is written."""
    xs, ws, c0 = make((100,), 2, 64, "f32", seed=9, with_state=True, N=2)
    bad = torch.tensor([0, 70, 60], dtype=torch.int32, device=DEV)
    outs = [torch.full_like(xs[0], 7.0) for _ in range(3)]
    st = torch.full_like(c0, 7.0)
    ws_buf = torch.zeros(kda.kda_fwd_workspace_bytes(2), dtype=torch.uint8, device=DEV)
    kda.kda_short_conv(*xs, *ws, c0, bad, q=outs[0], k=outs[1], v=outs[2], conv_T=st,
                       workspace=ws_buf)
    assert kda.kda_read_device_status(ws_buf) == kda.KDA_ERR_INVALID_ARGUMENT
    assert all(bool((o == 7.0).all()) for o in outs) and bool((st == 7.0).all())


def test_short_conv_bounds_checked_build(kda):
    """The bounds-checked build: packed sequences with empty and short ones,
    then decode steps -- no report, results against the oracle."""
    lib = kda.load_library(kbuild.build(bounds_check=True))
    lengths = [3, 0, 65, 1, 130]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=DEV)
    xs, ws, c0 = make((int(sum(lengths)),), 2, 128, "f32", seed=13, with_state=True,
                      N=len(lengths))
    wsb = torch.zeros(int(lib.kda_fwd_workspace_bytes(len(lengths))), dtype=torch.uint8,
                      device=DEV)
    got = kda.kda_short_conv(*xs, *ws, c0, cu, eps=1e-6, workspace=wsb, lib=lib)
    torch.cuda.synchronize()
    assert kda.kda_read_device_status(wsb, lib=lib) == kda.KDA_OK
    check(got, oracle.prologue(*xs, *ws, c0, cu.cpu().numpy(), eps=1e-6), "f32")
    tok = [torch.randn(len(lengths), 2, 128, device=DEV) for _ in range(3)]
    state = got[3].clone()
    q, k, v = kda.kda_short_conv_step(*tok, *ws, state, eps=1e-6, lib=lib)
    torch.cuda.synchronize()
    ref = oracle.prologue(*[t[:, None] for t in tok], *ws, got[3], eps=1e-6)
    check((q[:, None], k[:, None], v[:, None], state), ref, "f32")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_layer_step(kda, dtype, d):
    """Three decode tokens through kda_decode_layer_step (prologue, recurrence
    and epilogue in one kernel) against the oracle's prologue -> decode step ->
    gated RMSNorm, and against the three separate calls; the conv state is the
    same copy of the inputs on every path."""
    N, H = 6, 3
    g = torch.Generator(device="cpu").manual_seed(d + (dtype == "bf16"))
    r = lambda *s, sc=1.0: (sc * torch.randn(s, generator=g)).to(DEV)
    ws = [r(H, d, 4, sc=0.5) for _ in range(3)]
    nw = (torch.rand(d, generator=g) + 0.5).to(DEV)
    conv0, S0 = r(N, 3, 3, H, d), r(N, H, d, d, sc=0.02)
    conv_f, S_f = conv0.clone(), S0.clone()
    conv_s, S_s = conv0.clone(), S0.clone()
    conv_o, S_o = conv0.double().cpu().numpy(), S0.double().cpu().numpy()
    tol_y = 1e-4 if dtype == "f32" else 2e-2
    for step in range(3):
        xs = [r(N, H, d).to(DT[dtype]) for _ in range(3)]
        la = -torch.rand((N, H, d), generator=g).to(DEV) * 0.1
        beta = torch.sigmoid(r(N, H))
        gate = r(N, H, d, sc=2.0).to(DT[dtype])
        y_f = kda.kda_decode_layer_step(*xs, *ws, conv_f, la, beta, S_f, gate, nw, eps=1e-5,
                                        l2_eps=1e-6)
        q, k, v = kda.kda_short_conv_step(*xs, *ws, conv_s, eps=1e-6)
        y_s = kda.kda_decode_step_gated(q, k, v, la, beta, S_s, g=gate, norm_weight=nw,
                                        eps=1e-5)
        torch.cuda.synchronize()
        qo, ko, vo, conv_o = oracle.prologue(*[x[:, None] for x in xs], *ws, conv_o, eps=1e-6)
        o_o, S_o = oracle.decode_step(qo[:, 0], ko[:, 0], vo[:, 0], la, beta, S_o)
        y_o = oracle.gated_rmsnorm(o_o, gate, nw, eps=1e-5)
        assert rel_err(y_f, y_o) < tol_y, step
        assert rel_err(y_f, y_s.double().cpu().numpy()) < tol_y, step
        assert np.array_equal(conv_f.double().cpu().numpy(), conv_o)
        assert torch.equal(conv_f, conv_s)
    assert rel_err(S_f, S_o) < (1e-4 if dtype == "f32" else 1e-2)
