"""GPU parity of the fused output epilogue (head-wise RMSNorm times a sigmoid
gate) against the fp64 oracle: kda_fwd_gated on both engines, the fused decode
step and the stand-alone pass, y = sigmoid(g) * w * o / sqrt(mean(o^2) + eps)
with o from the oracle's recurrence.  Tolerances as for o: max-abs error over
max |y_ref|, 1e-4 for fp32 inputs and 2e-2 for bf16."""
import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrence_chunkwise_gb300 import build as kbuild
from linear_attention_recurrence_chunkwise_gb300 import inputs as I
from tests.gpu_util import cached_oracle, oracle_on_heads, rel_err, tol_o

pytestmark = pytest.mark.gpu
DEV = "cuda"
EPS = 1e-6


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    kbuild.build()
    from linear_attention_recurrence_chunkwise_gb300 import kda as mod
    mod.load()
    return mod


def gate_inputs(like, seed):
    """Gate logits ~ N(0, 2) in o's dtype and a norm weight ~ U(0.5, 1.5)."""
    g = torch.Generator(device=like.device).manual_seed(seed)
    gate = (2.0 * torch.randn(like.shape, generator=g, device=like.device)).to(like.dtype)
    w = torch.rand(like.shape[-1], generator=g, device=like.device) + 0.5
    return gate, w


def y_ref(o_ref, gate, w, eps=EPS):
    return oracle.gated_rmsnorm(o_ref, gate, w, eps)


@pytest.mark.parametrize("engine,epilogue", [("cudacore", "separate"), ("cudacore", "auto"),
                                             ("tensorcore", "fused"),
                                             ("tensorcore", "separate")])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T", [1, 65, 200])
def test_gated_prefill_small(kda, engine, epilogue, dtype, d, T):
    if engine == "tensorcore" and d == 128 and dtype != "bf16":
        pytest.skip("the tensor-core engine takes fp32 at d = 64 only")
    if engine == "tensorcore" and epilogue == "fused" and d != 128:
        pytest.skip("the fused epilogue lives in the d = 128 tensor-core kernel")
    prob = I.prefill_problem(2, T, 3, d, d, dtype, (-0.5, -0.001), 0.05, seed=T + d + 5,
                             device=DEV)
    gate, w = gate_inputs(prob.v, seed=T)
    y, ST = kda.kda_fwd_gated(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0,
                              g=gate, norm_weight=w, eps=EPS, engine=engine,
                              epilogue=epilogue)
    o, ST_plain = kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0,
                              engine=engine)
    torch.cuda.synchronize()
    assert torch.equal(ST, ST_plain)          # the epilogue leaves the state alone
    o_ref, _ = oracle_on_heads(prob, [0, 1, 2])
    e = rel_err(y, y_ref(o_ref, gate, w))
    assert e < tol_o(prob.q.dtype), e


def test_gated_fused_needs_the_d128_tensor_core_kernel(kda):
    prob = I.prefill_problem(1, 70, 2, 64, 64, "f32", (-0.5, -0.001), 0.05, seed=1, device=DEV)
    gate, w = gate_inputs(prob.v, seed=1)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_fwd_gated(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0, g=gate,
                          norm_weight=w, epilogue="fused")
    assert e.value.status == kda.KDA_ERR_UNSUPPORTED


@pytest.mark.parametrize("engine,epilogue", [("cudacore", "auto"), ("tensorcore", "fused"),
                                             ("tensorcore", "separate")])
def test_gated_prefill_varlen_wide_gates_no_weight(kda, engine, epilogue):
    """Packed sequences with empty, one-token and ragged ones; one head with
    gates past the chunk form's range (its outputs come from the token-serial
    pass, which applies the epilogue itself); no norm weight; a larger eps."""
    lengths = [130, 0, 1, 257, 64]
    prob = I.prefill_problem(1, 0, 3, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=12,
                             device=DEV, lengths=lengths)
    la = prob.log_alpha.cpu()
    la[:, 1] = -(torch.rand(la[:, 1].shape, generator=torch.Generator().manual_seed(3)) * 4.5
                 + 0.5)
    prob.log_alpha.copy_(la.to(DEV))
    gate, _ = gate_inputs(prob.v, seed=13)
    y, _ = kda.kda_fwd_gated(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0,
                             prob.cu_seqlens, g=gate, norm_weight=None, eps=1e-2,
                             engine=engine, epilogue=epilogue)
    torch.cuda.synchronize()
    o_ref, _ = oracle_on_heads(prob, [0, 1, 2])
    e = rel_err(y, y_ref(o_ref, gate, None, 1e-2))
    assert e < 2e-2, e


@pytest.mark.parametrize("engine,epilogue", [("tensorcore", "fused"),
                                             ("tensorcore", "separate"),
                                             ("cudacore", "auto")])
def test_gated_workload_prefill_all_heads(kda, engine, epilogue):
    """B=1, H=96, T=8192, d=128, bf16 with the epilogue: y of every head."""
    prob = I.preset_problem("prefill", seed=0, device=DEV)
    gate, w = gate_inputs(prob.v, seed=99)
    y, _ = kda.kda_fwd_gated(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0,
                             g=gate, norm_weight=w, eps=EPS, engine=engine, epilogue=epilogue)
    torch.cuda.synchronize()
    o_ref, _ = cached_oracle("prefill", prob, list(range(96)))
    e = rel_err(y, y_ref(o_ref, gate, w))
    print(f"[parity] gated prefill {engine} {epilogue}, all 96 heads: y {e:.2e}")
    assert e < 2e-2


@pytest.mark.parametrize("epilogue", ["fused", "separate"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_gated_decode_steps(kda, dtype, d, epilogue):
    N, H, steps = 3, 5, 6
    S = I.decode_state(N, H, d, d, 0.05, seed=d, device=DEV)
    S_ref = S.double().cpu().numpy()
    S_plain = S.clone()
    for s in range(steps):
        x = I.decode_token(N, H, d, d, dtype, (-0.1, -0.0005), seed=d, step=s, device=DEV)
        gate, w = gate_inputs(x["v"], seed=s)
        y = kda.kda_decode_step_gated(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S,
                                      g=gate, norm_weight=w, eps=EPS, epilogue=epilogue)
        kda.kda_decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S_plain)
        o_ref, S_ref = oracle.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                          S_ref)
        torch.cuda.synchronize()
        assert rel_err(y, y_ref(o_ref, gate, w)) < tol_o(x["q"].dtype)
    assert torch.equal(S, S_plain)


@pytest.mark.parametrize("epilogue", ["fused", "separate"])
def test_gated_decode_workload(kda, epilogue):
    """64 sessions x 96 heads, fp32 state: three steps with the epilogue, every
    pair (the fused kernel rotates four buffers per block: many pairs each)."""
    p = I.PRESETS["decode"]
    N, H, d = p["N"], p["H"], p["d"]
    S = I.decode_state(N, H, d, d, p["s0_std"], seed=5, device=DEV)
    S_ref = S.double().cpu().numpy()
    for s in range(3):
        x = I.decode_token(N, H, d, d, p["dtype"], p["la"], seed=5, step=s, device=DEV)
        gate, w = gate_inputs(x["v"], seed=40 + s)
        y = kda.kda_decode_step_gated(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S,
                                      g=gate, norm_weight=w, eps=EPS, epilogue=epilogue)
        o_ref, S_ref = oracle.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                          S_ref)
        torch.cuda.synchronize()
        e = rel_err(y, y_ref(o_ref, gate, w))
        print(f"[parity] gated decode {epilogue} step {s}, all pairs: y {e:.2e}")
        assert e < 2e-2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_gated_rmsnorm_alone_and_in_place(kda, dtype, d):
    dt = I.DTYPES[dtype]
    gen = torch.Generator(device=DEV).manual_seed(d)
    o = torch.randn((333, 7, d), generator=gen, device=DEV).mul_(
        torch.logspace(-3, 3, 7, device=DEV)[None, :, None]).to(dt)
    gate, w = gate_inputs(o, seed=d + 1)
    y = kda.kda_gated_rmsnorm(o, gate, w, 1e-5)
    ref = y_ref(o.double().cpu().numpy(), gate, w, 1e-5)
    torch.cuda.synchronize()
    assert rel_err(y, ref) < (1e-5 if dtype == "f32" else 8e-3)
    o2 = o.clone()
    kda.kda_gated_rmsnorm(o2, gate, w, 1e-5, y=o2)
    torch.cuda.synchronize()
    assert torch.equal(o2, y)
