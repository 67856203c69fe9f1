"""The tensor-core prefills' timeout paths, on a GPU, without a fault or a hang.

Every mbarrier wait in the tensor-core prefill kernels gives up after a time
limit; the kernel then records KDA_ERR_TIMEOUT, skips its remaining waits,
drains its copies and products, frees tensor memory and exits, and the CUDA
context stays usable.  A test-only build of the library (libkda_timeout.so)
sets the limit to 2 ms and leaves out the one mbarrier arrive that announces
the second chunk's T' to the carry warps -- an arrive nothing else makes -- so
the carry's wait for it runs out; in the d = 64 engine it leaves out the TMA
copy of the second chunk's rows, so the wait for them runs out.  The call must
report the timeout through the workspace status word, and ordinary calls must
still work afterwards."""
import pytest
import torch

from linear_attention_recurrence_chunkwise_gb300 import build as kbuild
from linear_attention_recurrence_chunkwise_gb300 import inputs as I
from tests.gpu_util import oracle_on_heads, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    kbuild.build()
    from linear_attention_recurrence_chunkwise_gb300 import kda as mod
    mod.load()
    return mod


def test_wait_limit_reports_timeout_and_context_survives(kda):
    probe = kda.load_library(kbuild.build(timeout_probe=True))
    # one sequence, one head, two 64-token chunks: the carry waits for chunk 1's T'
    prob = I.prefill_problem(1, 128, 1, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=5,
                             device=DEV)
    for _ in range(2):  # twice in a row: the second call starts from a clean state
        ws = torch.zeros(kda.kda_fwd_workspace_bytes(1), dtype=torch.uint8, device=DEV)
        kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0, workspace=ws,
                    engine="tensorcore", lib=probe)
        assert kda.kda_read_device_status(ws, lib=probe) == kda.KDA_ERR_TIMEOUT
    # the context is usable: ordinary calls run and match the oracle
    ws = torch.zeros(kda.kda_fwd_workspace_bytes(1), dtype=torch.uint8, device=DEV)
    o, ST = kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0,
                        workspace=ws, engine="tensorcore")
    assert kda.kda_read_device_status(ws) == kda.KDA_OK
    o_ref, S_ref = oracle_on_heads(prob, [0])
    assert rel_err(o, o_ref) < 2e-2
    assert rel_err(ST, S_ref) < 1e-2
    # a one-chunk call of the test build never reaches the left-out arrive
    one = I.prefill_problem(1, 64, 1, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=6,
                            device=DEV)
    ws.zero_()
    o1, S1 = kda.kda_fwd(one.q, one.k, one.v, one.log_alpha, one.beta, one.S0, workspace=ws,
                         engine="tensorcore", lib=probe)
    assert kda.kda_read_device_status(ws, lib=probe) == kda.KDA_OK
    o1_ref, S1_ref = oracle_on_heads(one, [0])
    assert rel_err(o1, o1_ref) < 2e-2
    assert rel_err(S1, S1_ref) < 1e-2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_d64_engine_wait_limit_reports_timeout(kda, dtype):
    """The d = 64 tensor-core engine's timeout path: in the test-only build the
    TMA copy of chunk 1's rows is never issued, so the wait for it runs out of
    time; the call reports KDA_ERR_TIMEOUT, a one-chunk call of the same build
    and ordinary calls afterwards still match the oracle."""
    probe = kda.load_library(kbuild.build(timeout_probe=True))
    prob = I.prefill_problem(1, 128, 2, 64, 64, dtype, (-0.5, -0.001), 0.05, seed=7,
                             device=DEV)
    tol = (1e-4, 1e-4) if dtype == "f32" else (2e-2, 1e-2)
    for _ in range(2):
        ws = torch.zeros(kda.kda_fwd_workspace_bytes(1), dtype=torch.uint8, device=DEV)
        kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0, workspace=ws,
                    engine="tensorcore", lib=probe)
        assert kda.kda_read_device_status(ws, lib=probe) == kda.KDA_ERR_TIMEOUT
    one = I.prefill_problem(1, 64, 2, 64, 64, dtype, (-0.5, -0.001), 0.05, seed=8, device=DEV)
    ws = torch.zeros(kda.kda_fwd_workspace_bytes(1), dtype=torch.uint8, device=DEV)
    o1, S1 = kda.kda_fwd(one.q, one.k, one.v, one.log_alpha, one.beta, one.S0, workspace=ws,
                         engine="tensorcore", lib=probe)
    assert kda.kda_read_device_status(ws, lib=probe) == kda.KDA_OK
    o1_ref, S1_ref = oracle_on_heads(one, [0, 1])
    assert rel_err(o1, o1_ref) < tol[0]
    assert rel_err(S1, S1_ref) < tol[1]
    ws.zero_()
    o, ST = kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0,
                        workspace=ws, engine="tensorcore")
    assert kda.kda_read_device_status(ws) == kda.KDA_OK
    o_ref, S_ref = oracle_on_heads(prob, [0, 1])
    assert rel_err(o, o_ref) < tol[0]
    assert rel_err(ST, S_ref) < tol[1]
