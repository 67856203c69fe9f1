"""kda_fwd_noalloc, the entry point for callers that cannot allocate device
memory, against kda_fwd (GPU).

kda_fwd takes a caller-allocated workspace; kda_fwd_noalloc keeps that scratch
in a fixed array inside the library, for callers that run where allocating is
not possible.  Both must give the same results.  This file is collected last
so that a run stopping at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from linear_attention_recurrence_chunkwise_gb300 import build as kbuild
from linear_attention_recurrence_chunkwise_gb300 import inputs as I
from tests.gpu_util import rel_err

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


def call_noalloc(lib, prob, o, S_T, status, stream):
    """Call kda_fwd_noalloc through the C ABI with raw device pointers."""
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    H, d = prob.q.shape[-2], prob.q.shape[-1]
    N = prob.cu_seqlens.numel() - 1
    return lib.kda_fwd_noalloc(P(prob.q), P(prob.k), P(prob.v), P(prob.log_alpha),
                               P(prob.beta), P(prob.S0), P(prob.cu_seqlens), 1,
                               prob.q.shape[0], H, d, d, N, 1, P(o), P(S_T), P(status),
                               ctypes.c_void_p(stream.cuda_stream))


def test_noalloc_matches_kda_fwd_on_two_calls_in_a_row(kda):
    """Two calls in a row, each against kda_fwd on the same inputs: the same
    kernels run on the same data, so o and S_T agree bit for bit."""
    lib = kda.load()
    stream = torch.cuda.current_stream()
    cases = [([300, 64, 1, 129, 0], 21), ([1000, 7, 250], 22)]
    for lengths, seed in cases:
        prob = I.prefill_problem(1, 0, 4, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=seed,
                                 device=DEV, lengths=lengths)
        o_ref, S_ref = kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta,
                                   prob.S0, prob.cu_seqlens)
        o = torch.full_like(prob.v, float("nan"))
        S_T = torch.full_like(S_ref, float("nan"))
        status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
        rc = call_noalloc(lib, prob, o, S_T, status, stream)
        torch.cuda.synchronize()
        assert rc == kda.KDA_OK
        assert int(status.item()) == kda.KDA_OK
        assert torch.equal(o, o_ref)
        assert torch.equal(S_T, S_ref)
        # and within the oracle's tolerance of kda_fwd, as every engine is
        assert rel_err(o, o_ref.double().cpu().numpy()) < 2e-2


def test_noalloc_error_status_then_a_clean_call(kda):
    """Device-side cu_seqlens that decrease: the call returns KDA_OK on the host
    (it cannot see device memory), reports KDA_ERR_INVALID_ARGUMENT through
    device_status and writes no output.  The status lives in the shared scratch
    array; the next, valid call clears it, reports KDA_OK and matches kda_fwd."""
    lib = kda.load()
    stream = torch.cuda.current_stream()
    prob = I.prefill_problem(1, 0, 2, 128, 128, "bf16", (-0.5, -0.001), 0.05, seed=23,
                             device=DEV, lengths=[50, 50])
    good_cu = prob.cu_seqlens
    prob.cu_seqlens = torch.tensor([0, 70, 60], dtype=torch.int32, device=DEV)  # decreasing
    o = torch.full_like(prob.v, 7.0)
    S_T = torch.full_like(prob.S0, 7.0)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    rc = call_noalloc(lib, prob, o, S_T, status, stream)
    torch.cuda.synchronize()
    assert rc == kda.KDA_OK
    assert int(status.item()) == kda.KDA_ERR_INVALID_ARGUMENT
    assert bool((o == 7.0).all()) and bool((S_T == 7.0).all())
    prob.cu_seqlens = good_cu
    status.fill_(-1)
    rc = call_noalloc(lib, prob, o, S_T, status, stream)
    torch.cuda.synchronize()
    assert rc == kda.KDA_OK
    assert int(status.item()) == kda.KDA_OK
    o_ref, S_ref = kda.kda_fwd(prob.q, prob.k, prob.v, prob.log_alpha, prob.beta, prob.S0,
                               prob.cu_seqlens)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(S_T, S_ref)


def test_noalloc_rejects_more_sequences_than_its_scratch_holds(kda):
    lib = kda.load()
    n = kda.KDA_NOALLOC_MAX_SEQS + 1
    cu = torch.zeros(n + 1, dtype=torch.int32, device=DEV)
    x = torch.zeros(1, 1, 128, dtype=torch.bfloat16, device=DEV)
    f = torch.zeros(1, 1, 128, device=DEV)
    b = torch.zeros(1, 1, device=DEV)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.kda_fwd_noalloc(P(x), P(x), P(x), P(f), P(b), None, P(cu), 1, 0, 1, 128, 128, n,
                             1, P(x), None, None, None)
    assert rc == kda.KDA_ERR_WORKSPACE
