"""Seeded synthetic inputs for the KDA operator.

This module only draws random tensors; it holds none of the operator's
arithmetic.  The same arrays feed both the GPU library and the fp64 oracle, so
it is the one module both sides of a parity check use.

Draw order for a prefill problem (one ``torch.Generator`` seeded once):
q, k, v, log_alpha, beta, S0.  q and k are drawn from N(0, 1) and
L2-normalised per (token, head) in fp32 before the cast to the storage dtype
(the pages put L2Norm in the q/k parameterisation, outside the recurrence).
beta = sigmoid(N(0, 1)); log_alpha ~ U(lo, hi); v ~ N(0, 1); S0 ~ N(0, s0_std)
when requested (else None = zero state).

Workload presets (the five problem shapes the operator is specified on):

============  =================================================================
name          shape
============  =================================================================
tiny          B=1, H=2, T=256, d=64, fp32 q/k/v, log_alpha U(-0.5, -0.001)
prefill       B=1, H=96, T=8192, d=128, bf16 q/k/v, log_alpha U(-0.5, -0.001)
decode        64 sessions, H=96, d=128, fp32 state N(0, 0.02), per step bf16
              q/k/v, log_alpha U(-0.1, -0.0005); 1000 steps, step s seeded
              from (seed, s)
long          B=1, H=96, T=131072, d=128, bf16, S0 N(0, 0.02),
              log_alpha U(-0.05, -0.0001)
varlen        16 sequences, lengths round(exp(U(ln 1024, ln 65536))), H=96,
              d=128, bf16, per-sequence S0 N(0, 0.02), then 256 decode steps
============  =================================================================
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

PRESETS = {
    "tiny": dict(B=1, H=2, T=256, d=64, dtype="f32", la=(-0.5, -0.001), s0_std=None),
    "prefill": dict(B=1, H=96, T=8192, d=128, dtype="bf16", la=(-0.5, -0.001), s0_std=None),
    "long": dict(B=1, H=96, T=131072, d=128, dtype="bf16", la=(-0.05, -0.0001), s0_std=0.02),
    # the long prefill on the 12 heads one GPU holds when tensor parallelism
    # splits K3's 96 heads over 8 GPUs (the segment-parallel workload)
    "long_tp8": dict(B=1, H=12, T=131072, d=128, dtype="bf16", la=(-0.05, -0.0001),
                     s0_std=0.02),
    "varlen": dict(n_seq=16, H=96, d=128, dtype="bf16", la=(-0.5, -0.001), s0_std=0.02,
                   len_lo=1024, len_hi=65536, decode_steps=256),
    "decode": dict(N=64, H=96, d=128, dtype="bf16", la=(-0.1, -0.0005), s0_std=0.02, steps=1000),
    # speculative decode on the decode state: the last verified token plus a
    # 7-token draft (the draft depth the K3 MTP layer is unrolled to)
    "draft": dict(N=64, H=96, d=128, dtype="bf16", la=(-0.1, -0.0005), s0_std=0.02, K=8),
}

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def step_seed(seed: int, step: int) -> int:
    """Integer seed for draw number `step` of a run seeded with `seed`."""
    return (int(seed) + 1) * 1_000_003 + int(step)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def _unit_rows(shape, gen, device, dtype):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    return x.to(dtype)


@dataclass
class Problem:
    """One prefill problem in packed layout (token axis first)."""
    q: torch.Tensor            # [Ttot, H, dk]  (or [B, T, H, dk])
    k: torch.Tensor
    v: torch.Tensor            # [.., H, dv]
    log_alpha: torch.Tensor    # [.., H, dk] fp32
    beta: torch.Tensor         # [.., H] fp32
    S0: torch.Tensor | None    # [N, H, dv, dk] fp32
    cu_seqlens: torch.Tensor | None  # [N+1] int32, or None for a fixed-length batch

    @property
    def n_seq(self) -> int:
        if self.cu_seqlens is not None:
            return self.cu_seqlens.numel() - 1
        return self.q.shape[0]


def prefill_problem(B: int, T: int, H: int, dk: int, dv: int, dtype="bf16",
                    la=(-0.5, -0.001), s0_std=None, seed: int = 0, device="cpu",
                    lengths=None) -> Problem:
    """Draw one prefill problem.

    With `lengths` (a list of sequence lengths) the problem is packed varlen:
    tensors are [sum(lengths), H, .] and cu_seqlens holds the offsets.
    Otherwise tensors are [B, T, H, .] with cu_seqlens None.
    """
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    gen = _gen(seed, device)
    if lengths is not None:
        lead = (int(sum(lengths)),)
        n = len(lengths)
        cu = torch.zeros(n + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(list(lengths), dtype=torch.int64), 0).to(torch.int32)
        cu = cu.to(device)
    else:
        lead = (B, T)
        n = B
        cu = None
    q = _unit_rows(lead + (H, dk), gen, device, dt)
    k = _unit_rows(lead + (H, dk), gen, device, dt)
    v = torch.randn(lead + (H, dv), generator=gen, device=device, dtype=torch.float32).to(dt)
    lo, hi = la
    log_alpha = torch.rand(lead + (H, dk), generator=gen, device=device,
                           dtype=torch.float32) * (hi - lo) + lo
    beta = torch.sigmoid(torch.randn(lead + (H,), generator=gen, device=device,
                                     dtype=torch.float32))
    S0 = None
    if s0_std is not None:
        S0 = torch.randn((n, H, dv, dk), generator=gen, device=device,
                         dtype=torch.float32) * float(s0_std)
    return Problem(q, k, v, log_alpha, beta, S0, cu)


def varlen_lengths(n_seq=16, lo=1024, hi=65536, seed: int = 0):
    """Sequence lengths round(exp(U(ln lo, ln hi))), drawn on the CPU."""
    gen = _gen(seed, "cpu")
    u = torch.rand(n_seq, generator=gen, dtype=torch.float64)
    return [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo)))))
            for x in u]


def decode_token(N: int, H: int, dk: int, dv: int, dtype="bf16", la=(-0.1, -0.0005),
                 seed: int = 0, step: int = 0, device="cpu"):
    """Inputs of one decode step for N sessions: dict of q, k, v, log_alpha, beta."""
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    gen = _gen(step_seed(seed, step), device)
    q = _unit_rows((N, H, dk), gen, device, dt)
    k = _unit_rows((N, H, dk), gen, device, dt)
    v = torch.randn((N, H, dv), generator=gen, device=device, dtype=torch.float32).to(dt)
    lo, hi = la
    log_alpha = torch.rand((N, H, dk), generator=gen, device=device,
                           dtype=torch.float32) * (hi - lo) + lo
    beta = torch.sigmoid(torch.randn((N, H), generator=gen, device=device,
                                     dtype=torch.float32))
    return dict(q=q, k=k, v=v, log_alpha=log_alpha, beta=beta)


def draft_tokens(N: int, K: int, H: int, dk: int, dv: int, dtype="bf16",
                 la=(-0.1, -0.0005), seed: int = 0, device="cpu"):
    """K consecutive decode tokens per session, stacked on dim 1: q, k, log_alpha
    [N, K, H, dk], v [N, K, H, dv], beta [N, K, H] (contiguous).  Token t is
    decode_token(..., step=t)."""
    toks = [decode_token(N, H, dk, dv, dtype, la, seed, t, device) for t in range(K)]
    return {key: torch.stack([x[key] for x in toks], dim=1).contiguous()
            for key in ("q", "k", "v", "log_alpha", "beta")}


def decode_state(N: int, H: int, dk: int, dv: int, std=0.02, seed: int = 0, device="cpu"):
    """Initial decode state [N, H, dv, dk] fp32 ~ N(0, std)."""
    gen = _gen(seed, device)
    return torch.randn((N, H, dv, dk), generator=gen, device=device,
                       dtype=torch.float32) * float(std)


def preset_problem(name: str, seed: int = 0, device="cpu") -> Problem:
    """Prefill problem of a named preset ('tiny', 'prefill', 'long', 'long_tp8',
    'varlen')."""
    p = PRESETS[name]
    if name == "varlen":
        lengths = varlen_lengths(p["n_seq"], p["len_lo"], p["len_hi"], seed)
        return prefill_problem(1, 0, p["H"], p["d"], p["d"], p["dtype"], p["la"],
                               p["s0_std"], seed, device, lengths=lengths)
    return prefill_problem(p["B"], p["T"], p["H"], p["d"], p["d"], p["dtype"], p["la"],
                           p["s0_std"], seed, device)


def sampled_heads(H: int, count: int, seed: int = 0):
    """`count` distinct head indices from a seeded permutation of range(H)."""
    gen = _gen(seed, "cpu")
    return sorted(int(x) for x in torch.randperm(H, generator=gen)[:count])
