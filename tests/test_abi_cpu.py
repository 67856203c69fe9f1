"""libkda host-side checks that need no GPU: symbols, accounting, argument errors.

No call here reaches a CUDA API: every call is rejected by host validation (or
by the host-only failure-injection hook) before anything would be enqueued.
"""
import ctypes
import os
import re

import pytest

from linear_attention_recurrence_chunkwise_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kda():
    kbuild.build()
    from linear_attention_recurrence_chunkwise_gb300 import kda as mod
    mod.load()
    return mod


def header_functions():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(kda):
    declared = header_functions()
    assert declared, "no functions parsed from include/kda.h"
    lib = kda.load()
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(kda.EXPORTED) == declared


def test_state_bytes_matches_pages(kda):
    for line in open(os.path.join(ROOT, "tests", "golden", "state_bytes.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = dict(kv.split("=") for kv in line.split())
        got = kda.kda_state_bytes(int(f["layers"]), int(f["N"]), int(f["H"]), int(f["dk"]),
                                  int(f["dv"]), int(f["elem"]))
        assert got == int(f["bytes"]), line


def test_state_bytes_edge_cases(kda):
    assert kda.kda_state_bytes(69, 1, 96, 128, 128, 4) == 2 * 217055232
    assert kda.kda_state_bytes(0, 5, 96, 128, 128, 4) == 0
    assert kda.kda_state_bytes(-1, 1, 1, 1, 1, 1) == 0
    assert kda.kda_state_bytes(2**31 - 1, 2**31 - 1, 2**31 - 1, 2**31 - 1, 2**31 - 1, 4) == 0


def test_status_strings(kda):
    for code, name in [(0, "KDA_OK"), (1, "KDA_ERR_INVALID_ARGUMENT"), (2, "KDA_ERR_UNSUPPORTED"),
                       (3, "KDA_ERR_WORKSPACE"), (4, "KDA_ERR_CUDA"), (5, "KDA_ERR_DOMAIN"),
                       (6, "KDA_ERR_TIMEOUT"), (7, "KDA_ERR_BOUNDS")]:
        assert kda.kda_status_string(code) == name


def test_workspace_bytes(kda):
    assert kda.kda_fwd_workspace_bytes(0) >= 16
    for n in (1, 16, 1000):
        b = kda.kda_fwd_workspace_bytes(n)
        assert b >= 16 + 4 * n and b % 16 == 0


# fake, never dereferenced, 16-byte aligned device addresses
P = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(12)]


def fwd_call(lib, **kw):
    a = dict(q=P[0], k=P[1], v=P[2], la=P[3], beta=P[4], S0=None, cu=None, B=1, T=64, H=2,
             dk=64, dv=64, N=1, dt=0, o=P[5], ST=P[6], ws=P[7], wsb=4096, stream=None,
             engine=0)
    a.update(kw)
    return lib.kda_fwd_engine(a["q"], a["k"], a["v"], a["la"], a["beta"], a["S0"], a["cu"],
                              a["B"], a["T"], a["H"], a["dk"], a["dv"], a["N"], a["dt"],
                              a["o"], a["ST"], a["ws"], a["wsb"], a["stream"], a["engine"])


def test_fwd_argument_errors(kda):
    lib = kda.load()
    E_INV, E_UNS, E_WS = 1, 2, 3
    assert fwd_call(lib, q=None) == E_INV
    assert fwd_call(lib, q=ctypes.c_void_p(0x10008)) == E_INV          # misaligned
    assert fwd_call(lib, S0=ctypes.c_void_p(0x10004)) == E_INV
    assert fwd_call(lib, beta=ctypes.c_void_p(0x10002)) == E_INV      # beta: 4-byte aligned
    assert fwd_call(lib, beta=ctypes.c_void_p(0x10004), ws=None) == E_WS  # 4 B is enough
    assert fwd_call(lib, dt=7) == E_INV
    assert fwd_call(lib, H=0) == E_INV
    assert fwd_call(lib, T=-1) == E_INV
    assert fwd_call(lib, N=2) == E_INV                                # N != B without cu_seqlens
    assert fwd_call(lib, cu=P[8], B=2, N=2) == E_INV                   # varlen needs B = 1
    assert fwd_call(lib, cu=ctypes.c_void_p(0x10002)) == E_INV         # misaligned offsets
    assert fwd_call(lib, dk=96, dv=96) == E_UNS
    assert fwd_call(lib, dk=64, dv=128) == E_UNS
    assert fwd_call(lib, ws=None) == E_WS
    assert fwd_call(lib, wsb=8) == E_WS
    assert fwd_call(lib, engine=9) == E_INV
    # tensor cores: bf16 at d = 128, fp32 or bf16 at d = 64; the blocked-path
    # variant bf16 at d = 128 only
    assert fwd_call(lib, engine=1, dt=0, dk=128, dv=128) == E_UNS
    assert fwd_call(lib, engine=3, dt=0, dk=128, dv=128) == E_UNS
    assert fwd_call(lib, engine=3, dt=1) == E_UNS


def cp_call(lib, segments=2, **kw):
    a = dict(q=P[0], k=P[1], v=P[2], la=P[3], beta=P[4], S0=None, cu=None, B=1, T=64, H=2,
             dk=64, dv=64, N=1, dt=0, o=P[5], ST=P[6], ws=P[7], wsb=1 << 30, stream=None,
             engine=0)
    a.update(kw)
    return lib.kda_fwd_cp(a["q"], a["k"], a["v"], a["la"], a["beta"], a["S0"], a["cu"],
                          a["B"], a["T"], a["H"], a["dk"], a["dv"], a["N"], a["dt"], a["o"],
                          a["ST"], segments, a["ws"], a["wsb"], a["stream"], a["engine"])


def test_cp_workspace_bytes(kda):
    """Segment-parallel workspace: the plain one for one segment; otherwise
    task tables, a 16 KB zero tile and four [H][d][d] fp32 state sets per later
    segment of every sequence (S~, M, start state) plus one per sequence."""
    assert kda.kda_fwd_cp_workspace_bytes(3, 4, 64, 64, 1) == kda.kda_fwd_workspace_bytes(3)
    for N, H, d, P in [(1, 12, 128, 6), (5, 2, 64, 3), (16, 96, 128, 2)]:
        b = kda.kda_fwd_cp_workspace_bytes(N, H, d, d, P)
        states = (N + 3 * N * (P - 1)) * H * d * d * 4
        assert states + 16384 <= b <= states + 16384 + 64 * N * (3 * P) + 8 * 256
        assert b % 256 == 0
    assert kda.kda_fwd_cp_workspace_bytes(1, 1, 64, 128, 2) == 0      # d_k != d_v
    assert kda.kda_fwd_cp_workspace_bytes(1, 1, 64, 64, 0) == 0


def test_cp_argument_errors(kda):
    lib = kda.load()
    E_INV, E_UNS, E_WS = 1, 2, 3
    assert cp_call(lib, segments=0) == E_INV
    assert cp_call(lib, segments=70000) == E_INV
    assert cp_call(lib, q=None) == E_INV
    assert cp_call(lib, dk=96, dv=96) == E_UNS
    assert cp_call(lib, engine=1, dt=0, dk=128, dv=128) == E_UNS      # fp32 at d = 128: CUDA cores
    assert cp_call(lib, ws=None) == E_WS
    need = kda.kda_fwd_cp_workspace_bytes(1, 2, 64, 64, 4)
    assert cp_call(lib, segments=4, wsb=need - 1) == E_WS
    assert cp_call(lib, N=2) == E_INV                                 # N != B without cu_seqlens


def test_cp_segments_without_gpu(kda):
    """With no device to size against, the suggestion is a plain pass."""
    assert kda.kda_fwd_cp_segments(1, 12, 131072) >= 1
    assert kda.kda_fwd_cp_segments(0, 12, 131072) == 1
    assert kda.kda_fwd_cp_segments(1, 12, 0) == 1


def test_decode_argument_errors(kda):
    lib = kda.load()

    def call(**kw):
        a = dict(q=P[0], k=P[1], v=P[2], la=P[3], beta=P[4], S=P[5], N=4, H=2, dk=128, dv=128,
                 dt=1, o=P[6], stream=None)
        a.update(kw)
        return lib.kda_decode_step(a["q"], a["k"], a["v"], a["la"], a["beta"], a["S"], a["N"],
                                   a["H"], a["dk"], a["dv"], a["dt"], a["o"], a["stream"])
    assert call(S=None) == 1
    assert call(o=ctypes.c_void_p(0x10001)) == 1                     # odd bf16 address
    assert call(S=ctypes.c_void_p(0x10008)) == 1                     # state needs 16 B
    assert call(dk=32, dv=32) == 2
    assert call(N=-1) == 1
    assert call(N=0, S=None) == 0  # nothing to do


def test_draft_token_argument_errors(kda):
    """kda_verify_tokens / kda_commit_tokens reject bad arguments before any
    launch (fake device addresses are never dereferenced)."""
    lib = kda.load()

    def verify(**kw):
        a = dict(q=P[0], k=P[1], v=P[2], la=P[3], beta=P[4], S=P[5], N=4, K=3, H=2, dk=128,
                 dv=128, dt=1, o=P[6], stream=None)
        a.update(kw)
        return lib.kda_verify_tokens(a["q"], a["k"], a["v"], a["la"], a["beta"], a["S"], a["N"],
                                     a["K"], a["H"], a["dk"], a["dv"], a["dt"], a["o"],
                                     a["stream"])

    def commit(**kw):
        a = dict(q=P[0], k=P[1], v=P[2], la=P[3], beta=P[4], S=P[5], acc=None, N=4, K=3, H=2,
                 dk=128, dv=128, dt=1, stream=None)
        a.update(kw)
        return lib.kda_commit_tokens(a["q"], a["k"], a["v"], a["la"], a["beta"], a["S"],
                                     a["acc"], a["N"], a["K"], a["H"], a["dk"], a["dv"], a["dt"],
                                     a["stream"])
    assert verify(K=0) == 1 and verify(K=kda.KDA_MAX_DRAFT_TOKENS + 1) == 1
    assert verify(o=None) == 1 and verify(S=ctypes.c_void_p(0x10008)) == 1
    assert verify(dk=32, dv=32) == 2 and verify(dt=5) == 1
    assert verify(N=0, S=None, o=None) == 0                        # nothing to do
    assert commit(acc=ctypes.c_void_p(0x10002)) == 1               # n_accept needs 4 B
    assert commit(q=None) == 1 and commit(N=-1) == 1
    assert commit(N=0, S=None) == 0


def test_short_conv_argument_errors(kda):
    """The prologue entry points validate sizes, pointers, alignment, eps and
    the workspace on the host, before any launch."""
    lib = kda.load()
    E_INV, E_UNS, E_WS = 1, 2, 3

    def conv(**kw):
        a = dict(x=P[0], w=P[1], c0=None, cu=None, B=1, T=64, H=2, d=64, N=1, dt=0, eps=1e-6,
                 y=P[2], cT=P[3], ws=P[4], wsb=4096)
        a.update(kw)
        return lib.kda_short_conv(a["x"], a["x"], a["x"], a["w"], a["w"], a["w"], a["c0"],
                                  a["cu"], a["B"], a["T"], a["H"], a["d"], a["N"], a["dt"],
                                  a["eps"], a["y"], a["y"], a["y"], a["cT"], a["ws"], a["wsb"],
                                  None)

    assert conv(dt=5) == E_INV
    assert conv(d=96) == E_UNS
    assert conv(H=0) == E_INV
    assert conv(N=2) == E_INV                                  # N != B without cu_seqlens
    assert conv(cu=P[8], B=2, N=2) == E_INV                    # varlen needs B = 1
    assert conv(eps=-1.0) == E_INV
    assert conv(eps=float("nan")) == E_INV
    assert conv(x=None) == E_INV
    assert conv(x=ctypes.c_void_p(0x10008)) == E_INV           # misaligned
    assert conv(w=None) == E_INV
    assert conv(c0=ctypes.c_void_p(0x10004)) == E_INV
    assert conv(ws=None) == E_WS
    assert conv(wsb=8) == E_WS

    def step(**kw):
        a = dict(x=P[0], w=P[1], c=P[2], N=4, H=2, d=128, dt=1, eps=0.0, y=P[3])
        a.update(kw)
        return lib.kda_short_conv_step(a["x"], a["x"], a["x"], a["w"], a["w"], a["w"], a["c"],
                                       a["N"], a["H"], a["d"], a["dt"], a["eps"], a["y"],
                                       a["y"], a["y"], None)

    assert step(d=32) == E_UNS
    assert step(N=-1) == E_INV
    assert step(c=None) == E_INV
    assert step(y=ctypes.c_void_p(0x10002)) == E_INV
    assert step(N=0) == 0                                      # nothing to do


def test_decode_layer_step_argument_errors(kda):
    """kda_decode_layer_step validates sizes, eps, pointers and alignment on the
    host, before any launch."""
    lib = kda.load()
    E_INV, E_UNS = 1, 2

    def call(**kw):
        a = dict(x=P[0], w=P[1], conv=P[2], l2=1e-6, la=P[3], b=P[4], S=P[5], N=2, H=2, d=128,
                 dt=1, g=P[6], nw=None, eps=1e-6, y=P[7])
        a.update(kw)
        return lib.kda_decode_layer_step(a["x"], a["x"], a["x"], a["w"], a["w"], a["w"],
                                         a["conv"], a["l2"], a["la"], a["b"], a["S"], a["N"],
                                         a["H"], a["d"], a["dt"], a["g"], a["nw"], a["eps"],
                                         a["y"], None)

    assert call(d=32) == E_UNS
    assert call(dt=3) == E_INV
    assert call(N=-1) == E_INV
    assert call(H=0) == E_INV
    assert call(l2=-1.0) == E_INV
    assert call(eps=float("inf")) == E_INV
    assert call(conv=None) == E_INV
    assert call(g=None) == E_INV
    assert call(S=ctypes.c_void_p(0x10008)) == E_INV          # misaligned
    assert call(b=ctypes.c_void_p(0x10002)) == E_INV          # beta: 4-byte aligned
    assert call(N=0) == 0                                      # nothing to do


def test_failure_injection_reports_cuda_error(kda, monkeypatch):
    """The host-only injection hook turns a valid call into KDA_ERR_CUDA
    without enqueueing anything."""
    lib = kda.load()
    monkeypatch.setenv("KDA_FAULT_INJECT", "launch")
    assert fwd_call(lib) == 4
    assert lib.kda_decode_step(P[0], P[1], P[2], P[3], P[4], P[5], 1, 1, 64, 64, 0, P[6],
                               None) == 4


def test_binding_rejects_cpu_tensors(kda):
    import torch
    x = torch.zeros(1, 64, 2, 64)
    with pytest.raises(ValueError):
        kda.kda_fwd(x, x, x, x, torch.zeros(1, 64, 2))


def test_bounds_checked_build_exports_every_symbol():
    """The bounds-checked variant compiles (nvcc cross-compiles without a GPU)
    and exports the same entry points."""
    import ctypes
    from linear_attention_recurrence_chunkwise_gb300 import build as kbuild
    from linear_attention_recurrence_chunkwise_gb300 import kda as mod
    lib = ctypes.CDLL(kbuild.build(bounds_check=True))
    for name in mod.EXPORTED:
        assert hasattr(lib, name), name
