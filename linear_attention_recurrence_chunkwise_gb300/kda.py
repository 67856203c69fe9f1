"""Thin Python binding of libkda: argument marshalling only.

Every function here has the name of the C entry point it wraps and only turns
torch tensors into device pointers (plus the current CUDA stream).  All of the
operator's work runs in libkda's CUDA kernels; there is no other code path, and
if the library is missing the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_OK = 0
KDA_ERR_INVALID_ARGUMENT = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_WORKSPACE = 3
KDA_ERR_CUDA = 4
KDA_ERR_DOMAIN = 5
KDA_ERR_TIMEOUT = 6
KDA_ERR_BOUNDS = 7

KDA_F32, KDA_BF16 = 0, 1
ENGINES = {"auto": 0, "tensorcore": 1, "cudacore": 2, "tensorcore_wide": 3}
EPILOGUES = {"auto": 0, "fused": 1, "separate": 2}

# every symbol include/kda.h declares
EXPORTED = ["kda_fwd_workspace_bytes", "kda_fwd", "kda_fwd_engine", "kda_fwd_noalloc",
            "kda_fwd_cp", "kda_fwd_cp_workspace_bytes", "kda_fwd_cp_segments",
            "kda_decode_step", "kda_verify_tokens", "kda_commit_tokens",
            "kda_fwd_gated", "kda_decode_step_gated", "kda_gated_rmsnorm",
            "kda_short_conv", "kda_short_conv_step", "kda_decode_layer_step",
            "kda_read_device_status", "kda_state_bytes", "kda_status_string"]
KDA_NOALLOC_MAX_SEQS = 16384
KDA_MAX_DRAFT_TOKENS = 16

_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {kda_status_string(status)} ({status})")


def load() -> ctypes.CDLL:
    """Load libkda.so (built by ``build.build()``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkda.so not built at {LIB_PATH}; run "
                               "linear_attention_recurrence_chunkwise_gb300.build.build()")
        _lib = load_library(LIB_PATH)
        return _lib


def load_library(path: str) -> ctypes.CDLL:
    """Open a build of libkda at `path` (for instance the bounds-checked
    libkda_bounds.so) with the entry points' signatures; pass it as `lib=` to
    the functions below."""
    lib = ctypes.CDLL(path)
    vp, sz, ci, fp = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p
    lib.kda_fwd_workspace_bytes.restype = sz
    lib.kda_fwd_workspace_bytes.argtypes = [ci]
    fwd_args = [vp, vp, vp, fp, fp, fp, vp, ci, ci, ci, ci, ci, ci, ci, vp, fp, vp, sz, vp]
    lib.kda_fwd.restype = ci
    lib.kda_fwd.argtypes = fwd_args
    lib.kda_fwd_engine.restype = ci
    lib.kda_fwd_engine.argtypes = fwd_args + [ci]
    lib.kda_fwd_cp.restype = ci
    lib.kda_fwd_cp.argtypes = fwd_args[:16] + [ci, vp, sz, vp, ci]
    lib.kda_fwd_cp_workspace_bytes.restype = sz
    lib.kda_fwd_cp_workspace_bytes.argtypes = [ci] * 5
    lib.kda_fwd_cp_segments.restype = ci
    lib.kda_fwd_cp_segments.argtypes = [ci, ci, ctypes.c_int64]
    lib.kda_fwd_noalloc.restype = ci
    lib.kda_fwd_noalloc.argtypes = fwd_args[:16] + [vp, vp]
    lib.kda_decode_step.restype = ci
    lib.kda_decode_step.argtypes = [vp, vp, vp, fp, fp, fp, ci, ci, ci, ci, ci, vp, vp]
    lib.kda_verify_tokens.restype = ci
    lib.kda_verify_tokens.argtypes = [vp, vp, vp, fp, fp, fp, ci, ci, ci, ci, ci, ci, vp, vp]
    lib.kda_commit_tokens.restype = ci
    lib.kda_commit_tokens.argtypes = [vp, vp, vp, fp, fp, fp, vp, ci, ci, ci, ci, ci, ci, vp]
    cf = ctypes.c_float
    lib.kda_fwd_gated.restype = ci
    lib.kda_fwd_gated.argtypes = fwd_args[:14] + [vp, fp, cf] + fwd_args[14:] + [ci, ci]
    lib.kda_decode_step_gated.restype = ci
    lib.kda_decode_step_gated.argtypes = [vp, vp, vp, fp, fp, fp, ci, ci, ci, ci, ci, vp, fp, cf,
                                          vp, vp, ci]
    lib.kda_gated_rmsnorm.restype = ci
    lib.kda_gated_rmsnorm.argtypes = [vp, vp, fp, cf, ctypes.c_int64, ci, ci, vp, vp]
    lib.kda_short_conv.restype = ci
    lib.kda_short_conv.argtypes = [vp, vp, vp, fp, fp, fp, fp, vp, ci, ci, ci, ci, ci, ci, cf,
                                   vp, vp, vp, fp, vp, sz, vp]
    lib.kda_short_conv_step.restype = ci
    lib.kda_short_conv_step.argtypes = [vp, vp, vp, fp, fp, fp, fp, ci, ci, ci, ci, cf, vp, vp,
                                        vp, vp]
    lib.kda_decode_layer_step.restype = ci
    lib.kda_decode_layer_step.argtypes = [vp, vp, vp, fp, fp, fp, fp, cf, fp, fp, fp, ci, ci, ci,
                                          ci, vp, fp, cf, vp, vp]
    lib.kda_read_device_status.restype = ci
    lib.kda_read_device_status.argtypes = [vp, sz, vp]
    lib.kda_state_bytes.restype = sz
    lib.kda_state_bytes.argtypes = [ci] * 6
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_status_string.argtypes = [ci]
    return lib


def kda_status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def kda_state_bytes(layers: int, N: int, H: int, d_k: int, d_v: int, elem_bytes: int) -> int:
    return int(load().kda_state_bytes(layers, N, H, d_k, d_v, elem_bytes))


def kda_fwd_workspace_bytes(N: int) -> int:
    return int(load().kda_fwd_workspace_bytes(N))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(dt) -> int:
    if dt == torch.bfloat16:
        return KDA_BF16
    if dt == torch.float32:
        return KDA_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {dt}")


def _check(t, name, dtype=None, device=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _check_shape(t, name, shape):
    """The library sees only pointers: a tensor of another shape would be read
    or written out of its bounds, so the shape is checked here."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be {list(shape)}, got {list(t.shape)}")


def _fwd_args(q, k, v, log_alpha, beta, S0, cu_seqlens, o, S_T, return_state):
    """Checks and sizes shared by the forward entry points: (B, T, H, d_k, d_v,
    N, o, S_T), with o and S_T allocated with torch when not given."""
    dev = q.device
    dt = q.dtype
    _check(q, "q", dt), _check(k, "k", dt, dev), _check(v, "v", dt, dev)
    _check(log_alpha, "log_alpha", torch.float32, dev)
    _check(beta, "beta", torch.float32, dev)
    _check(S0, "S0", torch.float32, dev)
    _check(cu_seqlens, "cu_seqlens", torch.int32, dev)
    H, d_k = q.shape[-2], q.shape[-1]
    d_v = v.shape[-1]
    if cu_seqlens is not None:
        if q.dim() != 3:
            raise ValueError("with cu_seqlens, q must be packed [Ttot, H, d_k]")
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
            raise ValueError("cu_seqlens must be [N + 1] with N >= 0")
        B, T = 1, q.shape[0]
        N = cu_seqlens.numel() - 1
    else:
        if q.dim() == 4:
            B, T = q.shape[0], q.shape[1]
        elif q.dim() == 3:
            B, T = 1, q.shape[0]
        else:
            raise ValueError("q must be [B, T, H, d_k] or [Ttot, H, d_k]")
        N = B
    if k.shape != q.shape or log_alpha.shape != q.shape or v.shape[:-1] != q.shape[:-1] \
            or beta.shape != q.shape[:-1]:
        raise ValueError("q, k, v, log_alpha, beta shapes disagree")
    _check_shape(S0, "S0", (N, H, d_v, d_k))
    if o is None:
        o = torch.empty(v.shape, dtype=dt, device=dev)
    _check(o, "o", dt, dev)
    _check_shape(o, "o", v.shape)
    if S_T is None and return_state:
        S_T = torch.empty((N, H, d_v, d_k), dtype=torch.float32, device=dev)
    _check(S_T, "S_T", torch.float32, dev)
    _check_shape(S_T, "S_T", (N, H, d_v, d_k))
    return B, T, H, d_k, d_v, N, o, S_T


def kda_fwd(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, *, o=None, S_T=None,
            workspace=None, return_state: bool = True, engine: str = "auto", stream=None,
            lib=None):
    """Chunkwise KDA forward (prefill).

    q, k, log_alpha [B, T, H, d_k] or packed [Ttot, H, d_k]; v [.., H, d_v];
    beta [.., H]; S0 [N, H, d_v, d_k] fp32 or None; cu_seqlens int32 [N+1]
    (device) or None.  Returns (o, S_T) (S_T None when return_state is False).
    Output tensors and the workspace are allocated with torch unless given.
    `lib` selects another build of the library (see load_library).
    """
    B, T, H, d_k, d_v, N, o, S_T = _fwd_args(q, k, v, log_alpha, beta, S0, cu_seqlens, o,
                                             S_T, return_state)
    lib = lib or load()
    if workspace is None:
        workspace = torch.empty(int(lib.kda_fwd_workspace_bytes(N)), dtype=torch.uint8,
                                device=q.device)
    _check(workspace, "workspace", None, q.device)
    rc = lib.kda_fwd_engine(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                            _ptr(S0), _ptr(cu_seqlens), B, T, H, d_k, d_v, N,
                            _dtype_code(q.dtype), _ptr(o), _ptr(S_T), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream),
                            ENGINES[engine])
    if rc != KDA_OK:
        raise KdaError(rc, "kda_fwd")
    return o, S_T


def _check_gate(g, norm_weight, like, dev):
    """The gate logits share o's shape and dtype; the norm weight is fp32 [d_v]."""
    _check(g, "g", like.dtype, dev)
    _check_shape(g, "g", like.shape)
    if norm_weight is not None:
        _check(norm_weight, "norm_weight", torch.float32, dev)
        _check_shape(norm_weight, "norm_weight", (like.shape[-1],))


def kda_fwd_gated(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, *, g, norm_weight=None,
                  eps: float = 1e-6, y=None, S_T=None, workspace=None,
                  return_state: bool = True, engine: str = "auto", epilogue: str = "auto",
                  stream=None, lib=None):
    """kda_fwd followed by the layer's output epilogue, y = sigmoid(g) * w * o /
    sqrt(mean(o^2) + eps) per (token, head).  g: gate logits shaped like v;
    norm_weight: fp32 [d_v] or None; epilogue: 'auto', 'fused' (in the
    tensor-core kernel's output stores) or 'separate' (a second pass).
    Returns (y, S_T)."""
    B, T, H, d_k, d_v, N, y, S_T = _fwd_args(q, k, v, log_alpha, beta, S0, cu_seqlens, y,
                                             S_T, return_state)
    _check_gate(g, norm_weight, y, q.device)
    lib = lib or load()
    if workspace is None:
        workspace = torch.empty(int(lib.kda_fwd_workspace_bytes(N)), dtype=torch.uint8,
                                device=q.device)
    _check(workspace, "workspace", None, q.device)
    rc = lib.kda_fwd_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0),
                           _ptr(cu_seqlens), B, T, H, d_k, d_v, N, _dtype_code(q.dtype),
                           _ptr(g), _ptr(norm_weight), float(eps), _ptr(y), _ptr(S_T),
                           _ptr(workspace), workspace.numel() * workspace.element_size(),
                           _stream(stream), ENGINES[engine], EPILOGUES[epilogue])
    if rc != KDA_OK:
        raise KdaError(rc, "kda_fwd_gated")
    return y, S_T


def kda_gated_rmsnorm(o, g, norm_weight=None, eps: float = 1e-6, *, y=None, stream=None):
    """The output epilogue alone over the last axis: y = sigmoid(g) * w * o /
    sqrt(mean(o^2) + eps).  y may be o itself (in place).  Returns y."""
    _check(o, "o", o.dtype, o.device)
    _check_gate(g, norm_weight, o, o.device)
    if y is None:
        y = torch.empty_like(o)
    _check(y, "y", o.dtype, o.device)
    _check_shape(y, "y", o.shape)
    d_v = o.shape[-1]
    rows = o.numel() // d_v if d_v else 0
    rc = load().kda_gated_rmsnorm(_ptr(o), _ptr(g), _ptr(norm_weight), float(eps), rows, d_v,
                                  _dtype_code(o.dtype), _ptr(y), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_gated_rmsnorm")
    return y


def _prologue_checks(xq, xk, xv, wq, wk, wv):
    dev, dt = xq.device, xq.dtype
    _dtype_code(dt)
    for t, name in ((xq, "xq"), (xk, "xk"), (xv, "xv")):
        _check(t, name, dt, dev)
        _check_shape(t, name, xq.shape)
    H, d = xq.shape[-2], xq.shape[-1]
    for t, name in ((wq, "wq"), (wk, "wk"), (wv, "wv")):
        _check(t, name, torch.float32, dev)
        _check_shape(t, name, (H, d, 4))
    return dev, dt, H, d


def kda_short_conv(xq, xk, xv, wq, wk, wv, conv0=None, cu_seqlens=None, *, eps: float = 1e-6,
                   q=None, k=None, v=None, conv_T=None, return_state: bool = True,
                   workspace=None, stream=None, lib=None):
    """The layer's input prologue over whole sequences: q, k =
    L2Norm(Swish(ShortConv(xq / xk))), v = Swish(ShortConv(xv)).  x: [B, T, H, d]
    or packed [Ttot, H, d] with cu_seqlens; w: [H, d, 4] fp32 taps (w[..., 3] on
    the current token); conv0 / conv_T: [N, 3, 3, H, d] fp32 conv states (conv_T
    may be conv0).  Returns (q, k, v, conv_T)."""
    dev, dt, H, d = _prologue_checks(xq, xk, xv, wq, wk, wv)
    _check(conv0, "conv0", torch.float32, dev)
    _check(cu_seqlens, "cu_seqlens", torch.int32, dev)
    if cu_seqlens is not None:
        if xq.dim() != 3 or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
            raise ValueError("with cu_seqlens, x must be packed [Ttot, H, d] and cu_seqlens [N + 1]")
        B, T, N = 1, xq.shape[0], cu_seqlens.numel() - 1
    elif xq.dim() == 4:
        B, T = xq.shape[0], xq.shape[1]
        N = B
    elif xq.dim() == 3:
        B, T, N = 1, xq.shape[0], 1
    else:
        raise ValueError("x must be [B, T, H, d] or [Ttot, H, d]")
    _check_shape(conv0, "conv0", (N, 3, 3, H, d))
    outs = []
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        if t is None:
            t = torch.empty(xq.shape, dtype=dt, device=dev)
        _check(t, name, dt, dev)
        _check_shape(t, name, xq.shape)
        outs.append(t)
    if conv_T is None and return_state:
        conv_T = torch.empty((N, 3, 3, H, d), dtype=torch.float32, device=dev)
    _check(conv_T, "conv_T", torch.float32, dev)
    _check_shape(conv_T, "conv_T", (N, 3, 3, H, d))
    lib = lib or load()
    if workspace is None:
        workspace = torch.empty(int(lib.kda_fwd_workspace_bytes(N)), dtype=torch.uint8, device=dev)
    rc = lib.kda_short_conv(_ptr(xq), _ptr(xk), _ptr(xv), _ptr(wq), _ptr(wk), _ptr(wv),
                            _ptr(conv0), _ptr(cu_seqlens), B, T, H, d, N, _dtype_code(dt),
                            float(eps), _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]),
                            _ptr(conv_T), _ptr(workspace), workspace.numel(), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_short_conv")
    return outs[0], outs[1], outs[2], conv_T


def kda_short_conv_step(xq, xk, xv, wq, wk, wv, conv, *, eps: float = 1e-6, q=None, k=None,
                        v=None, stream=None, lib=None):
    """The prologue for one token per session: x [N, H, d]; conv [N, 3, 3, H, d]
    fp32 is moved on by one token in place.  Returns (q, k, v)."""
    dev, dt, H, d = _prologue_checks(xq, xk, xv, wq, wk, wv)
    if xq.dim() != 3:
        raise ValueError("x must be [N, H, d]")
    N = xq.shape[0]
    _check(conv, "conv", torch.float32, dev)
    _check_shape(conv, "conv", (N, 3, 3, H, d))
    outs = []
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        if t is None:
            t = torch.empty(xq.shape, dtype=dt, device=dev)
        _check(t, name, dt, dev)
        _check_shape(t, name, xq.shape)
        outs.append(t)
    rc = (lib or load()).kda_short_conv_step(_ptr(xq), _ptr(xk), _ptr(xv), _ptr(wq), _ptr(wk),
                                             _ptr(wv), _ptr(conv), N, H, d, _dtype_code(dt),
                                             float(eps), _ptr(outs[0]), _ptr(outs[1]),
                                             _ptr(outs[2]), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_short_conv_step")
    return outs[0], outs[1], outs[2]


def kda_decode_layer_step(xq, xk, xv, wq, wk, wv, conv, log_alpha, beta, S, g,
                          norm_weight=None, eps: float = 1e-6, l2_eps: float = 1e-6, *, y=None,
                          stream=None, lib=None):
    """One decode token per session through the layer step in one kernel:
    prologue (conv state moved on in place), recurrence (S in place) and output
    epilogue.  x, g: [N, H, d]; conv [N, 3, 3, H, d]; S [N, H, d, d].  Returns y."""
    dev, dt, H, d = _prologue_checks(xq, xk, xv, wq, wk, wv)
    if xq.dim() != 3:
        raise ValueError("x must be [N, H, d]")
    N = xq.shape[0]
    _check(conv, "conv", torch.float32, dev)
    _check_shape(conv, "conv", (N, 3, 3, H, d))
    _check(log_alpha, "log_alpha", torch.float32, dev)
    _check_shape(log_alpha, "log_alpha", (N, H, d))
    _check(beta, "beta", torch.float32, dev)
    _check_shape(beta, "beta", (N, H))
    _check(S, "S", torch.float32, dev)
    _check_shape(S, "S", (N, H, d, d))
    _check(g, "g", dt, dev)
    _check_shape(g, "g", (N, H, d))
    _check(norm_weight, "norm_weight", torch.float32, dev)
    _check_shape(norm_weight, "norm_weight", (d,))
    if y is None:
        y = torch.empty((N, H, d), dtype=dt, device=dev)
    _check(y, "y", dt, dev)
    _check_shape(y, "y", (N, H, d))
    rc = (lib or load()).kda_decode_layer_step(
        _ptr(xq), _ptr(xk), _ptr(xv), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(conv), float(l2_eps),
        _ptr(log_alpha), _ptr(beta), _ptr(S), N, H, d, _dtype_code(dt), _ptr(g),
        _ptr(norm_weight), float(eps), _ptr(y), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_layer_step")
    return y


def kda_fwd_cp_workspace_bytes(N: int, H: int, d_k: int, d_v: int, segments: int) -> int:
    return int(load().kda_fwd_cp_workspace_bytes(N, H, d_k, d_v, segments))


def kda_fwd_cp_segments(N: int, H: int, Ttot: int) -> int:
    return int(load().kda_fwd_cp_segments(N, H, Ttot))


def kda_fwd_cp(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, *, segments=None, o=None,
               S_T=None, workspace=None, return_state: bool = True, engine: str = "auto",
               stream=None, lib=None):
    """Segment-parallel KDA forward on one GPU (same arguments and results as
    kda_fwd).  `segments` defaults to kda_fwd_cp_segments' choice."""
    B, T, H, d_k, d_v, N, o, S_T = _fwd_args(q, k, v, log_alpha, beta, S0, cu_seqlens, o,
                                             S_T, return_state)
    lib = lib or load()
    if segments is None:
        segments = int(lib.kda_fwd_cp_segments(N, H, B * T))
    if workspace is None:
        need = int(lib.kda_fwd_cp_workspace_bytes(N, H, d_k, d_v, segments))
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace", None, q.device)
    rc = lib.kda_fwd_cp(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0),
                        _ptr(cu_seqlens), B, T, H, d_k, d_v, N, _dtype_code(q.dtype), _ptr(o),
                        _ptr(S_T), int(segments), _ptr(workspace),
                        workspace.numel() * workspace.element_size(), _stream(stream),
                        ENGINES[engine])
    if rc != KDA_OK:
        raise KdaError(rc, "kda_fwd_cp")
    return o, S_T


def kda_fwd_noalloc(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, *, o=None,
                    S_T=None, device_status=None, stream=None):
    """kda_fwd for callers that cannot allocate device memory.

    The library keeps the scratch kda_fwd would take as a workspace in a fixed
    array of its own; only inputs and outputs are passed (o and S_T are
    allocated with torch here when not given, which callers that cannot
    allocate avoid by passing them).  `device_status` is an optional device
    int32 tensor that receives the call's status word.  Returns (o, S_T).
    """
    dt = q.dtype
    _check(device_status, "device_status", torch.int32, q.device)
    if device_status is not None and device_status.numel() < 1:
        raise ValueError("device_status must hold at least one int32")
    B, T, H, d_k, d_v, N, o, S_T = _fwd_args(q, k, v, log_alpha, beta, S0, cu_seqlens, o,
                                             S_T, True)
    rc = load().kda_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                _ptr(S0), _ptr(cu_seqlens), B, T, H, d_k, d_v, N,
                                _dtype_code(dt), _ptr(o), _ptr(S_T), _ptr(device_status),
                                _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_fwd_noalloc")
    return o, S_T


def kda_decode_step(q, k, v, log_alpha, beta, S, *, o=None, stream=None):
    """One decode token per session; S [N, H, d_v, d_k] fp32 is updated in place.

    q, k, log_alpha [N, H, d_k]; v [N, H, d_v]; beta [N, H].  Returns o [N, H, d_v].
    """
    dev = q.device
    dt = q.dtype
    _check(q, "q", dt), _check(k, "k", dt, dev), _check(v, "v", dt, dev)
    _check(log_alpha, "log_alpha", torch.float32, dev)
    _check(beta, "beta", torch.float32, dev)
    _check(S, "S", torch.float32, dev)
    if q.dim() != 3:
        raise ValueError("decode inputs are [N, H, d]")
    N, H, d_k = q.shape
    d_v = v.shape[-1]
    if k.shape != q.shape or log_alpha.shape != q.shape or v.shape[:-1] != q.shape[:-1] \
            or beta.shape != q.shape[:-1]:
        raise ValueError("q, k, v, log_alpha, beta shapes disagree")
    if S.shape != (N, H, d_v, d_k):
        raise ValueError(f"S must be [N, H, d_v, d_k] = {(N, H, d_v, d_k)}")
    if o is None:
        o = torch.empty((N, H, d_v), dtype=dt, device=dev)
    _check(o, "o", dt, dev)
    _check_shape(o, "o", (N, H, d_v))
    rc = load().kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                _ptr(S), N, H, d_k, d_v, _dtype_code(dt), _ptr(o),
                                _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_step")
    return o


def kda_decode_step_gated(q, k, v, log_alpha, beta, S, *, g, norm_weight=None,
                          eps: float = 1e-6, y=None, epilogue: str = "auto", stream=None):
    """kda_decode_step with the output epilogue: returns y [N, H, d_v] =
    sigmoid(g) * w * o / sqrt(mean(o^2) + eps); S is updated in place.
    epilogue: 'auto', 'fused' or 'separate'."""
    dev, dt = q.device, q.dtype
    _check(q, "q", dt), _check(k, "k", dt, dev), _check(v, "v", dt, dev)
    _check(log_alpha, "log_alpha", torch.float32, dev)
    _check(beta, "beta", torch.float32, dev)
    _check(S, "S", torch.float32, dev)
    if q.dim() != 3:
        raise ValueError("decode inputs are [N, H, d]")
    N, H, d_k = q.shape
    d_v = v.shape[-1]
    if k.shape != q.shape or log_alpha.shape != q.shape or v.shape[:-1] != q.shape[:-1] \
            or beta.shape != q.shape[:-1]:
        raise ValueError("q, k, v, log_alpha, beta shapes disagree")
    if S.shape != (N, H, d_v, d_k):
        raise ValueError(f"S must be [N, H, d_v, d_k] = {(N, H, d_v, d_k)}")
    if y is None:
        y = torch.empty((N, H, d_v), dtype=dt, device=dev)
    _check(y, "y", dt, dev)
    _check_shape(y, "y", (N, H, d_v))
    _check_gate(g, norm_weight, y, dev)
    rc = load().kda_decode_step_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                      _ptr(S), N, H, d_k, d_v, _dtype_code(dt), _ptr(g),
                                      _ptr(norm_weight), float(eps), _ptr(y), _stream(stream),
                                      EPILOGUES[epilogue])
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_step_gated")
    return y


def _check_draft(q, k, v, log_alpha, beta, S):
    dev, dt = q.device, q.dtype
    _check(q, "q", dt), _check(k, "k", dt, dev), _check(v, "v", dt, dev)
    _check(log_alpha, "log_alpha", torch.float32, dev)
    _check(beta, "beta", torch.float32, dev)
    _check(S, "S", torch.float32, dev)
    if q.dim() != 4:
        raise ValueError("draft tokens are [N, K, H, d]")
    N, K, H, d_k = q.shape
    d_v = v.shape[-1]
    if k.shape != q.shape or log_alpha.shape != q.shape or v.shape[:-1] != q.shape[:-1] \
            or beta.shape != q.shape[:-1]:
        raise ValueError("q, k, v, log_alpha, beta shapes disagree")
    if S.shape != (N, H, d_v, d_k):
        raise ValueError(f"S must be [N, H, d_v, d_k] = {(N, H, d_v, d_k)}")
    return N, K, H, d_k, d_v


def kda_verify_tokens(q, k, v, log_alpha, beta, S, *, o=None, stream=None):
    """Outputs of K draft tokens per session run in order from the committed
    state S, which is left unchanged.  q, k, log_alpha [N, K, H, d_k]; v
    [N, K, H, d_v]; beta [N, K, H].  Returns o [N, K, H, d_v]."""
    N, K, H, d_k, d_v = _check_draft(q, k, v, log_alpha, beta, S)
    if o is None:
        o = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    _check(o, "o", q.dtype, q.device)
    _check_shape(o, "o", v.shape)
    rc = load().kda_verify_tokens(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                  _ptr(S), N, K, H, d_k, d_v, _dtype_code(q.dtype), _ptr(o),
                                  _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_verify_tokens")
    return o


def kda_commit_tokens(q, k, v, log_alpha, beta, S, n_accept=None, *, stream=None):
    """Apply the first n_accept[n] of session n's K draft tokens to S in place
    (n_accept: device int32 [N], clamped to [0, K]; None applies all K)."""
    N, K, H, d_k, d_v = _check_draft(q, k, v, log_alpha, beta, S)
    _check(n_accept, "n_accept", torch.int32, q.device)
    if n_accept is not None and n_accept.shape != (N,):
        raise ValueError("n_accept must be [N]")
    rc = load().kda_commit_tokens(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                  _ptr(S), _ptr(n_accept), N, K, H, d_k, d_v,
                                  _dtype_code(q.dtype), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_commit_tokens")
    return S


def kda_read_device_status(workspace, stream=None, lib=None) -> int:
    """Synchronise the stream and return the status word left by kda_fwd."""
    rc = (lib or load()).kda_read_device_status(_ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream))
    return int(rc)
