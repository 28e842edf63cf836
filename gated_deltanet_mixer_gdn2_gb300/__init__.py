"""Gated DeltaNet-2 token-mixer core for GB300 (sm_103a): thin Python binding of libgdn2.so.

Every step of the computation runs in the library's CUDA kernels; this module only marshals
arguments (device pointers, sizes, the current CUDA stream) from torch tensors to the C ABI declared
in include/gdn2.h, and raises on a non-zero status. torch provides device memory and streams only.

The binding fails loudly: importing it raises if libgdn2.so has not been built.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgdn2.so")

GDN2_OK, GDN2_ERR_INVALID_ARG, GDN2_ERR_UNSUPPORTED = 0, -1, -2
GDN2_ERR_MISALIGNED, GDN2_ERR_WORKSPACE, GDN2_ERR_CUDA, GDN2_ERR_TIMEOUT = -3, -4, -5, -6
GDN2_F32, GDN2_BF16 = 0, 1
PATHS = {"auto": 0, "simt": 1, "tcgen05": 2}

#: names of the extern "C" functions exported by libgdn2.so (all declared in include/gdn2.h)
EXPORTS = (
    "gdn2_status_string", "gdn2_version", "gdn2_chunk_fwd_workspace_size",
    "gdn2_chunk_fwd_workspace_size_path", "gdn2_chunk_fwd", "gdn2_chunk_fwd_path",
    "gdn2_recurrent_step", "gdn2_last_device_status", "gdn2_set_wait_limit", "gdn2_selftest_umma",
    "gdn2_chunk_fwd_noalloc", "gdn2_recurrent_update", "gdn2_fg2_inputs", "gdn2_mixer_prologue",
    "gdn2_mixer_epilogue", "gdn2_backward_workspace_size", "gdn2_backward",
    "gdn2_backward_recurrent_workspace_size", "gdn2_backward_recurrent", "gdn2_mixer_decode_step",
)


class Gdn2Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()' "
            "or python gated_deltanet_mixer_gdn2_gb300/_build.py)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, Z, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_longlong
    sig = {
        "gdn2_status_string": (ctypes.c_char_p, [I]),
        "gdn2_version": (I, []),
        "gdn2_chunk_fwd_workspace_size": (Z, [I] * 7 + [I]),
        "gdn2_chunk_fwd_workspace_size_path": (Z, [I] + [I] * 7 + [I]),
        "gdn2_chunk_fwd": (I, [P] * 9 + [I] * 7 + [F, I, P, Z, P]),
        "gdn2_chunk_fwd_path": (I, [I] + [P] * 9 + [I] * 7 + [F, I, P, Z, P]),
        "gdn2_recurrent_step": (I, [P] * 8 + [I] * 5 + [F, I, P]),
        "gdn2_last_device_status": (I, [P]),
        "gdn2_set_wait_limit": (None, [L]),
        "gdn2_selftest_umma": (I, [I, I, P, P, P, P]),
        "gdn2_chunk_fwd_noalloc": (I, [P] * 9 + [I] * 7 + [F, I, P]),
        "gdn2_recurrent_update": (I, [P] * 7 + [I, P, I, P] + [I] * 6 + [F, I, P]),
        "gdn2_fg2_inputs": (I, [P] * 7 + [I] * 5 + [I, P]),
        "gdn2_mixer_prologue": (I, [P] * 18 + [I] * 7 + [I, P]),
        "gdn2_mixer_epilogue": (I, [P, P, P, F, P] + [I] * 4 + [I, P]),
        "gdn2_backward_workspace_size": (Z, [I] * 6 + [I]),
        "gdn2_backward": (I, [P] * 16 + [I] * 6 + [F, I, P, Z, P]),
        "gdn2_backward_recurrent_workspace_size": (Z, [I] * 6 + [I]),
        "gdn2_backward_recurrent": (I, [P] * 16 + [I] * 6 + [F, I, P, Z, P]),
        "gdn2_mixer_decode_step": (I, [P] * 15 + [F, P] + [I] * 6 + [F, I, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.gdn2_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != GDN2_OK:
        raise Gdn2Error(status, what)


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return GDN2_BF16
    if t.dtype == torch.float32:
        return GDN2_F32
    raise TypeError(f"unsupported token dtype {t.dtype} (float32 or bfloat16)")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def gdn2_version() -> int:
    return lib.gdn2_version()


def gdn2_chunk_fwd_workspace_size(B, T, Hk, Hv, dk, dv, C=64, dtype=GDN2_BF16, path="auto") -> int:
    return lib.gdn2_chunk_fwd_workspace_size_path(PATHS[path], B, T, Hk, Hv, dk, dv, C, dtype)


def gdn2_chunk_fwd(q, k, v, g, b, w, o, initial_state=None, final_state=None, *, C=64, scale=1.0,
                   workspace=None, path="auto", stream=None):
    """Chunked forward (C ABI gdn2_chunk_fwd_path). Writes `o` and, if given, `final_state`.

    q, k: [B, T, H_k, d_k]; v, w: [B, T, H_v, d_v]; g, b: [B, T, H_v, d_k]; o: like v;
    states: [B, H_v, d_k, d_v] float32. `workspace`: a uint8 CUDA tensor of at least
    gdn2_chunk_fwd_workspace_size(...) bytes (allocated here when None).
    """
    import torch

    B, T, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    dt = _dtype_code(q)
    for t in (k, v, g, b, w, o):
        if t.dtype != q.dtype:
            raise TypeError("all token tensors and o must share one dtype")
    for t in (initial_state, final_state):
        if t is not None and t.dtype != torch.float32:
            raise TypeError("states are float32")
    need = gdn2_chunk_fwd_workspace_size(B, T, Hk, Hv, dk, dv, C, dt, path)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = lib.gdn2_chunk_fwd_path(PATHS[path], _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(w),
                                 _ptr(initial_state), _ptr(final_state), _ptr(o), B, T, Hk, Hv, dk, dv,
                                 C, float(scale), dt, _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "gdn2_chunk_fwd")
    return o, final_state


def gdn2_chunk_fwd_noalloc(q, k, v, g, b, w, o, initial_state=None, final_state=None, *, C=64, scale=1.0,
                           stream=None):
    """Chunked forward without a caller workspace (C ABI gdn2_chunk_fwd_noalloc): for callers that
    cannot allocate device memory; the library's fixed 32 MiB device array serves as workspace."""
    B, T, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    st = lib.gdn2_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(w), _ptr(initial_state),
                                    _ptr(final_state), _ptr(o), B, T, Hk, Hv, dk, dv, C, float(scale),
                                    _dtype_code(q), _stream(stream))
    _check(st, "gdn2_chunk_fwd_noalloc")
    return o, final_state


def gdn2_recurrent_step(q, k, v, g, b, w, state, o, *, scale=1.0, stream=None):
    """One decode token (C ABI gdn2_recurrent_step); updates `state` in place and writes `o`.

    q, k: [B, H_k, d_k]; v, w: [B, H_v, d_v]; g, b: [B, H_v, d_k]; state: [B, H_v, d_k, d_v] fp32.
    """
    B, Hk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    dt = _dtype_code(q)
    st = lib.gdn2_recurrent_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(w), _ptr(state),
                                 _ptr(o), B, Hk, Hv, dk, dv, float(scale), dt, _stream(stream))
    _check(st, "gdn2_recurrent_step")
    return o


def gdn2_recurrent_update(q, k, v, g, b, w, state, o, slots=None, *, scale=1.0, stream=None):
    """N tokens per call (C ABI gdn2_recurrent_update); updates `state` in place and writes `o`.

    q, k: [B, N, H_k, d_k]; v, w, o: [B, N, H_v, d_v]; g, b: [B, N, H_v, d_k]. state: float32 or
    bfloat16, [B, H_v, d_k, d_v], or a pool [n_slots, H_v, d_k, d_v] when `slots` (int32 [B]) is given.
    """
    import torch

    B, N, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    sdt = _dtype_code(state)
    n_slots = state.shape[0] if slots is not None else 0
    if slots is not None and slots.dtype != torch.int32:
        raise TypeError("slots must be int32")
    st = lib.gdn2_recurrent_update(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(b), _ptr(w), _ptr(state), sdt,
                                   _ptr(slots), n_slots, _ptr(o), B, N, Hk, Hv, dk, dv, float(scale),
                                   _dtype_code(q), _stream(stream))
    _check(st, "gdn2_recurrent_update")
    return o


def gdn2_fg2_inputs(q, k, beta, q_out, k_out, b_out, w_out, *, stream=None):
    """FG^2-GDN inputs for the GDN-2 core (C ABI gdn2_fg2_inputs): writes q_out, k_out = sqrt(beta).k,
    b_out = 1, w_out = sqrt(beta), all per value head.

    q, k: [B, T, H_k, d] (or [B, H_k, d] for decode tokens); beta and the outputs: [B, T, H_v, d]
    (or [B, H_v, d]).
    """
    if q.dim() == 3:
        B, Hk, d = q.shape
        T, Hv = 1, beta.shape[1]
    else:
        B, T, Hk, d = q.shape
        Hv = beta.shape[2]
    st = lib.gdn2_fg2_inputs(_ptr(q), _ptr(k), _ptr(beta), _ptr(q_out), _ptr(k_out), _ptr(b_out), _ptr(w_out),
                             B, T, Hk, Hv, d, _dtype_code(q), _stream(stream))
    _check(st, "gdn2_fg2_inputs")
    return q_out, k_out, b_out, w_out


def fg2_inputs(q, k, beta, *, stream=None):
    """Returns (q_out, k_out, b_out, w_out) for running FG^2-GDN on the GDN-2 core (H_k = H_v)."""
    import torch

    outs = [torch.empty(beta.shape, dtype=q.dtype, device=q.device) for _ in range(4)]
    return gdn2_fg2_inputs(q, k, beta, *outs, stream=stream)


def gdn2_mixer_prologue(xq, xk, xv, conv_q, conv_k, conv_v, ag, ab, aw, q, k, v, g, b, w, states=None, *,
                        neg_eigval=False, stream=None):
    """ShortConv + L2 norm + gate activations (C ABI gdn2_mixer_prologue). Shapes as the core's
    inputs ([B, T, H, d], or [B, H, d] for one decode token); conv weights fp32 [H * d, 4];
    `states`: None or (state_q, state_k, state_v) fp32 [B, 3, H * d] tensors (each may be None),
    updated in place."""
    if xq.dim() == 3:
        B, Hk, dk = xq.shape
        T, Hv, dv = 1, xv.shape[1], xv.shape[2]
    else:
        B, T, Hk, dk = xq.shape
        Hv, dv = xv.shape[2], xv.shape[3]
    sq, sk, sv = states if states is not None else (None, None, None)
    st = lib.gdn2_mixer_prologue(*(_ptr(t) for t in (xq, xk, xv, conv_q, conv_k, conv_v, ag, ab, aw, sq, sk, sv,
                                                    q, k, v, g, b, w)),
                                 B, T, Hk, Hv, dk, dv, int(bool(neg_eigval)), _dtype_code(xq), _stream(stream))
    _check(st, "gdn2_mixer_prologue")
    return q, k, v, g, b, w


def gdn2_mixer_epilogue(o, z, weight, y, *, eps=1e-5, stream=None):
    """Gated RMSNorm with a SiLU gate (C ABI gdn2_mixer_epilogue); o, z, y: [B, T, H_v, d_v] (or
    [B, H_v, d_v]); weight: fp32 [d_v]."""
    if o.dim() == 3:
        B, Hv, dv = o.shape
        T = 1
    else:
        B, T, Hv, dv = o.shape
    st = lib.gdn2_mixer_epilogue(_ptr(o), _ptr(z), _ptr(weight), float(eps), _ptr(y), B, T, Hv, dv,
                                 _dtype_code(o), _stream(stream))
    _check(st, "gdn2_mixer_epilogue")
    return y


def gdn2_backward(q, k, v, g, b, w, d_o, dq, dk, dv, dg, db, dw, initial_state=None, d_final_state=None,
                  d_initial_state=None, *, scale=1.0, workspace=None, stream=None, recurrent=False):
    """Gradients of the core (C ABI gdn2_backward, or gdn2_backward_recurrent when `recurrent`);
    writes dq, dk, dv, dg, db, dw and, if given, d_initial_state. Shapes as gdn2_chunk_fwd's
    inputs; states fp32 [B, H_v, d_k, d_v]."""
    import torch

    B, T, Hk, dk_ = q.shape
    Hv, dv_ = v.shape[2], v.shape[3]
    dt = _dtype_code(q)
    size_fn = lib.gdn2_backward_recurrent_workspace_size if recurrent else lib.gdn2_backward_workspace_size
    fn = lib.gdn2_backward_recurrent if recurrent else lib.gdn2_backward
    need = size_fn(B, T, Hk, Hv, dk_, dv_, dt)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    st = fn(*(_ptr(t) for t in (q, k, v, g, b, w, initial_state, d_o, d_final_state, dq, dk, dv, dg, db, dw,
                                d_initial_state)),
            B, T, Hk, Hv, dk_, dv_, float(scale), dt, _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "gdn2_backward_recurrent" if recurrent else "gdn2_backward")
    return dq, dk, dv, dg, db, dw


def backward(q, k, v, g, b, w, d_o, initial_state=None, d_final_state=None, *, scale=1.0, stream=None,
             recurrent=False):
    """Returns (dq, dk, dv, dg, db, dw, d_initial_state)."""
    import torch

    outs = [torch.empty_like(t) for t in (q, k, v, g, b, w)]
    B, Hv, dk_, dv_ = q.shape[0], v.shape[2], q.shape[3], v.shape[3]
    ds0 = torch.empty((B, Hv, dk_, dv_), dtype=torch.float32, device=q.device)
    gdn2_backward(q, k, v, g, b, w, d_o, *outs, initial_state, d_final_state, ds0, scale=scale, stream=stream,
                  recurrent=recurrent)
    return (*outs, ds0)


def gdn2_last_device_status(stream=None) -> int:
    return lib.gdn2_last_device_status(_stream(stream))


def gdn2_set_wait_limit(ns: int) -> None:
    lib.gdn2_set_wait_limit(int(ns))


def gdn2_selftest_umma(case_id: int, soft: int, a, b, d, stream=None):
    _check(lib.gdn2_selftest_umma(case_id, soft, _ptr(a), _ptr(b), _ptr(d), _stream(stream)),
           "gdn2_selftest_umma")
    return d


# ---- convenience wrappers that allocate outputs (torch is used for memory only) -------------------

def chunk_fwd(q, k, v, g, b, w, initial_state=None, *, output_final_state=True, C=64, scale=1.0,
              path="auto", workspace=None, stream=None):
    """Returns (o, final_state or None)."""
    import torch

    B, T, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    o = torch.empty((B, T, Hv, dv), dtype=q.dtype, device=q.device)
    fs = torch.empty((B, Hv, dk, dv), dtype=torch.float32, device=q.device) if output_final_state else None
    return gdn2_chunk_fwd(q, k, v, g, b, w, o, initial_state, fs, C=C, scale=scale, workspace=workspace,
                          path=path, stream=stream)


def recurrent_step(q, k, v, g, b, w, state, *, scale=1.0, stream=None):
    """Returns o; `state` is updated in place."""
    import torch

    o = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    return gdn2_recurrent_step(q, k, v, g, b, w, state, o, scale=scale, stream=stream)


def gdn2_mixer_decode_step(xq, xk, xv, conv_q, conv_k, conv_v, ag, ab, aw, state, z, weight, y, *,
                           states=(None, None, None), eps=1e-5, neg_eigval=False, scale=1.0, stream=None):
    """One decode token of the whole mixer (C ABI gdn2_mixer_decode_step): conv + L2 norm + gates,
    the recurrent update of `state` (in place) and the gated RMSNorm into `y`.

    xq, xk: [B, H_k, d_k]; xv, z, y: [B, H_v, d_v]; ag, ab: [B, H_v, d_k]; aw: [B, H_v, d_v] (one dtype);
    conv_*: float32 [channels, 4]; states: float32 conv states [B, 3, channels] or None (updated in
    place); state: float32 [B, H_v, d_k, d_v]; weight: float32 [d_v].
    """
    B, Hk, dk = xq.shape
    Hv, dv = xv.shape[1], xv.shape[2]
    sq, sk, sv = states
    st = lib.gdn2_mixer_decode_step(_ptr(xq), _ptr(xk), _ptr(xv), _ptr(conv_q), _ptr(conv_k), _ptr(conv_v),
                                    _ptr(ag), _ptr(ab), _ptr(aw), _ptr(sq), _ptr(sk), _ptr(sv), _ptr(state),
                                    _ptr(z), _ptr(weight), float(eps), _ptr(y), B, Hk, Hv, dk, dv,
                                    int(bool(neg_eigval)), float(scale), _dtype_code(xq), _stream(stream))
    _check(st, "gdn2_mixer_decode_step")
    return y