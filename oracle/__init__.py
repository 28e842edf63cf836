"""fp64 CPU oracle for the Gated DeltaNet-2 token-mixer core (ctypes wrapper of gdn2_oracle.c).

TEST INFRASTRUCTURE. Only tests/, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import this package. It shares no code with the CUDA path and the CUDA path
never imports it.

The recurrence it follows is the one printed in the burn-gdn2 0.1.5 docs ("Architecture"):
``S_t = (I - k_t (b_t . k_t)^T) diag(alpha_t) S_{t-1} + k_t (w_t . v_t)^T``, ``o_t = S_t^T q_t``,
``alpha_t = exp(g_t)``. See gdn2_oracle.c for the three forms and the readings taken where the
page is silent.

Every function here is pinned by tests/test_oracle_pins.py (retrieval invariant, linear-attention
and scalar gated-delta-rule reductions, exact standard-basis-key cases, agreement of the three
forms, linearity, state chaining, and a set of planted mistakes that the pins must reject).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn2_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FORMS = {"recurrent": 0, "literal": 1, "chunked": 2}


def build(force: bool = False) -> str:
    """Compile gdn2_oracle.c into liboracle.so next to it (plain gcc, -O2, portable flags)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            f = lib.gdn2_oracle_run
            P = ctypes.c_void_p
            f.argtypes = [ctypes.c_int] + [P] * 9 + [ctypes.c_int] * 7 + [ctypes.c_double, ctypes.c_int]
            f.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def run(q, k, v, g, b, w, s0=None, *, form: str = "recurrent", C: int = 64, scale: float = 1.0,
        nthreads: int | None = None, want_o: bool = True):
    """Run the oracle.

    q, k: [B, T, H_k, d_k]; g, b: [B, T, H_v, d_k]; v, w: [B, T, H_v, d_v] (float arrays holding the
    stored values); s0: [B, H_v, d_k, d_v] or None (zeros). Returns (o [B, T, H_v, d_v] float64 or
    None, S_T [B, H_v, d_k, d_v] float64).
    """
    lib = _load()
    q, k, v, g, b, w = map(_f32, (q, k, v, g, b, w))
    B, T, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    assert k.shape == q.shape and g.shape == (B, T, Hv, dk) and b.shape == g.shape
    assert v.shape == (B, T, Hv, dv) and w.shape == v.shape
    s0d = None if s0 is None else np.ascontiguousarray(s0, dtype=np.float64)
    if s0d is not None:
        assert s0d.shape == (B, Hv, dk, dv)
    o = np.zeros((B, T, Hv, dv), np.float64) if want_o else None
    sT = np.zeros((B, Hv, dk, dv), np.float64)
    ptr = lambda a: None if a is None else a.ctypes.data
    rc = lib.gdn2_oracle_run(FORMS[form], ptr(q), ptr(k), ptr(v), ptr(g), ptr(b), ptr(w), ptr(s0d),
                             ptr(o), ptr(sT), B, T, Hk, Hv, dk, dv, C, float(scale),
                             nthreads or default_threads())
    if rc != 0:
        raise RuntimeError("gdn2_oracle_run failed (bad arguments or out of memory)")
    return o, sT


def run_inputs(inp, s0=None, **kw):
    """run() on a synth.Inputs; s0 defaults to the inputs' own initial state."""
    s0 = inp.s0 if s0 is None else s0
    return run(inp.q, inp.k, inp.v, inp.g, inp.b, inp.w, s0, **kw)


def max_rel_err(x, ref) -> float:
    """Normwise-max relative error max|x - ref| / max|ref| (0 when both are all-zero)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(x - ref))) if ref.size else 0.0
    if den == 0.0:
        return num
    return num / den


def max_rel_err_elementwise(x, ref, floor_frac: float = 1e-3) -> float:
    """Largest element-by-element relative error max_i |x_i - ref_i| / max(|ref_i|, floor), with the
    floor floor_frac * max|ref| (so elements near zero are measured against a small fraction of the
    tensor's scale rather than against themselves)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if not ref.size:
        return 0.0
    scale = float(np.max(np.abs(ref)))
    if scale == 0.0:
        return float(np.max(np.abs(x - ref)))
    den = np.maximum(np.abs(ref), floor_frac * scale)
    return float(np.max(np.abs(x - ref) / den))
