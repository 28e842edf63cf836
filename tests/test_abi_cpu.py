"""The C ABI without a GPU: the library loads, exports every function include/gdn2.h declares, and
rejects bad arguments on the host before touching the device (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "gdn2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn2_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def g():
    import __graft_entry__

    __graft_entry__._build_module().build()
    import gated_deltanet_mixer_gdn2_gb300 as mod

    return mod


def test_header_declares_the_two_entry_points():
    names = _declared_functions()
    for fn in ("gdn2_chunk_fwd", "gdn2_recurrent_step", "gdn2_chunk_fwd_workspace_size",
               "gdn2_status_string", "gdn2_last_device_status"):
        assert fn in names


def test_every_declared_symbol_is_exported(g):
    lib = ctypes.CDLL(g.LIB_PATH)
    for fn in _declared_functions():
        assert hasattr(lib, fn), f"{fn} declared in include/gdn2.h but not exported"
    assert set(g.EXPORTS) == set(_declared_functions())


def _declared_arity():
    """Parameter count of every prototype in include/gdn2.h."""
    src = open(os.path.join(ROOT, "include", "gdn2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    out = {}
    for m in re.finditer(r"\b(gdn2_[a-z0-9_]+)\s*\(", src):
        depth, i = 1, m.end()
        while depth:
            depth += {"(": 1, ")": -1}.get(src[i], 0)
            i += 1
        params = src[m.end():i - 1].strip()
        if src[i:].lstrip().startswith(";"):  # a prototype, not a use inside another declaration
            out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header(g):
    arity = _declared_arity()
    assert set(arity) == set(g.EXPORTS)
    for fn, n in arity.items():
        assert len(getattr(g.lib, fn).argtypes) == n, (fn, n, len(getattr(g.lib, fn).argtypes))


def test_status_strings(g):
    for s in range(0, -7, -1):
        assert g.status_string(s) and g.status_string(s) != "unknown status"
    assert g.status_string(42) == "unknown status"


def test_workspace_sizes(g):
    # tensor-core path: one 66048-byte unit per (chunk, batch, value head), then the exact kernel's list
    # (a count and one int32 per unit, rounded up to 256 bytes)
    tail = lambda units: -(-4 * (units + 1) // 256) * 256
    assert g.gdn2_chunk_fwd_workspace_size(2, 32768, 16, 32, 128, 128, 64, g.GDN2_BF16) == \
        66048 * 512 * 64 + tail(512 * 64)
    # ragged tail rounds the chunk count up
    assert g.gdn2_chunk_fwd_workspace_size(1, 65, 1, 1, 128, 128, 64, g.GDN2_BF16) == 66048 * 2 + 256
    # the no-alloc entry point's 32 MiB array holds exactly 508 units and their list
    assert 66048 * 508 + tail(508) == 32 << 20
    # fp32 goes to the SIMT path: (3 dk C + C^2 + dv C + dk) floats, rounded to 4
    n = 3 * 64 * 64 + 64 * 64 + 64 * 64 + 64
    assert g.gdn2_chunk_fwd_workspace_size(1, 256, 4, 4, 64, 64, 64, g.GDN2_F32) == 4 * n * 4 * 4
    assert g.gdn2_chunk_fwd_workspace_size(1, 0, 4, 4, 64, 64, 64, g.GDN2_F32) == 0
    assert g.gdn2_chunk_fwd_workspace_size(1, 10, 3, 4, 64, 64, 64, g.GDN2_F32) == 0        # Hv % Hk
    assert g.gdn2_chunk_fwd_workspace_size(1, 10, 4, 4, 72, 64, 64, g.GDN2_F32) == 0        # dk % 16
    assert g.gdn2_chunk_fwd_workspace_size(1, 10, 4, 4, 32, 64, 64, g.GDN2_BF16, "tcgen05") == 0
    # d_k = 64 runs as d_k = 128 with zero channels: the same units
    assert g.gdn2_chunk_fwd_workspace_size(1, 10, 4, 4, 64, 64, 64, g.GDN2_BF16, "tcgen05") == 66048 * 4 + 256
    # the tensor-core units hold d_k-side factors only: the same workspace for every d_v
    for dv in (64, 256, 512):
        assert g.gdn2_chunk_fwd_workspace_size(1, 65, 1, 1, 128, dv, 64, g.GDN2_BF16) == 66048 * 2 + 256


def _chunk(g, path=0, B=1, T=8, Hk=1, Hv=1, dk=128, dv=128, C=64, dt=1, ptr=0x10000, ws=None, wsb=1 << 30,
           s0=None, sT=None):
    p = ctypes.c_void_p(ptr) if ptr else None
    return g.lib.gdn2_chunk_fwd_path(path, p, p, p, p, p, p, s0, sT, p, B, T, Hk, Hv, dk, dv, C, 1.0, dt,
                                     ctypes.c_void_p(ws if ws is not None else ptr), wsb, None)


def test_chunk_argument_errors(g):
    assert _chunk(g, ptr=0) == g.GDN2_ERR_INVALID_ARG                 # null tensors
    assert _chunk(g, Hk=3, Hv=4) == g.GDN2_ERR_INVALID_ARG            # H_v % H_k
    assert _chunk(g, T=-1) == g.GDN2_ERR_INVALID_ARG
    assert _chunk(g, dt=7) == g.GDN2_ERR_INVALID_ARG
    assert _chunk(g, path=9) == g.GDN2_ERR_INVALID_ARG
    assert _chunk(g, dk=72) == g.GDN2_ERR_UNSUPPORTED
    assert _chunk(g, C=48) == g.GDN2_ERR_UNSUPPORTED
    assert _chunk(g, path=2, dt=0) == g.GDN2_ERR_UNSUPPORTED           # tensor cores need bf16
    assert _chunk(g, path=2, dk=32, dv=64) == g.GDN2_ERR_UNSUPPORTED    # tensor cores: d_k 128 or 64
    assert _chunk(g, path=2, dv=96) == g.GDN2_ERR_UNSUPPORTED           # tensor cores: d_v in 64-column slices
    assert _chunk(g, path=2, dv=576) == g.GDN2_ERR_UNSUPPORTED
    assert _chunk(g, path=1, dv=272) == g.GDN2_ERR_UNSUPPORTED          # SIMT: d_v up to 256
    assert _chunk(g, B=32768, T=1, Hv=4) == g.GDN2_ERR_UNSUPPORTED     # B * H_v beyond the grid's y range
    assert g.lib.gdn2_chunk_fwd_workspace_size(32768, 1, 1, 4, 128, 128, 64, 1) == 0
    assert _chunk(g, ptr=0x10008) == g.GDN2_ERR_MISALIGNED
    assert _chunk(g, ws=0) == g.GDN2_ERR_WORKSPACE
    assert _chunk(g, wsb=100) == g.GDN2_ERR_WORKSPACE
    assert _chunk(g, ws=0x10004) == g.GDN2_ERR_MISALIGNED
    assert _chunk(g, s0=ctypes.c_void_p(0x10004)) == g.GDN2_ERR_MISALIGNED
    # empty problems need no tensors at all (nothing to copy without a final state)
    assert _chunk(g, ptr=0, T=0) == g.GDN2_OK
    assert _chunk(g, ptr=0, B=0) == g.GDN2_OK


def test_decode_argument_errors(g):
    P = ctypes.c_void_p(0x10000)
    f = lambda B=1, Hk=1, Hv=1, dk=128, dv=128, dt=1, p=P: g.lib.gdn2_recurrent_step(
        p, p, p, p, p, p, p, p, B, Hk, Hv, dk, dv, 1.0, dt, None)
    assert f(p=None) == g.GDN2_ERR_INVALID_ARG
    assert f(Hk=2, Hv=3) == g.GDN2_ERR_INVALID_ARG
    assert f(dk=96) == g.GDN2_ERR_UNSUPPORTED
    assert f(dv=100) == g.GDN2_ERR_UNSUPPORTED
    assert f(dv=1024) == g.GDN2_ERR_UNSUPPORTED
    assert f(p=ctypes.c_void_p(0x10002)) == g.GDN2_ERR_MISALIGNED
    assert f(B=0, p=None) == g.GDN2_OK
    assert f(dt=3) == g.GDN2_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(g):
    import torch

    x = torch.zeros(1, 4, 1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        g.chunk_fwd(x, x, x, x, x, x)


def test_product_path_does_not_touch_the_oracle():
    """The package and its sources never import or name the oracle / test infrastructure."""
    pkg = os.path.join(ROOT, "gated_deltanet_mixer_gdn2_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.lower(), f"{f} mentions the oracle"
                assert "import synth" not in src and "from synth" not in src


def test_recurrent_update_argument_errors(g):
    P = ctypes.c_void_p(0x10000)
    f = lambda sdt=0, slots=None, n_slots=0, B=1, N=2, dk=128, dv=128, dt=1, p=P: g.lib.gdn2_recurrent_update(
        p, p, p, p, p, p, p, sdt, slots, n_slots, p, B, N, 1, 1, dk, dv, 1.0, dt, None)
    assert f(sdt=5) == g.GDN2_ERR_INVALID_ARG
    assert f(N=-1) == g.GDN2_ERR_INVALID_ARG
    assert f(slots=ctypes.c_void_p(0x20000), n_slots=-1) == g.GDN2_ERR_INVALID_ARG
    assert f(slots=ctypes.c_void_p(0x20002), n_slots=4) == g.GDN2_ERR_MISALIGNED
    assert f(dk=48) == g.GDN2_ERR_UNSUPPORTED
    assert f(p=None) == g.GDN2_ERR_INVALID_ARG
    assert f(N=0, p=None) == g.GDN2_OK


def test_fg2_inputs_argument_errors(g):
    P = lambda a: ctypes.c_void_p(a) if a else None
    f = lambda ptr=0x10000, B=1, T=4, Hk=1, Hv=2, d=128, dt=1: g.lib.gdn2_fg2_inputs(
        *(P(ptr),) * 7, B, T, Hk, Hv, d, dt, None)
    assert f(B=0) == g.GDN2_OK                                   # nothing to do, nothing launched
    assert f(ptr=0) == g.GDN2_ERR_INVALID_ARG
    assert f(Hk=3, Hv=4) == g.GDN2_ERR_INVALID_ARG
    assert f(dt=5) == g.GDN2_ERR_INVALID_ARG
    assert f(T=-1) == g.GDN2_ERR_INVALID_ARG
    assert f(d=12) == g.GDN2_ERR_UNSUPPORTED
    assert f(ptr=0x10008) == g.GDN2_ERR_MISALIGNED


def test_mixer_argument_errors(g):
    P = lambda a: ctypes.c_void_p(a) if a else None
    pro = lambda ptr=0x10000, B=1, T=4, Hk=1, Hv=2, dk=128, dv=128, dt=1, st=0: g.lib.gdn2_mixer_prologue(
        *(P(ptr),) * 9, *(P(st),) * 3, *(P(ptr),) * 6, B, T, Hk, Hv, dk, dv, 0, dt, None)
    assert pro(T=0) == g.GDN2_OK
    assert pro(ptr=0) == g.GDN2_ERR_INVALID_ARG
    assert pro(Hk=3, Hv=4) == g.GDN2_ERR_INVALID_ARG
    assert pro(dt=3) == g.GDN2_ERR_INVALID_ARG
    assert pro(dk=96) == g.GDN2_ERR_UNSUPPORTED
    assert pro(ptr=0x10004) == g.GDN2_ERR_MISALIGNED
    assert pro(st=0x10008) == g.GDN2_ERR_MISALIGNED
    epi = lambda ptr=0x10000, eps=1e-5, dv=128, B=1: g.lib.gdn2_mixer_epilogue(
        P(ptr), P(ptr), P(ptr), eps, P(ptr), B, 4, 2, dv, 1, None)
    assert epi(B=0) == g.GDN2_OK
    assert epi(ptr=0) == g.GDN2_ERR_INVALID_ARG
    assert epi(eps=-1.0) == g.GDN2_ERR_INVALID_ARG
    assert epi(eps=float("nan")) == g.GDN2_ERR_INVALID_ARG
    assert epi(dv=48) == g.GDN2_ERR_UNSUPPORTED
    assert epi(ptr=0x10002) == g.GDN2_ERR_MISALIGNED


@pytest.mark.parametrize("entry", ["gdn2_backward", "gdn2_backward_recurrent"])
def test_backward_argument_errors(g, entry):
    P = lambda a: ctypes.c_void_p(a) if a else None
    fn = getattr(g.lib, entry)
    f = lambda ptr=0x10000, B=1, T=4, Hk=1, Hv=2, dk=128, dv=128, dt=1, ws=0x10000, wsb=1 << 40: fn(
        *(P(ptr),) * 6, None, P(ptr), None, *(P(ptr),) * 6, None, B, T, Hk, Hv, dk, dv, 1.0, dt, P(ws), wsb, None)
    assert f(ptr=0) == g.GDN2_ERR_INVALID_ARG
    assert f(Hk=3, Hv=4) == g.GDN2_ERR_INVALID_ARG
    assert f(dt=4) == g.GDN2_ERR_INVALID_ARG
    assert f(dk=64, dv=64, dt=0) == g.GDN2_ERR_UNSUPPORTED  # fp32: head size 128 only
    assert f(dk=32, dv=128) == g.GDN2_ERR_UNSUPPORTED
    assert f(dk=128, dv=192) == g.GDN2_ERR_UNSUPPORTED
    assert f(ptr=0x10004) == g.GDN2_ERR_MISALIGNED
    assert f(ws=0) == g.GDN2_ERR_WORKSPACE
    assert f(wsb=16) == g.GDN2_ERR_WORKSPACE
    assert f(B=32768, T=1, Hv=4) == g.GDN2_ERR_UNSUPPORTED  # (batch, value head) beyond the grid's y range
    size = getattr(g.lib, entry + "_workspace_size")
    assert size(2, 100, 1, 2, 64, 64, 0) == 0
    assert size(2, 100, 1, 2, 32, 32, 1) == 0
    assert size(32768, 1, 1, 4, 128, 128, 1) == 0
    assert size(2, 0, 1, 2, 128, 128, 1) == 0
    # bf16: the chunked form also takes head size 64 (the per-token form does not)
    assert (size(2, 100, 1, 2, 64, 64, 1) > 0) == (entry == "gdn2_backward")
    assert (f(dk=64, dv=64, wsb=16) == g.GDN2_ERR_WORKSPACE) == (entry == "gdn2_backward")


def test_backward_workspace_sizes(g):
    n = g.lib.gdn2_backward_workspace_size(2, 100, 1, 2, 128, 128, g.GDN2_F32)
    units = 2 * 2 * ((100 + 31) // 32)   # (batch, value head, 32-token chunk)
    # fp32 path, per unit: S entering and dS leaving the chunk, U and dU, T; then fp32 dq and dk per value head
    assert n >= units * (2 * 128 * 128 + 2 * 32 * 128 + 32 * 32) * 4 + 2 * 2 * 100 * 2 * 128 * 4
    nb = g.lib.gdn2_backward_workspace_size(2, 100, 1, 2, 128, 128, g.GDN2_BF16)
    units64 = 2 * 2 * ((100 + 63) // 64)  # (batch, value head, 64-token chunk)
    # tensor-core path, per unit: the forward factors (66 048 bytes), bf16 S, dS', U, dU; then fp32 dq and dk
    # per value head
    assert nb >= units64 * (66048 + (2 * 128 * 128 + 2 * 64 * 128) * 2) + 2 * 2 * 100 * 2 * 128 * 4
    r = g.lib.gdn2_backward_recurrent_workspace_size(2, 100, 1, 2, 128, 128, 1)
    # one fp32 state per 32-token stretch for each (batch, value head)
    assert r >= units * 128 * 128 * 4


def test_mixer_decode_step_argument_errors(g):
    P = ctypes.c_void_p(0x10000)

    def f(B=1, Hk=1, Hv=2, dk=128, dv=128, dt=1, eps=1e-5, p=P, sq=None):
        return g.lib.gdn2_mixer_decode_step(p, p, p, p, p, p, p, p, p, sq, None, None, p, p, p, eps, p, B, Hk, Hv, dk,
                                            dv, 0, 1.0, dt, None)

    assert f(dt=5) == g.GDN2_ERR_INVALID_ARG
    assert f(Hk=2, Hv=3) == g.GDN2_ERR_INVALID_ARG
    assert f(eps=-1.0) == g.GDN2_ERR_INVALID_ARG
    assert f(eps=float("nan")) == g.GDN2_ERR_INVALID_ARG
    assert f(p=None) == g.GDN2_ERR_INVALID_ARG
    assert f(dk=32) == g.GDN2_ERR_UNSUPPORTED
    assert f(dv=256) == g.GDN2_ERR_UNSUPPORTED
    assert f(p=ctypes.c_void_p(0x10008)) == g.GDN2_ERR_MISALIGNED
    assert f(sq=ctypes.c_void_p(0x10004)) == g.GDN2_ERR_MISALIGNED
    assert f(B=0) == g.GDN2_OK
