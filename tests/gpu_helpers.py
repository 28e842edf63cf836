"""Helpers shared by the GPU tests: upload synthetic inputs, run the CUDA path through the C ABI
binding, bring results back as float64 numpy arrays."""
from __future__ import annotations

import numpy as np

import synth

BF16_TOL = 2e-2   # max normwise relative error, bf16 token inputs, fp32 state / accumulation
F32_TOL = 1e-4    # same for fp32 token inputs


def tol_for(dtype: str) -> float:
    return BF16_TOL if dtype == "bf16" else F32_TOL


def check(name: str, got, ref, tol: float, head_axis: int | None = 2) -> str:
    """Parity of a CUDA result with the oracle's: finite, normwise max relative error <= tol over the
    whole tensor and, when head_axis is given, over every (batch, head) slice on its own (a bad head
    of small magnitude cannot hide under the others). Returns a one-line report that also gives the
    elementwise relative error with a floor of 1e-3 * max|ref| (reported, not bounded: near-zero
    elements of bf16 results carry the rounding of much larger ones)."""
    import oracle

    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{name}: shape {got.shape} != {ref.shape}"
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    err = oracle.max_rel_err(got, ref)
    ele = oracle.max_rel_err_elementwise(got, ref)
    assert err <= tol, f"{name}: max rel err {err:.3e} > {tol:.1e} (elementwise {ele:.3e})"
    worst = 0.0
    if head_axis is not None and got.ndim == 4:
        g2 = np.moveaxis(got, head_axis, 1)
        r2 = np.moveaxis(ref, head_axis, 1)
        for bi in range(g2.shape[0]):
            for h in range(g2.shape[1]):
                e = oracle.max_rel_err(g2[bi, h], r2[bi, h])
                assert e <= tol, f"{name}: head ({bi}, {h}) max rel err {e:.3e} > {tol:.1e}"
                worst = max(worst, e)
    return f"{name}: normwise {err:.2e}, worst head {worst:.2e}, elementwise (floor 1e-3 max) {ele:.2e}"


def upload(inp: synth.Inputs, t0: int, t1: int, device="cuda"):
    """Token tensors for tokens [t0, t1) as device tensors of the storage dtype."""
    sl = lambda a: np.ascontiguousarray(a[:, t0:t1])
    return tuple(synth.to_torch(sl(getattr(inp, n)), inp.dtype, device) for n in ("q", "k", "v", "g", "b", "w"))


def upload_token(inp: synth.Inputs, t: int, device="cuda"):
    """Token t of every token tensor, shaped [B, H, d] for a decode step."""
    return tuple(synth.to_torch(np.ascontiguousarray(getattr(inp, n)[:, t]), inp.dtype, device)
                 for n in ("q", "k", "v", "g", "b", "w"))


def state_to_device(s0, device="cuda"):
    import torch

    if s0 is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(s0, dtype=np.float32)).to(device)


def to_np(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def run_chunk(g, inp: synth.Inputs, C: int = 64, path: str = "auto", t0: int = 0, t1: int | None = None,
              s0=None, scale: float = 1.0):
    """Chunked forward on tokens [t0, t1); s0 defaults to the inputs' own initial state."""
    t1 = inp.q.shape[1] if t1 is None else t1
    q, k, v, gg, b, w = upload(inp, t0, t1)
    s0d = state_to_device(inp.s0 if s0 is None else s0)
    o, st = g.chunk_fwd(q, k, v, gg, b, w, s0d, C=C, path=path, scale=scale)
    status = g.gdn2_last_device_status()
    assert status == g.GDN2_OK, g.status_string(status)
    return to_np(o), st


def run_decode(g, inp: synth.Inputs, state, t0: int, t1: int, scale: float = 1.0):
    """Decode steps for tokens [t0, t1) against `state` (device fp32, updated in place)."""
    import torch

    outs = []
    for t in range(t0, t1):
        q, k, v, gg, b, w = upload_token(inp, t)
        outs.append(g.recurrent_step(q, k, v, gg, b, w, state, scale=scale))
    torch.cuda.synchronize()
    return to_np(torch.stack(outs, dim=1)) if outs else None


def heads_of(x: np.ndarray, units, axis_h: int = 2):
    """Gather (batch, value head) units from an array [B, T, H, d] (axis_h=2) or [B, H, dk, dv] (1)."""
    if axis_h == 2:
        return np.stack([x[bi, :, h] for bi, h in units])
    return np.stack([x[bi, h] for bi, h in units])
