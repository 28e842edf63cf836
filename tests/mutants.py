"""Planted mistakes for the oracle's pins (CPU only, numpy, fp64).

Each mutant is a small re-implementation of the recurrence with ONE plausible mistake (a factor on
the wrong axis, a wrong order, a dropped term, a sign, an index). The pins in pins.py must reject
every one of them; test_oracle_mutants.py checks that. These are test fixtures, not oracles.
"""
from __future__ import annotations

import numpy as np


def _gate_dv(gate_dk, dv):
    """Reuse key-axis gates on the value axis (for mutants that put a key gate on the wrong axis)."""
    dk = gate_dk.shape[-1]
    if dv <= dk:
        return gate_dk[..., :dv]
    return np.concatenate([gate_dk, np.repeat(gate_dk[..., -1:], dv - dk, axis=-1)], axis=-1)


def recurrence(q, k, v, g, b, w, s0, mistake=None, scale=1.0):
    B, T, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    G = Hv // Hk
    o = np.zeros((B, T, Hv, dv))
    sT = np.zeros((B, Hv, dk, dv))
    for bi in range(B):
        for h in range(Hv):
            hk = (h % Hk) if mistake == "gqa_interleaved" else h // G
            S = np.zeros((dk, dv)) if s0 is None else np.array(s0[bi, h], dtype=np.float64)
            for t in range(T):
                qt, kt = q[bi, t, hk], k[bi, t, hk]
                gt, bt, vt, wt = g[bi, t, h], b[bi, t, h], v[bi, t, h], w[bi, t, h]
                prev = S
                tg = t - 1 if mistake == "decay_previous_token" else t
                alpha = np.exp(g[bi, max(tg, 0), h]) if tg >= 0 else np.ones(dk)
                if mistake == "decay_on_value_axis":
                    Sp = S * np.exp(_gate_dv(gt, dv))[None, :]
                elif mistake == "decay_missing":
                    Sp = S
                elif mistake == "decay_after_erase":
                    Sp = S                     # erase reads the undecayed state; decay applied after
                else:
                    Sp = alpha[:, None] * S
                if mistake == "erase_on_written_factor":
                    Snew = Sp - np.outer(bt * kt, kt @ Sp) + np.outer(kt, wt * vt)
                elif mistake == "erase_sign":
                    Snew = Sp + np.outer(kt, (bt * kt) @ Sp) + np.outer(kt, wt * vt)
                elif mistake == "write_gate_dropped":
                    Snew = Sp - np.outer(kt, (bt * kt) @ Sp) + np.outer(kt, vt)
                elif mistake == "erase_gate_dropped":
                    Snew = Sp - np.outer(kt, kt @ Sp) + np.outer(kt, wt * vt)
                elif mistake == "write_gate_on_key_axis":
                    Snew = Sp - np.outer(kt, (bt * kt) @ Sp) + np.outer(_gate_dv(wt, dk) * kt, vt)
                else:
                    Snew = Sp - np.outer(kt, (bt * kt) @ Sp) + np.outer(kt, wt * vt)
                if mistake == "decay_after_erase":
                    Snew = alpha[:, None] * Snew
                S = Snew
                if mistake == "readout_before_update":
                    o[bi, t, h] = scale * (prev.T @ qt)
                elif mistake == "transposed_readout" and dk == dv:
                    o[bi, t, h] = scale * (S @ qt)
                else:
                    o[bi, t, h] = scale * (S.T @ qt)
            sT[bi, h] = S
    return o, sT


def chunked(q, k, v, g, b, w, s0, C=4, mistake=None):
    """Chunked WY/UT form (fp64, numpy), with one planted mistake."""
    B, T, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    G_ = Hv // Hk
    o = np.zeros((B, T, Hv, dv))
    sT = np.zeros((B, Hv, dk, dv))
    for bi in range(B):
        for h in range(Hv):
            hk = h // G_
            S = np.zeros((dk, dv)) if s0 is None else np.array(s0[bi, h], dtype=np.float64)
            for t0 in range(0, T, C):
                n = min(C, T - t0)
                qc, kc = q[bi, t0:t0 + n, hk], k[bi, t0:t0 + n, hk]
                gc, bc, vc, wc = g[bi, t0:t0 + n, h], b[bi, t0:t0 + n, h], v[bi, t0:t0 + n, h], w[bi, t0:t0 + n, h]
                Gm = np.cumsum(gc, axis=0)
                if mistake == "cumdecay_exclusive":
                    Gm = Gm - gc
                D = np.exp(Gm[:, None, :] - Gm[None, :, :])            # [i, j, c]
                A = np.einsum("ic,ic,jc,ijc->ij", bc, kc, kc, D)
                M = np.einsum("ic,jc,ijc->ij", qc, kc, D)
                A = np.tril(A, -1)
                M = np.tril(M, -1) if mistake == "causal_mask_strict" else np.tril(M, 0)
                Tm = np.linalg.inv(np.eye(n) + A)
                if mistake == "inverse_sign":
                    Tm = np.linalg.inv(np.eye(n) - A)
                W = Tm @ (bc * kc * np.exp(Gm))
                Ut = Tm @ (wc * vc)
                U = Ut if mistake == "u_without_state" else Ut - W @ S
                O = (qc * np.exp(Gm)) @ S + M @ U
                S = np.exp(Gm[-1])[:, None] * S + (kc * np.exp(Gm[-1] - Gm)).T @ U
                o[bi, t0:t0 + n, h] = O
            sT[bi, h] = S
    return o, sT


RECURRENT_MISTAKES = [
    "erase_on_written_factor", "decay_after_erase", "readout_before_update", "write_gate_dropped",
    "decay_on_value_axis", "erase_sign", "transposed_readout", "gqa_interleaved",
    "decay_previous_token", "decay_missing", "erase_gate_dropped", "write_gate_on_key_axis",
]
CHUNKED_MISTAKES = ["cumdecay_exclusive", "causal_mask_strict", "inverse_sign", "u_without_state"]
