"""fp64 CPU oracle for the gradients of the GDN-2 core (the recurrence of the burn-gdn2 0.1.5 docs,
"Architecture"): reverse-mode differentiation of the plain per-token recurrence with PyTorch's CPU
autograd in float64.

TEST INFRASTRUCTURE. Only tests/ may import this module. It shares no code with the CUDA path (and
none with oracle/gdn2_oracle.c: the forward below is written again, with torch operations, so that
autograd can differentiate it).

    S_t = (I - k_t (b_t . k_t)^T) diag(exp(g_t)) S_{t-1} + k_t (w_t . v_t)^T,   o_t = scale * S_t^T q_t
Given upstream gradients dO (for o) and dS_T (for the final state, optional), returns the gradients
of sum(o * dO) + sum(S_T * dS_T) with respect to q, k, v, g, b, w and the initial state.

Pinned by tests/test_backward_oracle.py: its forward equals the C oracle, and every gradient equals
central finite differences of the same functional on small inputs.
"""
from __future__ import annotations

import numpy as np


def forward_torch(q, k, v, g, b, w, s0, scale=1.0):
    """torch float64 tensors; q, k: [B, T, H_k, d_k]; v, w: [B, T, H_v, d_v]; g, b: [B, T, H_v, d_k];
    s0: [B, H_v, d_k, d_v]. Returns (o [B, T, H_v, d_v], S_T)."""
    import torch

    B, T, Hk, dk = q.shape
    Hv = v.shape[2]
    group = Hv // Hk
    qh = q.repeat_interleave(group, dim=2)      # key head of value head h: h // group
    kh = k.repeat_interleave(group, dim=2)
    S = s0
    outs = []
    for t in range(T):
        kt, qt = kh[:, t], qh[:, t]                                  # [B, H_v, d_k]
        S = torch.exp(g[:, t]).unsqueeze(-1) * S                     # diag(alpha) S
        r = torch.einsum("bhk,bhkv->bhv", b[:, t] * kt, S)           # (b . k)^T S'
        S = S + kt.unsqueeze(-1) * (w[:, t] * v[:, t] - r).unsqueeze(-2)
        outs.append(scale * torch.einsum("bhkv,bhk->bhv", S, qt))
    return torch.stack(outs, dim=1), S


def gradients(q, k, v, g, b, w, s0, do, ds_t=None, scale=1.0):
    """numpy inputs (any float dtype holding the stored values). Returns a dict of float64 arrays:
    dq, dk (per key head), dv, dg, db, dw, ds0, plus the forward o and S_T."""
    import torch

    t = lambda a: torch.tensor(np.asarray(a, dtype=np.float64), requires_grad=True)
    xs = [t(a) for a in (q, k, v, g, b, w)]
    B, T, Hv, dv = np.shape(v)
    dk = np.shape(q)[3]
    S0 = t(s0 if s0 is not None else np.zeros((B, Hv, dk, dv)))
    o, S = forward_torch(*xs, S0, scale=scale)
    loss = (o * torch.tensor(np.asarray(do, dtype=np.float64))).sum()
    if ds_t is not None:
        loss = loss + (S * torch.tensor(np.asarray(ds_t, dtype=np.float64))).sum()
    loss.backward()
    names = ("dq", "dk", "dv", "dg", "db", "dw")
    out = {n: x.grad.numpy() for n, x in zip(names, xs)}
    out["ds0"] = S0.grad.numpy()
    out["o"] = o.detach().numpy()
    out["s_t"] = S.detach().numpy()
    return out
