"""fp64 CPU oracle for FG^2-GDN, the gated delta rule with a per-channel learning rate.

TEST INFRASTRUCTURE. Only tests/ may import this module. It shares no code with the CUDA path.

Written from "FG^2-GDN: Enhancing Long-Context Gated Delta Networks with Doubly Fine-Grained
Control", section 2.A (FG2-GDN: vector learning rate): the rate beta_t in R^{d_k} is absorbed
symmetrically into key and value,
    k~_t = sqrt(beta_t) . k_t,   v~_t = sqrt(beta_t) . v_t,
    S_t  = (I - k~_t k~_t^T) Diag(alpha_t) S_{t-1} + k~_t v~_t^T,   alpha_t = exp(g_t).
The page prints the state update only; the readout o_t = scale * S_t^T q_t (after the update), the
head grouping (key head of value head h = floor(h * H_k / H_v)) and beta per value head are the
readings taken for the GDN-2 core and carried over. The value transform needs d_k = d_v.

Pinned by tests/test_fg2_oracle.py: with beta = 1 it equals the plain delta rule computed by the
GDN-2 oracle with b = w = 1; for unit k~ and no decay it retrieves v~ exactly; and planted mistakes
(the rate on the key only, a missing square root) are rejected.
"""
from __future__ import annotations

import numpy as np


def fg2_recurrent(q, k, v, g, beta, s0=None, scale=1.0):
    """q, k: [B, T, H_k, d]; v, g, beta: [B, T, H_v, d]; s0: [B, H_v, d, d] or None.
    Returns (o [B, T, H_v, d], S_T [B, H_v, d, d]) in float64."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    B, T, Hk, d = q.shape
    Hv = v.shape[2]
    if v.shape[3] != d:
        raise ValueError("FG^2-GDN's value transform needs d_k = d_v")
    o = np.zeros((B, T, Hv, d))
    s_out = np.zeros((B, Hv, d, d))
    for bi in range(B):
        for h in range(Hv):
            hk = h * Hk // Hv
            S = np.array(s0[bi, h], dtype=np.float64) if s0 is not None else np.zeros((d, d))
            for t in range(T):
                root = np.sqrt(beta[bi, t, h])
                kt = root * k[bi, t, hk]
                vt = root * v[bi, t, h]
                S = np.exp(g[bi, t, h])[:, None] * S              # Diag(alpha_t) S_{t-1}
                S = S - np.outer(kt, kt @ S) + np.outer(kt, vt)   # (I - k~ k~^T) (.) + k~ v~^T
                o[bi, t, h] = scale * (S.T @ q[bi, t, hk])
            s_out[bi, h] = S
    return o, s_out
