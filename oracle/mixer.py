"""fp64 CPU oracle for the operations around the GDN-2 core in the token mixer: the prologue
(ShortConv, L2 norm of q and k, gate activations) and the epilogue (gated RMSNorm with a SiLU gate).

TEST INFRASTRUCTURE. Only tests/ may import this module. It shares no code with the CUDA path.

Written from the burn-gdn2 0.1.5 docs ("Architecture": projections -> ShortConv -> L2-Norm -> core ->
Gated RMS Norm <- SiLU Gate; configuration table: use_short_conv "depthwise conv before
recurrence", allow_neg_eigval "b x 2", norm_eps 1e-5 "output norm epsilon") and the llama.cpp GDN
decode study (section 1: conv_kernel = 4; section 2: the causal-conv state keeps the previous
conv_kernel - 1 = 3 samples, the new token is appended and the last 3 are written back).
Readings where the pages are silent (each listed in the design notes):
  * the conv runs on q, k and v (the projections that feed the core's matrix products), depthwise,
    causal, kernel 4, no bias and no activation after it:
        y_t[c] = sum_{j=0..3} W[c, j] x_{t-3+j}[c],  x_{t'} for t' < 0 taken from the carried state;
  * L2 norm of q and k per (token, head) over the head dimension: x / sqrt(sum x^2 + 1e-6);
  * gates: g = -softplus(a_g) (log alpha <= 0), b = sigmoid(a_b) (x 2 when negative eigenvalues are
    allowed), w = sigmoid(a_w);
  * epilogue per (token, value head) over d_v: y = o / sqrt(mean(o^2) + eps) * weight * silu(z),
    weight [d_v] shared by the heads, silu(z) = z * sigmoid(z), eps = 1e-5.
Pinned by tests/test_mixer_oracle.py.
"""
from __future__ import annotations

import numpy as np

CONV_K = 4
L2_EPS = 1e-6


def short_conv(x, weight, state=None):
    """x: [B, T, C]; weight: [C, 4] (tap 3 multiplies the current token); state: [B, 3, C] holding
    x_{-3}, x_{-2}, x_{-1} (None = zeros). Returns (y [B, T, C], new_state [B, 3, C])."""
    x = np.asarray(x, dtype=np.float64)
    B, T, C = x.shape
    prev = np.zeros((B, CONV_K - 1, C)) if state is None else np.asarray(state, dtype=np.float64)
    ext = np.concatenate([prev, x], axis=1)            # token t of x is row t + 3
    y = np.zeros((B, T, C))
    for t in range(T):
        for j in range(CONV_K):
            y[:, t] += np.asarray(weight, dtype=np.float64)[:, j] * ext[:, t + j]
    return y, ext[:, -(CONV_K - 1):].copy()


def l2_norm(x):
    """over the last axis"""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + L2_EPS)


def softplus(a):
    a = np.asarray(a, dtype=np.float64)
    return np.log1p(np.exp(-np.abs(a))) + np.maximum(a, 0.0)


def sigmoid(a):
    a = np.asarray(a, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-a))


def prologue(xq, xk, xv, wq, wk, wv, ag, ab, aw, states=(None, None, None), neg_eigval=False):
    """xq, xk: [B, T, H_k, d_k]; xv: [B, T, H_v, d_v]; wq, wk: [H_k * d_k, 4]; wv: [H_v * d_v, 4];
    ag, ab: [B, T, H_v, d_k]; aw: [B, T, H_v, d_v]; states: conv states [B, 3, channels] or None.
    Returns (q, k, v, g, b, w, (state_q, state_k, state_v))."""
    outs, new_states = [], []
    for x, wt, st in zip((xq, xk, xv), (wq, wk, wv), states):
        B, T, H, d = np.shape(x)
        y, ns = short_conv(np.reshape(x, (B, T, H * d)), wt, st)
        outs.append(y.reshape(B, T, H, d))
        new_states.append(ns)
    q, k, v = l2_norm(outs[0]), l2_norm(outs[1]), outs[2]
    g = -softplus(ag)
    b = sigmoid(ab) * (2.0 if neg_eigval else 1.0)
    w = sigmoid(aw)
    return q, k, v, g, b, w, tuple(new_states)


def epilogue(o, z, weight, eps=1e-5):
    """o, z: [B, T, H_v, d_v]; weight: [d_v]. Gated RMSNorm over d_v with a SiLU gate."""
    o = np.asarray(o, dtype=np.float64)
    z = np.asarray(z, dtype=np.float64)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return o / rms * np.asarray(weight, dtype=np.float64) * (z * sigmoid(z))
