"""Seeded synthetic inputs for the Gated DeltaNet-2 token-mixer core.

This module is shared by the CPU oracle's tests, the GPU parity tests, ``smoke()`` and
``bench.py``. It holds random draws and the input recipe only (distributions, the
L2-normalisation of q and k that the mixer layer applies before its core, rounding to the
storage dtype). None of the recurrence's arithmetic lives here.

Recipe. Each (workload seed, tensor, batch index, head) slab has its own numpy PCG64 stream:

  q, k  ~ N(0,1), L2-normalised over d_k per (token, head)        [B, T, H_k, d_k]
  v     ~ N(0,1)                                                    [B, T, H_v, d_v]
  g     = -softplus(N(0,1))   (log alpha, one per key channel)      [B, T, H_v, d_k]
          decay variants (the whole domain alpha in [0, 1]):
            "strong": -softplus(N(3,1)) (about -3 per token, a 64-token chunk spans ~195)
            "bursts": the standard draw, plus runs of 8 tokens at g = -20 starting at each
                      (token, channel) with probability 1/8192 (about one run per 64 x 128
                      chunk, so chunks with and without a run alternate)
            "reset":  the standard draw, plus g = -inf (alpha = 0) at each (token, channel)
                      with probability 1/32 and on every channel of tokens t = 50 (mod 97)
  b     = sigmoid(N(0,1)); 2*sigmoid(N(0,1)) when negative
          eigenvalues are allowed (the "b x 2" option)              [B, T, H_v, d_k]
  w     = sigmoid(N(0,1))                                           [B, T, H_v, d_v]
  S0    ~ N(0, std^2), float32, or absent                           [B, H_v, d_k, d_v]

Values are drawn and transformed in float64, rounded to float32 (round to nearest even) and,
for bf16 workloads, rounded again to bfloat16 (round to nearest even). The stored bits are the
ground truth that both the GPU path and the oracle consume.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

_TENSOR_ID = {"q": 1, "k": 2, "v": 3, "g": 4, "b": 5, "w": 6, "s0": 7, "g_extra": 8}
DECAYS = ("standard", "strong", "bursts", "reset")


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, storage dtype and input distribution switches."""

    name: str
    B: int
    T: int  # tokens of the chunked forward (0 for a pure decode workload)
    Hk: int
    Hv: int
    dk: int
    dv: int
    C: int = 64
    dtype: str = "bf16"  # "f32" or "bf16": storage type of the token tensors and of o
    seed: int = 0
    s0_std: float = 0.0  # 0 => no initial state (zeros)
    neg_eigval: bool = False
    decode_steps: int = 0  # single-token steps after the chunked forward
    description: str = ""
    decay: str = "standard"  # distribution of g (see DECAYS and the module docstring)

    @property
    def tokens_total(self) -> int:
        return self.T + self.decode_steps

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads of the build contract, named by what they are.
WORKLOADS = {
    "tiny_f32": Workload(
        "tiny_f32", B=1, T=256, Hk=4, Hv=4, dk=64, dv=64, C=64, dtype="f32", seed=0,
        description="fp32 chunk forward, B=1 H=4 T=256 d=64 C=64, S0=0"),
    "train_bf16": Workload(
        "train_bf16", B=4, T=2048, Hk=8, Hv=8, dk=128, dv=128, C=64, dtype="bf16", seed=1,
        s0_std=0.02, description="bf16 chunk forward, B=4 H=8 T=2048 d=128 C=64, S0~N(0,0.02^2)"),
    "long_negeig_bf16": Workload(
        "long_negeig_bf16", B=1, T=8192, Hk=16, Hv=16, dk=128, dv=128, C=64, dtype="bf16",
        seed=2, neg_eigval=True,
        description="bf16 chunk forward, B=1 H=16 T=8192 d=128 C=64, b in (0,2), S0=0"),
    "decode_b64": Workload(
        "decode_b64", B=64, T=0, Hk=16, Hv=48, dk=128, dv=128, C=64, dtype="bf16", seed=3,
        s0_std=0.02, decode_steps=256,
        description="256 single-token steps, B=64 H_k=16 H_v=48 d=128, fp32 state ~N(0,0.02^2)"),
    "prefill32k_decode": Workload(
        "prefill32k_decode", B=2, T=32768, Hk=16, Hv=32, dk=128, dv=128, C=64, dtype="bf16",
        seed=4, decode_steps=64,
        description="bf16 chunk forward B=2 T=32768 H_k=16 H_v=32 d=128 C=64 from S0=0, "
                    "then 64 single-token steps from its final state"),
}


# ----------------------------------------------------------------------------------------------
# rounding helpers (storage formats only)

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16, nearest-even; returns the 16-bit patterns (uint16)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_to(x64: np.ndarray, dtype: str) -> np.ndarray:
    """float64 -> float32 (RNE) -> bfloat16 (RNE) when dtype == 'bf16'; returns float32 values."""
    x32 = x64.astype(np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f32(f32_to_bf16_bits(x32))
    if dtype == "f32":
        return x32
    raise ValueError(dtype)


# ----------------------------------------------------------------------------------------------
# slabs

def _rng(seed: int, name: str, bi: int, h: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _TENSOR_ID[name], bi, h])))


def _softplus(x):
    return np.logaddexp(0.0, x)


def _sigmoid(x):
    return 0.5 * (1.0 + np.tanh(0.5 * x))


def _decay_slab(x: np.ndarray, decay: str, seed: int, bi: int, h: int) -> np.ndarray:
    """g = log alpha from the standard-normal draw x [T, d] for one decay variant."""
    if decay == "strong":
        return -_softplus(x + 3.0)
    g = -_softplus(x)
    if decay == "standard":
        return g
    T, d = x.shape
    u = _rng(seed, "g_extra", bi, h).random((T, d))
    if decay == "bursts":
        start = u < 1.0 / 8192.0
        burst = np.zeros((T, d), bool)
        for s in range(8):
            burst[s:] |= start[:T - s]
        return np.where(burst, -20.0, g)
    if decay == "reset":
        g = np.where(u < 1.0 / 32.0, -np.inf, g)
        g[np.arange(T) % 97 == 50] = -np.inf
        return g
    raise ValueError(decay)


def slab(seed: int, name: str, bi: int, h: int, T: int, d: int, dtype: str,
         neg_eigval: bool = False, decay: str = "standard") -> np.ndarray:
    """One [T, d] slab of token tensor `name` for batch index bi and head h (float32 values)."""
    x = _rng(seed, name, bi, h).standard_normal((T, d))
    if name in ("q", "k"):
        nrm = np.sqrt(np.sum(x * x, axis=1, keepdims=True))
        x = x / np.where(nrm > 0, nrm, 1.0)
    elif name == "g":
        x = _decay_slab(x, decay, seed, bi, h)
    elif name == "b":
        x = _sigmoid(x) * (2.0 if neg_eigval else 1.0)
    elif name == "w":
        x = _sigmoid(x)
    elif name == "v":
        pass
    else:
        raise ValueError(name)
    return round_to(x, dtype)


def state_slab(seed: int, bi: int, h: int, dk: int, dv: int, std: float) -> np.ndarray:
    x = _rng(seed, "s0", bi, h).standard_normal((dk, dv)) * std
    return x.astype(np.float32)


@dataclass
class Inputs:
    """Token tensors (float32 arrays holding values exactly representable in `dtype`)."""

    dtype: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    b: np.ndarray
    w: np.ndarray
    s0: np.ndarray | None
    meta: dict = field(default_factory=dict)

    def bits(self, name: str) -> np.ndarray:
        """bfloat16 bit patterns (uint16) of tensor `name`; only for bf16 inputs."""
        assert self.dtype == "bf16"
        return f32_to_bf16_bits(getattr(self, name))

    def tokens(self, t0: int, t1: int) -> "Inputs":
        """Sub-sequence [t0, t1) of every token tensor (copies); s0 is kept."""
        sl = lambda a: np.ascontiguousarray(a[:, t0:t1])
        return Inputs(self.dtype, sl(self.q), sl(self.k), sl(self.v), sl(self.g), sl(self.b),
                      sl(self.w), self.s0, dict(self.meta))

    def heads(self, bi: int, hv: int, Hk: int, Hv: int) -> "Inputs":
        """Single-head problem (B=1, H_k=H_v=1) for value head hv of batch bi.

        The key head is chosen by the contiguous grouping h_k = hv // (H_v / H_k).
        """
        hk = hv // (Hv // Hk)
        one = lambda a, h: np.ascontiguousarray(a[bi:bi + 1, :, h:h + 1])
        s0 = None if self.s0 is None else np.ascontiguousarray(self.s0[bi:bi + 1, hv:hv + 1])
        return Inputs(self.dtype, one(self.q, hk), one(self.k, hk), one(self.v, hv),
                      one(self.g, hv), one(self.b, hv), one(self.w, hv), s0, dict(self.meta))


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def make_inputs(wl: Workload, T: int | None = None, dtype: str | None = None, b0: int = 0) -> Inputs:
    """All token tensors of workload `wl` for T tokens (default: chunk tokens + decode steps).

    b0 offsets the batch indices used for seeding, so that batch element i of the result is batch
    element b0 + i of a larger batch (how ranks of a multi-GPU run get disjoint sequences).
    """
    T = wl.tokens_total if T is None else T
    dtype = wl.dtype if dtype is None else dtype
    B, Hk, Hv, dk, dv = wl.B, wl.Hk, wl.Hv, wl.dk, wl.dv
    out = {
        "q": np.empty((B, T, Hk, dk), np.float32), "k": np.empty((B, T, Hk, dk), np.float32),
        "v": np.empty((B, T, Hv, dv), np.float32), "w": np.empty((B, T, Hv, dv), np.float32),
        "g": np.empty((B, T, Hv, dk), np.float32), "b": np.empty((B, T, Hv, dk), np.float32),
    }
    jobs = []
    for name, arr in out.items():
        H = arr.shape[2]
        d = arr.shape[3]
        for bi in range(B):
            for h in range(H):
                jobs.append((name, arr, bi, h, d))

    def run(job):
        name, arr, bi, h, d = job
        arr[bi, :, h, :] = slab(wl.seed, name, b0 + bi, h, T, d, dtype, wl.neg_eigval, wl.decay)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(run, jobs))
    s0 = None
    if wl.s0_std > 0:
        s0 = np.empty((B, Hv, dk, dv), np.float32)
        for bi in range(B):
            for h in range(Hv):
                s0[bi, h] = state_slab(wl.seed, b0 + bi, h, dk, dv, wl.s0_std)
    return Inputs(dtype, s0=s0, meta={"workload": wl.name, "T": T, "b0": b0}, **out)


def make_head_inputs(wl: Workload, bi: int, hv: int, T: int | None = None) -> Inputs:
    """The single-head problem of (bi, hv) without generating the other heads.

    Equal, bit for bit, to ``make_inputs(wl).heads(bi, hv, wl.Hk, wl.Hv)``.
    """
    T = wl.tokens_total if T is None else T
    hk = hv // (wl.Hv // wl.Hk)
    f = lambda name, h, d: slab(wl.seed, name, bi, h, T, d, wl.dtype, wl.neg_eigval, wl.decay)[None, :, None, :]
    s0 = None
    if wl.s0_std > 0:
        s0 = state_slab(wl.seed, bi, hv, wl.dk, wl.dv, wl.s0_std)[None, None]
    return Inputs(wl.dtype, f("q", hk, wl.dk), f("k", hk, wl.dk), f("v", hv, wl.dv),
                  f("g", hv, wl.dk), f("b", hv, wl.dk), f("w", hv, wl.dv), s0,
                  {"workload": wl.name, "T": T, "bi": bi, "hv": hv})


def sample_heads(wl: Workload, n: int, seed: int = 12345) -> list[tuple[int, int]]:
    """n distinct (batch, value head) pairs, always including the first and the last head."""
    units = [(bi, h) for bi in range(wl.B) for h in range(wl.Hv)]
    if n >= len(units):
        return units
    rng = np.random.default_rng(seed)
    pick = {units[0], units[-1]}
    while len(pick) < n:
        pick.add(units[int(rng.integers(len(units)))])
    return sorted(pick)


def to_torch(x: np.ndarray, dtype: str, device=None):
    """Upload float32 values as a torch tensor of the storage dtype (bit-exact)."""
    import torch

    if dtype == "bf16":
        t = torch.from_numpy(f32_to_bf16_bits(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(device) if device is not None else t
