"""Benchmark of the Gated DeltaNet-2 core on GB300.

One step = the whole hot path once: the chunked forward (gdn2_chunk_fwd) over a 2 x 32768-token
prefill with 16 key / 32 value heads, d_k = d_v = 128, C = 64, from a zero state, then 64
single-token decode steps (gdn2_recurrent_step) from its final state. Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun (one process per GPU); every rank runs its own copy of the workload
(independent sequences: weak scaling, no data-path collective); rank 0 prints. `--impl reference`
times the fp64 CPU oracle on a bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "chunk-fwd tokens/s & % bf16 TC peak; decode step GB/s vs HBM peak (1×GB300)"
WORKLOAD = "prefill32k_decode"
DECODE_WORKLOAD = "decode_b64"
FLUSH_BYTES = 256 << 20  # > 129 MB L2


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one gdn2_chunk_fwd on this
# workload: a single-pass ncu capture of factors_tc + factors_exact + state_tc on the same heads at a
# quarter of the tokens (B 2, T 8192: 8192 units, inputs and workspace 1.2 GB >> L2), times 4 (the
# traffic grows with the units; the ~0.1 GB that stays in L2 across a kernel boundary is not
# counted). Reported only while the tensor-core forward's source is the one that was measured.
TRAFFIC_RECORD = {"chunk_tc_sha256_16": "63a4b2b168aa7d99", "bytes": 4 * (1837580288)}


def chunk_tc_source_sha() -> str:
    """First 16 hex digits of the sha256 of the tensor-core forward's sources (kernels and shared helpers)."""
    import hashlib

    h = hashlib.sha256()
    for name in ("chunk_tc.cu", "tc_common.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "gated_deltanet_mixer_gdn2_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    try:
        sha = chunk_tc_source_sha()
    except OSError:
        return None
    return TRAFFIC_RECORD["bytes"] if sha == TRAFFIC_RECORD["chunk_tc_sha256_16"] else None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---- algorithmic work --------------------------------------------------------------------------

def chunk_bytes(wl) -> int:
    """Bytes the chunked forward must move: every token input once, o once, the final state once."""
    tok = wl.B * wl.T
    per_tok = 2 * wl.Hk * wl.dk * 2 + wl.Hv * (2 * wl.dk + 2 * wl.dv) * 2 + wl.Hv * wl.dv * 2
    return tok * per_tok + wl.B * wl.Hv * wl.dk * wl.dv * 4 * (2 if wl.s0_std > 0 else 1)


def chunk_flops(wl) -> int:
    """Triangle-aware flops of the chunked form per (head, token): C(3 d_k + 2 d_v) + 6 d_k d_v."""
    return wl.B * wl.T * wl.Hv * (wl.C * (3 * wl.dk + 2 * wl.dv) + 6 * wl.dk * wl.dv)


def backward_flops(tokens: int, Hv: int, d: int) -> int:
    """Flops the backward is counted at: the recurrent form's forward (4 d^2 FMA) and backward (9 d^2 FMA)
    per token and value head, 2 flops per FMA."""
    return 26 * d * d * tokens * Hv


def decode_step_bytes(B, Hk, Hv, dk, dv) -> int:
    """State read + write, token inputs, output; bf16 tokens, fp32 state."""
    return 2 * B * Hv * dk * dv * 4 + B * (2 * Hk * dk + Hv * (2 * dk + 2 * dv)) * 2 + B * Hv * dv * 2


# ---- multi-GPU host logic (replicas over disjoint sequences; timing reduce only) ------------------

def rank_batch_offset(rank: int, batch_per_rank: int) -> int:
    """First global batch index of this rank: rank r runs sequences [r*B, (r+1)*B)."""
    return rank * batch_per_rank


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of `value` over ranks (the slowest rank times the job); identity for one process."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms_max * 1e-3)


# ---- clocks ------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            if self.uuid and parts[1] != self.uuid:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
            except Exception:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = [r for r in rows if self.t0 is not None and self.t0 - 1 <= r[0] <= self.t1 + 1] or rows
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for name, val in zip(names[1:], r[3][1:]):
                if val.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


# ---- our implementation -------------------------------------------------------------------------

def run_ours(args, rank, world, device):
    import torch

    import gated_deltanet_mixer_gdn2_gb300 as g

    hbm, tc_burst, tc_sust, peak_kind = peaks()
    wl = synth.WORKLOADS[WORKLOAD]
    # each rank runs its own B sequences (disjoint global batch indices)
    inp = synth.make_inputs(wl, b0=rank_batch_offset(rank, wl.B))
    T, D = wl.T, wl.decode_steps
    host = {n: synth.to_torch(np.ascontiguousarray(getattr(inp, n)), "bf16").pin_memory()
            for n in ("q", "k", "v", "g", "b", "w")}
    dev = {n: t.to(device) for n, t in host.items()}
    pre = {n: dev[n][:, :T].contiguous() for n in dev}
    dec = [{n: dev[n][:, t].contiguous() for n in dev} for t in range(T, T + D)]
    del dev
    B, Hk, Hv, dk, dv = wl.B, wl.Hk, wl.Hv, wl.dk, wl.dv
    o = torch.empty((B, T, Hv, dv), dtype=torch.bfloat16, device=device)
    od = torch.empty((D, B, Hv, dv), dtype=torch.bfloat16, device=device)
    state = torch.empty((B, Hv, dk, dv), dtype=torch.float32, device=device)
    ws_bytes = g.gdn2_chunk_fwd_workspace_size(B, T, Hk, Hv, dk, dv, wl.C, g.GDN2_BF16)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def decode_steps():
        for i in range(D):
            d = dec[i]
            g.gdn2_recurrent_step(d["q"], d["k"], d["v"], d["g"], d["b"], d["w"], state, od[i])

    # the D single-token launches are a launch-bound loop: captured once in a CUDA graph, replayed every
    # step (the same kernels on the same buffers, without the host's per-launch cost)
    side = torch.cuda.Stream(device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        decode_steps()  # warm-up outside the capture
    stream.wait_stream(side)
    torch.cuda.synchronize(device)
    dec_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dec_graph):
        decode_steps()
    torch.cuda.synchronize(device)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        g.gdn2_chunk_fwd(pre["q"], pre["k"], pre["v"], pre["g"], pre["b"], pre["w"], o, None, state, C=wl.C,
                         workspace=ws)
        if ev:
            ev[1].record(stream)
        dec_graph.replay()
        if ev:
            ev[2].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(device)
    assert g.gdn2_last_device_status() == g.GDN2_OK

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    clk = ClockSampler(uuid)
    clk.start()
    time.sleep(0.3)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(device)
    clk.mark("t0")
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()                          # L2 flush between steps, outside the events
        step(events[i])
    torch.cuda.synchronize(device)
    wall1 = time.perf_counter()
    clk.mark("t1")
    if world > 1:
        dist.barrier()
    clocks = clk.stop()
    status = g.gdn2_last_device_status()
    chunk_ms = [e[0].elapsed_time(e[1]) for e in events]
    dec_ms = [e[1].elapsed_time(e[2]) for e in events]
    step_ms = [a + b for a, b in zip(chunk_ms, dec_ms)]
    ms_per_step = reduce_max(sum(step_ms) / len(step_ms), world, device)
    tokens = B * T + B * D
    value = job_throughput(tokens, world, ms_per_step)

    # roofline of the dominant operation: the chunked forward (factors + state kernels)
    ch_ms = statistics.mean(chunk_ms)
    cb = chunk_bytes(wl)
    ach_gbs = cb / (ch_ms * 1e-3) / 1e9
    flops = chunk_flops(wl)
    ach_tf = flops / (ch_ms * 1e-3) / 1e12
    dstep_b = decode_step_bytes(B, Hk, Hv, dk, dv)
    d_ms = statistics.mean(dec_ms) / D

    decode_line = decode_roofline(g, device, hbm) if rank == 0 and not args.no_decode_workload else None
    next_rows = next_rows_rooflines(g, device, hbm, wl) if rank == 0 and not args.no_decode_workload else None
    head_shapes = head_shape_rooflines(g, device, hbm) if rank == 0 and not args.no_decode_workload else None

    # end to end through the public API with host buffers (inputs H2D, results D2H every step)
    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(g, wl, host, device, args, tokens)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: {wl.description}", "B": B, "T": T, "H_k": Hk, "H_v": Hv,
                   "d_k": dk, "d_v": dv, "chunk": wl.C, "decode_steps": D, "tokens_per_step": tokens,
                   "l2": "flushed between steps (256 MB write); prefill inputs 2.7 GB > L2",
                   "decode_launch": "the 64 single-token launches replayed from one CUDA graph",
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU"},
        "roofline": {"kernel": "gdn2_chunk_fwd (factors_tc + factors_exact + state_tc)", "bound": "hbm",
                     "achieved": round(ach_gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(ach_gbs / hbm, 4), "traffic": recorded_traffic(),
                     "algorithmic_bytes": cb, "ms": round(ch_ms, 4), "peak_kind": f"{peak_kind} hbm_gbs",
                     "tflops": round(ach_tf, 1), "tc_frac": round(ach_tf / tc_burst, 4),
                     "tc_peak": tc_burst, "flops": flops,
                     # the tensor-core fraction the call would reach at the HBM roof: these flops over
                     # the time its algorithmic bytes take at the measured copy bandwidth
                     "tc_frac_at_hbm_roof": round(flops / (cb / (hbm * 1e9)) / (tc_burst * 1e12), 4)},
        "decode_in_step": {"us_per_step": round(d_ms * 1e3, 2), "bytes_per_step": dstep_b,
                           "GB/s": round(dstep_b / (d_ms * 1e-3) / 1e9, 1),
                           "note": "4.2 MB state, L2-resident across steps"},
        "gpu_launches": args.steps * (3 + D),  # factors_tc, factors_exact, state_tc and the decode steps
        "clocks": clocks,
        "status": g.status_string(status),
        "wall_s_timed": round(wall1 - wall0, 3),
    }
    if decode_line:
        line["decode"] = decode_line
    if next_rows:
        line["next_rows"] = next_rows
    if head_shapes:
        line["head_shapes"] = head_shapes
    if e2e:
        line["e2e"] = e2e
    return line


def decode_roofline(g, device, hbm):
    """The decode kernel alone on the 64-sequence / 48-value-head workload (201 MB state)."""
    import torch

    wl = synth.WORKLOADS[DECODE_WORKLOAD]
    B, Hk, Hv, dk, dv = wl.B, wl.Hk, wl.Hv, wl.dk, wl.dv
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed)
    steps = wl.decode_steps
    st = torch.randn((B, Hv, dk, dv), generator=gen, device=device) * wl.s0_std
    toks = []
    for name, H, d in (("q", Hk, dk), ("k", Hk, dk), ("v", Hv, dv), ("g", Hv, dk), ("b", Hv, dk), ("w", Hv, dv)):
        x = torch.randn((steps, B, H, d), generator=gen, device=device, dtype=torch.float32)
        if name in ("q", "k"):
            x = x / x.norm(dim=-1, keepdim=True)
        elif name == "g":
            x = -torch.nn.functional.softplus(x)
        elif name in ("b", "w"):
            x = torch.sigmoid(x)
        toks.append(x.to(torch.bfloat16))
    o = torch.empty((steps, B, Hv, dv), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream(device)

    def run_all():
        for t in range(steps):
            g.gdn2_recurrent_step(toks[0][t], toks[1][t], toks[2][t], toks[3][t], toks[4][t], toks[5][t], st, o[t])

    for _ in range(3):
        run_all()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 3
    e0.record(stream)
    for _ in range(reps):
        run_all()
    e1.record(stream)
    torch.cuda.synchronize(device)
    us = e0.elapsed_time(e1) * 1e3 / (reps * steps)
    b = decode_step_bytes(B, Hk, Hv, dk, dv)
    gbs = b / (us * 1e-6) / 1e9
    return {"workload": f"{DECODE_WORKLOAD}: {wl.description}", "kernel": "recurrent_stream_kernel (gdn2_recurrent_step)",
            "us_per_step": round(us, 2), "bytes_per_step": b, "achieved": round(gbs, 1), "peak": hbm,
            "unit": "GB/s", "frac": round(gbs / hbm, 4), "bound": "hbm",
            "l2": "state 201 MB > L2; 256 back-to-back steps"}


def head_shape_rooflines(g, device, hbm):
    """The chunked forward on the pages' other head shapes (head_dim 64; expand_v = 2 at head_dim 128),
    bf16, 2 x 16384 tokens, 16 key / 32 value heads, each against the HBM roof of its algorithmic bytes
    (chunk_bytes); inputs > L2, CUDA events over back-to-back calls."""
    import torch

    B, T, Hk, Hv = 2, 16384, 16, 32
    bf = torch.bfloat16
    gen = torch.Generator(device=device)
    gen.manual_seed(77)
    rnd = lambda *s: torch.randn(s, generator=gen, device=device)
    stream = torch.cuda.current_stream(device)
    res = []
    for dk, dv in ((64, 64), (64, 128), (128, 256)):
        q = torch.nn.functional.normalize(rnd(B, T, Hk, dk), dim=-1).to(bf)
        k = torch.nn.functional.normalize(rnd(B, T, Hk, dk), dim=-1).to(bf)
        v, w = rnd(B, T, Hv, dv).to(bf), torch.sigmoid(rnd(B, T, Hv, dv)).to(bf)
        gg = (-torch.nn.functional.softplus(rnd(B, T, Hv, dk))).to(bf)
        bb = torch.sigmoid(rnd(B, T, Hv, dk)).to(bf)
        o = torch.empty_like(v)
        sT = torch.empty((B, Hv, dk, dv), dtype=torch.float32, device=device)
        ws = torch.empty(g.gdn2_chunk_fwd_workspace_size(B, T, Hk, Hv, dk, dv, 64), dtype=torch.uint8, device=device)
        fn = lambda: g.gdn2_chunk_fwd(q, k, v, gg, bb, w, o, None, sT, C=64, workspace=ws)
        for _ in range(3):
            fn()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(device)
        ms = e0.elapsed_time(e1) / reps
        nbytes = chunk_bytes(synth.Workload("head-shape", B=B, T=T, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype="bf16",
                                            seed=0, s0_std=0.0))
        gbs = nbytes / (ms * 1e-3) / 1e9
        res.append({"shape": f"d_k {dk}, d_v {dv}", "path": "tcgen05", "ms": round(ms, 4),
                    "algorithmic_bytes": int(nbytes), "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(gbs / hbm, 4)})
        del q, k, v, w, gg, bb, o, sT, ws
    return {"workload": f"B={B} T={T} H_k={Hk} H_v={Hv} bf16, chunk 64, from S0 = 0", "shapes": res}


def next_rows_rooflines(g, device, hbm, wl):
    """The widened rows on the bench workload's shapes, each HBM-bound: the fused mixer prologue and
    epilogue, and the FG^2-GDN input transform. Algorithmic bytes = every tensor read once and
    written once; inputs are GBs (> L2), timed with CUDA events over back-to-back calls."""
    import torch

    B, T, Hk, Hv, d = wl.B, wl.T, wl.Hk, wl.Hv, wl.dk
    bf = torch.bfloat16
    gen = torch.Generator(device=device)
    gen.manual_seed(1234)
    rnd = lambda *s: torch.randn(s, generator=gen, device=device).to(bf)
    xq, xk, xv = rnd(B, T, Hk, d), rnd(B, T, Hk, d), rnd(B, T, Hv, d)
    ag, ab, aw = rnd(B, T, Hv, d), rnd(B, T, Hv, d), rnd(B, T, Hv, d)
    cw = [torch.randn((n, 4), generator=gen, device=device) * 0.5 for n in (Hk * d, Hk * d, Hv * d)]
    states = [torch.zeros((B, 3, n), device=device) for n in (Hk * d, Hk * d, Hv * d)]
    outs = [torch.empty_like(t) for t in (xq, xk, xv, ag, ab, aw)]
    z, o = rnd(B, T, Hv, d), rnd(B, T, Hv, d)
    wt = torch.ones(d, device=device)
    y = torch.empty_like(o)
    f_outs = [torch.empty((B, T, Hv, d), dtype=bf, device=device) for _ in range(4)]
    stream = torch.cuda.current_stream(device)
    tok = B * T
    e = 2  # bytes per bf16 element
    calls = {
        "mixer_prologue": (lambda: g.gdn2_mixer_prologue(xq, xk, xv, *cw, ag, ab, aw, *outs, states=states),
                           2 * tok * (2 * Hk * d + 4 * Hv * d) * e + sum(c.numel() for c in cw) * 4
                           + 2 * sum(s_.numel() for s_ in states) * 4,
                           "gdn2_mixer_prologue (conv_tile_kernel + gates_kernel + conv_state_kernel)"),
        "mixer_epilogue": (lambda: g.gdn2_mixer_epilogue(o, z, wt, y), 3 * tok * Hv * d * e + d * 4,
                           "gdn2_mixer_epilogue (epilogue_kernel)"),
        "fg2_inputs": (lambda: g.gdn2_fg2_inputs(xq, xk, ag, *f_outs), (2 * Hk + 5 * Hv) * tok * d * e,
                       "gdn2_fg2_inputs (fg2_inputs_kernel)"),
    }
    res = {}
    for name, (fn, nbytes, kernel) in calls.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(device)
        ms = e0.elapsed_time(e1) / reps
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"kernel": kernel, "ms": round(ms, 4), "algorithmic_bytes": int(nbytes),
                     "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                     "bound": "hbm"}
    # backward (bf16: chunked WY form on the tensor cores, 64-token chunks)
    tk = [rnd(B, T, Hk, d), rnd(B, T, Hk, d)]
    tk[0] = (tk[0].float() / tk[0].float().norm(dim=-1, keepdim=True)).to(bf)
    tk[1] = (tk[1].float() / tk[1].float().norm(dim=-1, keepdim=True)).to(bf)
    vv, do_ = rnd(B, T, Hv, d), rnd(B, T, Hv, d)
    gg = (-torch.nn.functional.softplus(torch.randn((B, T, Hv, d), generator=gen, device=device))).to(bf)
    bb = torch.sigmoid(torch.randn((B, T, Hv, d), generator=gen, device=device)).to(bf)
    ww = torch.sigmoid(torch.randn((B, T, Hv, d), generator=gen, device=device)).to(bf)
    grads = [torch.empty_like(t) for t in (tk[0], tk[1], vv, gg, bb, ww)]
    wsb = g.lib.gdn2_backward_workspace_size(B, T, Hk, Hv, d, d, g.GDN2_BF16)
    ws = torch.empty(wsb, dtype=torch.uint8, device=device)
    fn = lambda: g.gdn2_backward(tk[0], tk[1], vv, gg, bb, ww, do_, *grads, workspace=ws)
    fn()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(2):
        fn()
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / 2
    flops = backward_flops(tok, Hv, d)
    _, tc_peak, _, pk_kind = peaks()
    ach = flops / (ms * 1e-3) / 1e12
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    res["backward"] = {"kernel": "gdn2_backward (factors_tc_kernel + state_tc_kernel keeping S_n and U_n + "
                                 "rchain_tc_kernel + grad_tc_kernel + group_sum_tc_kernel)", "ms": round(ms, 3),
                       "algorithmic_flops": int(flops), "achieved": round(ach, 2), "peak": round(tc_peak, 1),
                       "peak_kind": pk_kind, "unit": "TFLOP/s", "frac": round(ach / tc_peak, 4), "bound": "latency",
                       "note": (f"flops counted at the recurrent form's 26 d^2 per (token, head); every product runs "
                                f"on tcgen05, but the per-chunk gradient kernel (one CTA per (chunk, head), all of "
                                f"shared memory and tensor memory) is a chain of dependent products and read-outs, "
                                f"and the two chains over chunks use {min(2 * B * Hv, sms)} of {sms} SMs")}
    res["shape"] = f"B={B} T={T} H_k={Hk} H_v={Hv} d={d} bf16 (the bench workload's token tensors)"
    return res


def run_variants(device):
    """Serving decode variants (gdn2_recurrent_update) on the 64-sequence, 48-value-head decode shape:
    one JSON line each, with the kernel's algorithmic bytes per call against measured HBM bandwidth."""
    import torch

    import gated_deltanet_mixer_gdn2_gb300 as g

    hbm, _, _, peak_kind = peaks()
    wl = synth.WORKLOADS[DECODE_WORKLOAD]
    B, Hk, Hv, dk, dv = wl.B, wl.Hk, wl.Hv, wl.dk, wl.dv
    gen = torch.Generator(device=device)
    gen.manual_seed(7)

    def tokens(N):
        out = []
        for name, H, d in (("q", Hk, dk), ("k", Hk, dk), ("v", Hv, dv), ("g", Hv, dk), ("b", Hv, dk), ("w", Hv, dv)):
            x = torch.randn((B, N, H, d), generator=gen, device=device)
            if name in ("q", "k"):
                x = x / x.norm(dim=-1, keepdim=True)
            elif name == "g":
                x = -torch.nn.functional.softplus(x)
            elif name in ("b", "w"):
                x = torch.sigmoid(x)
            out.append(x.to(torch.bfloat16))
        return out

    cases = [
        ("fp32 state, 1 token per call", 1, torch.float32, False),
        ("fp32 state, 4 tokens per call", 4, torch.float32, False),
        ("bf16 state, 1 token per call", 1, torch.bfloat16, False),
        ("bf16 state, 4 tokens per call", 4, torch.bfloat16, False),
        ("fp32 state pool, permuted slot map, 1 token per call", 1, torch.float32, True),
    ]
    stream = torch.cuda.current_stream(device)
    for name, N, sdt, use_slots in cases:
        n_slots = B + 8 if use_slots else B
        st = (torch.randn((n_slots, Hv, dk, dv), generator=gen, device=device) * 0.02).to(sdt)
        slots = torch.randperm(n_slots, generator=gen, device=device)[:B].to(torch.int32) if use_slots else None
        tk = tokens(N)
        o = torch.empty((B, N, Hv, dv), dtype=torch.bfloat16, device=device)
        for _ in range(3):
            g.gdn2_recurrent_update(*tk, st, o, slots)
        torch.cuda.synchronize(device)
        reps = 100
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.gdn2_recurrent_update(*tk, st, o, slots)
        e1.record(stream)
        torch.cuda.synchronize(device)
        us = e0.elapsed_time(e1) * 1e3 / reps
        sbytes = 2 * B * Hv * dk * dv * st.element_size()
        tbytes = N * (B * (2 * Hk * dk + Hv * (2 * dk + 2 * dv)) * 2 + B * Hv * dv * 2)
        b = sbytes + tbytes + (B * 4 if use_slots else 0)
        gbs = b / (us * 1e-6) / 1e9
        print(json.dumps({"variant": name, "workload": f"{DECODE_WORKLOAD} shape: B={B} H_k={Hk} H_v={Hv} d={dk}",
                          "us_per_call": round(us, 2), "tokens_per_s": round(B * N / (us * 1e-6), 1),
                          "bytes_per_call": b, "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                          "frac": round(gbs / hbm, 4), "peak_kind": f"{peak_kind} hbm_gbs",
                          "l2": "state >= 100 MB > L2; 100 back-to-back calls"}), flush=True)
    run_mixer_step_variants(device, hbm, peak_kind)


def run_mixer_step_variants(device, hbm, peak_kind):
    """The whole mixer around the core for one decode token: gdn2_mixer_decode_step (one launch) against
    gdn2_mixer_prologue + gdn2_recurrent_step + gdn2_mixer_epilogue (five launches), at the decode
    workload's batch and at batch 1; 100 back-to-back calls of each."""
    import torch

    import gated_deltanet_mixer_gdn2_gb300 as g

    wl = synth.WORKLOADS[DECODE_WORKLOAD]
    Hk, Hv, d = wl.Hk, wl.Hv, wl.dk
    gen = torch.Generator(device=device)
    gen.manual_seed(11)
    bf = torch.bfloat16
    for B in (wl.B, 1):
        rn = lambda *s: torch.randn(s, generator=gen, device=device)
        xq, xk, xv = rn(B, 1, Hk, d).to(bf), rn(B, 1, Hk, d).to(bf), rn(B, 1, Hv, d).to(bf)
        ag, ab, aw, z = rn(B, 1, Hv, d).to(bf), rn(B, 1, Hv, d).to(bf), rn(B, 1, Hv, d).to(bf), rn(B, Hv, d).to(bf)
        cw = [0.5 * rn(n, 4) for n in (Hk * d, Hk * d, Hv * d)]
        cs = [rn(B, 3, n) for n in (Hk * d, Hk * d, Hv * d)]
        st = 0.02 * rn(B, Hv, d, d)
        wt = torch.ones(d, device=device)
        y = torch.empty((B, Hv, d), dtype=bf, device=device)
        outs = [torch.empty_like(t) for t in (xq, xk, xv, ag, ab, aw)]
        o = torch.empty((B, Hv, d), dtype=bf, device=device)

        def fused():
            g.gdn2_mixer_decode_step(xq[:, 0], xk[:, 0], xv[:, 0], *cw, ag[:, 0], ab[:, 0], aw[:, 0], st, z, wt, y,
                                     states=cs)

        def separate():
            g.gdn2_mixer_prologue(xq, xk, xv, *cw, ag, ab, aw, *outs, states=cs)
            g.gdn2_recurrent_step(*(t[:, 0] for t in outs), st, o)
            g.gdn2_mixer_epilogue(o[:, None], z[:, None], wt, y[:, None])

        stream = torch.cuda.current_stream(device)
        res = {}
        for name, fn in (("fused", fused), ("separate", separate)):
            for _ in range(3):
                fn()
            torch.cuda.synchronize(device)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(100):
                fn()
            e1.record(stream)
            torch.cuda.synchronize(device)
            res[name] = e0.elapsed_time(e1) * 1e3 / 100
        # bytes of the fused step: core state read + written, conv states read + written, the token's
        # vectors in and y out, the conv weights
        b = (2 * B * Hv * d * d * 4 + 2 * B * 3 * (2 * Hk + Hv) * d * 4 + B * (2 * Hk + 5 * Hv) * d * 2
             + (2 * Hk + Hv) * d * 16 + d * 4)
        gbs = b / (res["fused"] * 1e-6) / 1e9
        print(json.dumps({"variant": f"mixer decode step (conv + L2 norm + gates + core + gated RMSNorm), B={B}",
                          "workload": f"{DECODE_WORKLOAD} heads: H_k={Hk} H_v={Hv} d={d}, bf16 tokens, fp32 state",
                          "us_per_call_fused": round(res["fused"], 2), "launches_fused": 1,
                          "us_per_call_separate": round(res["separate"], 2), "launches_separate": 5,
                          "bytes_per_call": b, "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                          "frac": round(gbs / hbm, 4), "peak_kind": f"{peak_kind} hbm_gbs",
                          "l2": "100 back-to-back calls"}), flush=True)


def end_to_end(g, wl, host, device, args, tokens):
    """Same step through the public API with host (pinned) buffers: inputs copied in, o copied out."""
    import torch

    T, D = wl.T, wl.decode_steps
    B, Hv, dv = wl.B, wl.Hv, wl.dv
    hpre = {n: host[n][:, :T].contiguous().pin_memory() for n in host}
    hdec = {n: host[n][:, T:T + D].transpose(0, 1).contiguous().pin_memory() for n in host}  # [D, B, H, d]
    o_h = torch.empty((B, T, Hv, dv), dtype=torch.bfloat16).pin_memory()
    od_h = torch.empty((B, D, Hv, dv), dtype=torch.bfloat16).pin_memory()
    stream = torch.cuda.current_stream(device)
    h2d = sum(t.numel() * t.element_size() for t in hpre.values()) + sum(
        t.numel() * t.element_size() for t in hdec.values())
    d2h = o_h.numel() * 2 + od_h.numel() * 2

    from gated_deltanet_mixer_gdn2_gb300.host_stream import chunk_fwd_from_host

    def step():
        # prefill streamed in segments (uploads, kernels and downloads overlap), then the decode tokens
        st = chunk_fwd_from_host(*(hpre[n] for n in ("q", "k", "v", "g", "b", "w")), o_h, None, C=wl.C, segment_tokens=4096,
                                 device=device, stream=stream)
        dd = {n: t.to(device, non_blocking=True) for n, t in hdec.items()}
        outs = []
        for i in range(D):
            outs.append(g.recurrent_step(*(dd[n][i] for n in ("q", "k", "v", "g", "b", "w")), st))
        od_h.copy_(torch.stack(outs, dim=1), non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize(device)
    n = max(2, min(args.steps, 5))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / n
    return {"value": round(tokens / (ms * 1e-3), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms, 3), "steps": n}


# ---- CPU baseline (the fp64 oracle) --------------------------------------------------------------

def cpu_sample():
    """Time the oracle on one full sequence of the bench workload: its 32768-token prefill and 64
    decode tokens, all 32 value heads (one half of a bench step). Returns (tokens/s, description,
    threads, seconds)."""
    import oracle

    wl = synth.WORKLOADS[WORKLOAD]
    nth = min(oracle.default_threads(), wl.Hv)
    inp = synth.make_inputs(wl.with_(B=1))
    t0 = time.perf_counter()
    oracle.run_inputs(inp, nthreads=nth)
    dt = time.perf_counter() - t0
    Ts = wl.tokens_total
    return Ts / dt, (f"1 of the {wl.B} sequences of {WORKLOAD}: {wl.T}-token prefill + {wl.decode_steps} "
                     f"decode tokens, {wl.Hv} value heads (fp64 recurrent form)"), nth, dt


def run_reference(args):
    import oracle  # noqa: F401

    wl = synth.WORKLOADS[WORKLOAD]
    nth = min(os.cpu_count() or 1, wl.Hv)
    Ts = 256
    inp = synth.make_inputs(wl.with_(B=1), T=Ts)
    import oracle as orc
    for _ in range(args.warmup):
        orc.run_inputs(inp, nthreads=nth)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        orc.run_inputs(inp, nthreads=nth)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = Ts / (ms * 1e-3)
    sample = f"each step: 1 sequence x {wl.Hv} value heads x {Ts} tokens of {WORKLOAD} (fp64 recurrent form)"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: {wl.description}"},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": nth, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_profile(spec: str):
    """One operation of one workload, twice (the second call is the one to capture with ncu -s 1).
    spec: 'chunk:<workload>[:T]', 'decode:<workload>', 'update:<workload>:<N>[:bf16]' (gdn2_recurrent_update,
    N tokens per call, fp32 or bf16 state), 'step:<workload>' (gdn2_mixer_decode_step on that workload's
    heads, bf16 tokens) or 'next:<workload>' (prologue, epilogue, FG2 transform, backward on that
    workload's shapes); T overrides the workload's token count (a smaller case of the same heads for
    captures beyond the one-pass launch list)."""
    import torch

    import gated_deltanet_mixer_gdn2_gb300 as g

    parts = spec.split(":")
    op, name = parts[0], parts[1]
    wl = synth.WORKLOADS[name]
    if len(parts) > 2:
        wl = wl.with_(T=int(parts[2]))
    device = torch.device("cuda", 0)
    if op == "chunk":
        inp = synth.make_inputs(wl, T=wl.T)
        q, k, v, gg, b, w = (synth.to_torch(np.ascontiguousarray(getattr(inp, n)), wl.dtype, device)
                             for n in ("q", "k", "v", "g", "b", "w"))
        s0 = None if inp.s0 is None else torch.from_numpy(inp.s0).to(device)
        for _ in range(2):
            g.chunk_fwd(q, k, v, gg, b, w, s0, C=wl.C)
    elif op == "next":
        # the widened rows on the given workload's token shapes (one call each after a warm-up call)
        from types import SimpleNamespace

        hbm = peaks()[0]
        res = next_rows_rooflines(g, device, hbm, SimpleNamespace(B=wl.B, T=wl.T, Hk=wl.Hk, Hv=wl.Hv, dk=wl.dk))
        print(json.dumps({k: (v["ms"] if isinstance(v, dict) else v) for k, v in res.items()}))
    elif op == "update":
        inp = synth.make_inputs(wl, T=wl.T)
        sdt = torch.bfloat16 if len(parts) > 3 and parts[3] == "bf16" else torch.float32
        st = torch.from_numpy(inp.s0).to(device).to(sdt)
        tok = [synth.to_torch(np.ascontiguousarray(getattr(inp, n)), wl.dtype, device)
               for n in ("q", "k", "v", "g", "b", "w")]
        o = torch.empty_like(tok[2])
        for _ in range(2):
            g.gdn2_recurrent_update(*tok, st, o)
    elif op == "step":
        gen = torch.Generator(device=device)
        gen.manual_seed(11)
        rn = lambda *s: torch.randn(s, generator=gen, device=device)
        bf = torch.bfloat16
        B, Hk, Hv, d = wl.B, wl.Hk, wl.Hv, wl.dk
        xq, xk, xv = rn(B, Hk, d).to(bf), rn(B, Hk, d).to(bf), rn(B, Hv, d).to(bf)
        ag, ab, aw, z = (rn(B, Hv, d).to(bf) for _ in range(4))
        cw = [0.5 * rn(n, 4) for n in (Hk * d, Hk * d, Hv * d)]
        cs = [rn(B, 3, n) for n in (Hk * d, Hk * d, Hv * d)]
        st = 0.02 * rn(B, Hv, d, d)
        y = torch.empty((B, Hv, d), dtype=bf, device=device)
        for _ in range(2):
            g.gdn2_mixer_decode_step(xq, xk, xv, *cw, ag, ab, aw, st, z, torch.ones(d, device=device), y, states=cs)
    elif op == "decode":
        inp = synth.make_inputs(wl, T=2)
        st = torch.from_numpy(inp.s0).to(device)
        for t in range(2):
            tok = [synth.to_torch(np.ascontiguousarray(getattr(inp, n)[:, t]), wl.dtype, device)
                   for n in ("q", "k", "v", "g", "b", "w")]
            g.recurrent_step(*tok, st)
    else:
        raise SystemExit(f"unknown op {op}")
    torch.cuda.synchronize()
    status = g.gdn2_last_device_status()
    print(json.dumps({"profile": spec, "status": g.status_string(status)}))
    if status != g.GDN2_OK:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile", default=None, help="op:workload, e.g. chunk:long_negeig_bf16 (for ncu)")
    ap.add_argument("--variants", action="store_true", help="measure the serving decode variants instead")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-decode-workload", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.profile:
        run_profile(args.profile)
        return
    if args.variants:
        import torch

        run_variants(torch.device("cuda", 0))
        return
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    # the oracle's CPU baseline runs before any GPU work of this process touches a thread pool
    cpu = None
    if rank == 0 and not args.no_cpu:
        tps, sample, cores, secs = cpu_sample()
        cpu = {"value": round(tps, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
               "seconds": round(secs, 2)}
    line = run_ours(args, rank, world, device)
    if cpu:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
