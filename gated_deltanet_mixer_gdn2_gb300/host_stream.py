"""Chunked forward on token tensors that live in (pinned) host memory.

The sequence is cut into segments of whole chunks. Segment s + 1 is copied to the device while the
chunked forward runs on segment s, and the output of segment s - 1 is copied back meanwhile; the
state at the end of each segment is the initial state of the next (the recurrence chains exactly).
The host link is the bottleneck, so the first segments grow (512, 1024, ... tokens: a short upload
before the first kernel) and the last ones shrink the same way (a short compute and download after
the last upload). Every computation runs in libgdn2.so's kernels; this module only moves memory and
orders streams.
"""
from __future__ import annotations

import gated_deltanet_mixer_gdn2_gb300 as _g

_NAMES = ("q", "k", "v", "g", "b", "w")


def segment_plan(T, segment_tokens=4096, C=64):
    """Segment lengths (summing to T): a doubling ramp from 8 chunks up to segment_tokens, full
    segments, then the mirrored ramp down. Every length but possibly one in the middle is a
    multiple of C."""
    seg = max(C, (segment_tokens // C) * C)
    head = []
    s, used = max(C, min(seg, 8 * C)), 0
    while s < seg and T - used >= 2 * s:
        head.append(s)
        used += 2 * s
        s *= 2
    body = T - used
    mids = [seg] * (body // seg)
    if body % seg:
        mids.append(body % seg)
    return head + mids + head[::-1]


def chunk_fwd_from_host(q, k, v, g, b, w, o, initial_state=None, *, segment_tokens=4096, C=64, scale=1.0,
                        device=None, stream=None):
    """q, k: [B, T, H_k, d_k]; v, w, o: [B, T, H_v, d_v]; g, b: [B, T, H_v, d_k] -- pinned CPU tensors
    (o is written). initial_state: device fp32 [B, H_v, d_k, d_v] or None. Returns the final state
    (device). The work is queued on `stream` (default: the current stream) and two helper streams;
    `stream` waits for all of it, so the host may synchronise on it."""
    import torch

    device = device or torch.device("cuda", torch.cuda.current_device())
    main = stream or torch.cuda.current_stream(device)
    B, T, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    plan = segment_plan(T, segment_tokens, C)
    seg = max(plan) if plan else C
    starts = [sum(plan[:i]) for i in range(len(plan))]
    host = dict(zip(_NAMES, (q, k, v, g, b, w)))
    h2d, d2h = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    h2d.wait_stream(main)
    d2h.wait_stream(main)
    # flat per-slot storage; each segment uses a contiguous [B, n, H, d] view of it
    flat = [{n: torch.empty(B * seg * host[n].shape[2] * host[n].shape[3], dtype=host[n].dtype, device=device)
             for n in _NAMES} for _ in range(2)]
    oflat = [torch.empty(B * seg * Hv * dv, dtype=o.dtype, device=device) for _ in range(2)]

    def view(buf, n, shape):
        return buf[:B * n * shape[0] * shape[1]].view(B, n, shape[0], shape[1])

    loaded = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]
    state = initial_state
    ws = None

    def upload(i):
        t0, n, slot = starts[i], plan[i], i & 1
        with torch.cuda.stream(h2d):
            if i >= 2:
                h2d.wait_event(consumed[slot])        # the chunked forward of segment i-2 has read it
            for name in _NAMES:
                dst = view(flat[slot][name], n, host[name].shape[2:])
                for bi in range(B):
                    dst[bi].copy_(host[name][bi, t0:t0 + n], non_blocking=True)
            loaded[slot].record(h2d)

    if plan:
        upload(0)
    for i, t0 in enumerate(starts):
        n, slot = plan[i], i & 1
        if i + 1 < len(plan):
            upload(i + 1)
        main.wait_event(loaded[slot])
        if i >= 2:
            main.wait_event(drained[slot])            # o of segment i-2 has been copied out
        with torch.cuda.stream(main):
            d = [view(flat[slot][name], n, host[name].shape[2:]) for name in _NAMES]
            ob = view(oflat[slot], n, (Hv, dv))
            if ws is None:
                ws = torch.empty(max(16, _g.gdn2_chunk_fwd_workspace_size(B, seg, Hk, Hv, dk, dv, C)),
                                 dtype=torch.uint8, device=device)
            new_state = torch.empty((B, Hv, dk, dv), dtype=torch.float32, device=device)
            _g.gdn2_chunk_fwd(*d, ob, state, new_state, C=C, scale=scale, workspace=ws, stream=main)
            state = new_state
            consumed[slot].record(main)
            computed[slot].record(main)
        with torch.cuda.stream(d2h):
            d2h.wait_event(computed[slot])
            for bi in range(B):
                o[bi, t0:t0 + n].copy_(ob[bi], non_blocking=True)
            drained[slot].record(d2h)
    main.wait_stream(d2h)
    main.wait_stream(h2d)
    return state
