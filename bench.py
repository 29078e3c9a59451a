#!/usr/bin/env python
"""Benchmark of the KDA recurrent-state serving path on one GB300 (or N replicas).

One step = one pass of every entry point over one batch of synthetic input:
  * kda_chunk_prefill    : 8 packed sequences, lengths ~U[1024, 8192] (seed 1), H=32,
                           d=128, chunk 64, bf16 in/out, fp32 state pool (64 slots,
                           in-place init/final) and one fp32 snapshot per sequence.
  * kda_recurrent_decode : 256 requests x 1 token, H=32, 1024-slot fp32 pool.
  * kda_spec_verify + kda_spec_accept_commit : 64 requests, K=7, H=32; each
                           draft agrees with the sampled token with probability
                           0.7; the commit launch derives the accepted lengths
                           from the token ids, rebuilds the states in place and
                           moves the q / k / v short-convolution windows of the
                           same requests (4096 bf16 channels each, keep 3).
  * kda_slot_copy        : 256 parents x 8 children + 512 clears, 4096-slot pool
                           of 1 MiB fp32 states (H=16).
`value` is the prefill throughput in tokens/s (device time of the prefill call,
inputs resident in HBM); the other calls are reported in microseconds per
call.  L2 is flushed (256 MiB write) before every timed call.  Two long-sequence prefills
are timed the same way outside the step and reported beside it: one sequence of 131 072
tokens at H=16 (`prefill_long`) and four of 32 768 tokens at H=4 (`prefill_tp_slice`).

`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
prefill workload on the host cores (the method has no runnable reference
implementation; the oracle is the reference arm).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "KDA prefill tokens/s and decode/verify+commit µs/step; % of HBM/TC roofline"
D, C = 128, 64
STATE_BYTES = D * D * 4


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# --------------------------------------------------------------------------
# algorithmic work per call


def prefill_work(lengths, H, M, in_bytes=2, out_bytes=2):
    """Bytes and flops of one prefill call (per (token, head): q, k, v, raw gate,
    raw beta, o; per (sequence, head): initial + final state and M snapshots)."""
    T = sum(lengths)
    per_tok = 4 * D * in_bytes + in_bytes + D * out_bytes
    n_states = len(lengths) * H * (2 + M)
    byts = T * H * per_tok + n_states * STATE_BYTES
    flops = T * H * (10 * C * D + 6 * D * D + C * C / 3)
    return byts, flops


# DRAM traffic of one two-phase prefill call, from ncu captures of its two kernels
# (dram__bytes_read.sum + dram__bytes_write.sum of prep and sweep: 201.94 + 379.37 and
# 548.30 + 62.24 MB) on the `--profile prefill` case (8 x 2048 tokens, 16 heads); traffic
# grows with the token-heads processed, so a launch is charged this much per token-head.
# The figure belongs to the kernel source it was captured on: the line reports null traffic
# once that file's sha256 no longer starts with the recorded prefix.
PREFILL_TRAFFIC = {
    "source": "serving_kda_chunk_gb300/csrc/prefill_2p.cu",
    "sha256_prefix": "d683cc7bea0733af",
    "capture": "profiles/prefill_2p_prep_kernel_batched_8x2048_h16.md, "
               "profiles/prefill_2p_sweep_kernel_batched_8x2048_h16.md",
    "bytes_per_token_head": (201.940992e6 + 379.373312e6 + 548.301056e6 + 62.239744e6) / (8 * 2048 * 16),
}


def prefill_traffic(token_heads):
    """Measured DRAM bytes of a prefill call over token_heads, or None if the kernel source has
    changed since the capture."""
    import hashlib

    try:
        with open(os.path.join(ROOT, PREFILL_TRAFFIC["source"]), "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    if not digest.startswith(PREFILL_TRAFFIC["sha256_prefix"]):
        return None
    return PREFILL_TRAFFIC["bytes_per_token_head"] * token_heads


def decode_work(R, H, sb=STATE_BYTES):
    return R * H * (2 * sb + 4 * D * 2 + 2 + D * 2)


def verify_work(R, K, H, sb=STATE_BYTES):
    return R * H * (sb + K * (4 * D * 2 + 2 + D * 2 + D * 4 + 2 * D * 2))


def commit_work(acc, H, K, sb=STATE_BYTES):
    """Checkpoint read + state write and the a kept records per (request, head),
    plus the token ids read and the lengths / next tokens written once each."""
    ids = len(acc) * (2 * K * 4 + 2 * 4)
    return ids + sum(H * (2 * sb + a * (D * 4 + 2 * D * 2)) for a in acc if a > 0)


# --------------------------------------------------------------------------
# clocks sampled during the timed region


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        load = [s for s, p in zip(sm, pw) if p is not None] or sm
        hi = sorted(load)[len(load) // 2:] or load  # samples under load: upper half by clock
        return {"sm_mhz": statistics.median(hi), "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons)}


# --------------------------------------------------------------------------
# workloads on the device


def to_dev(a, dtype, dev):
    import torch

    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)


def i32(a, dev):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)


class Step:
    """The entry points on resident device buffers.  `parts` selects which workloads are built
    (all of them for the benchmark; one for a profiler capture).  compact_decode_pool keeps only
    the 256 slots the decode batch touches (same work per call, 512 MiB instead of 2 GiB)."""

    PARTS = ("prefill", "decode", "spec", "copy")

    def __init__(self, dev, parts=PARTS, compact_decode_pool=False):
        import torch

        import serving_kda_chunk_gb300 as kda

        self.kda = kda
        self.dev = dev
        self.parts = tuple(parts)
        t0 = time.time()
        if "prefill" in parts:
            c1 = _batched_prefill()
            self.c1 = c1
            self.pre = {n: to_dev(c1[n], "bf16", dev) for n in ("q", "k", "v", "beta", "gate")}
            self.pre_host = {n: torch.from_numpy(c1[n].view(np.int16)).view(torch.bfloat16)
                             .pin_memory() for n in ("q", "k", "v", "beta", "gate")}
            self.cu = i32(c1["cu_seqlens"], dev)
            self.pool1 = torch.from_numpy(c1["pool"]).to(dev)
            self.slots1 = i32(c1["init_slot"], dev)
            self.track1 = i32(c1["track"], dev)
            self.snap1 = torch.empty(c1["N"], 1, 32, D, D, device=dev)
            self.out1 = torch.empty(c1["T"], 32, D, dtype=torch.bfloat16, device=dev)
            self.out1_host = torch.empty(c1["T"], 32, D, dtype=torch.bfloat16).pin_memory()
            ws = kda.kda_chunk_prefill_workspace_size(c1["T"], c1["N"], 32)
            self.ws1 = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        if "decode" in parts:
            c2 = W.decode_256req_h32()
            self.dec = {n: to_dev(c2[n], "bf16", dev) for n in ("q", "k", "v", "beta", "gate")}
            if compact_decode_pool:
                self.pool2 = torch.from_numpy(c2["pool"][c2["slot"]]).to(dev)
                self.slot2 = i32(np.arange(len(c2["slot"])), dev)
            else:
                self.pool2 = torch.from_numpy(c2["pool"]).to(dev)
                self.slot2 = i32(c2["slot"], dev)
            self.out2 = torch.empty(256, 32, D, dtype=torch.bfloat16, device=dev)
        if "spec" in parts:
            c3 = W.spec_64req_k7_h32()
            self.c3 = c3
            self.spec = {n: to_dev(c3[n], "bf16", dev) for n in ("q", "k", "v", "beta", "gate")}
            self.pool3 = torch.from_numpy(c3["pool"]).to(dev)
            self.ckpt3 = i32(c3["ckpt"], dev)
            a3 = W.accept_case(3, 64, 7, p_match=0.7)
            self.tok3, self.smp3 = i32(a3["tokens"], dev), i32(a3["sampled"], dev)
            self.acc3 = torch.empty(64, dtype=torch.int32, device=dev)
            self.next3 = torch.empty(64, dtype=torch.int32, device=dev)
            self.rec_u = torch.empty(64, 32, 7, D, device=dev)
            self.rec_kg = torch.empty(64, 32, 7, 2 * D, dtype=torch.bfloat16, device=dev)
            self.out3 = torch.empty(64 * 7, 32, D, dtype=torch.bfloat16, device=dev)
            # short-convolution windows of q, k and v: 4096 bf16 channels, width 4 (keep 3)
            cc = W.conv_case(5, 64, 7, 3, 4096, 3, 64, dtype="bf16")
            self.conv3 = [torch.from_numpy(x.view(np.int16)).to(dev) for x in cc["pools"]]
            self.conv_slot3 = i32(cc["slots"], dev)
        if "copy" in parts:
            c4 = W.slot_fanout_256x8_pool4096()
            g = torch.Generator(device=dev).manual_seed(4)
            self.pool4 = torch.empty(4096, 16, D, D, device=dev)
            for i in range(0, 4096, 512):
                self.pool4[i:i + 512].normal_(0.0, 0.1, generator=g)
            self.c4 = {n: i32(c4[n], dev) for n in ("clear", "src", "dst_offsets", "dst")}
            self.n4 = (len(c4["src"]), len(c4["dst"]), len(c4["clear"]))
            self.ws4 = torch.empty(kda.kda_slot_copy_workspace_size(4096), dtype=torch.uint8,
                                   device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.setup_s = time.time() - t0
        torch.cuda.synchronize()

    def prefill(self, pre=None):
        p = pre or self.pre
        self.kda.kda_chunk_prefill(p["q"], p["k"], p["v"], p["beta"], p["gate"], self.cu,
                                   self.out1, state_pool=self.pool1, init_slot=self.slots1,
                                   final_slot=self.slots1, track_chunk_idx=self.track1,
                                   track_state=self.snap1, workspace=self.ws1,
                                   dev_status=self.status)

    def decode(self):
        d = self.dec
        self.kda.kda_recurrent_decode(d["q"], d["k"], d["v"], d["beta"], d["gate"], self.pool2,
                                      self.slot2, self.out2, dev_status=self.status)

    def verify(self):
        s = self.spec
        self.kda.kda_spec_verify(s["q"], s["k"], s["v"], s["beta"], s["gate"], self.pool3,
                                 self.ckpt3, self.rec_u, self.rec_kg, self.out3, K=7,
                                 dev_status=self.status)

    def commit(self):
        # accepted lengths from the token ids, the recurrent-state rebuild and the q / k / v
        # conv windows, one launch
        self.kda.kda_spec_accept_commit(self.pool3, self.ckpt3, self.tok3, self.smp3, self.rec_u,
                                        self.rec_kg, num_accepted=self.acc3,
                                        next_token=self.next3, convs=self.conv3,
                                        conv_slot=self.conv_slot3, conv_keep=3,
                                        dev_status=self.status)

    def conv_compact(self):
        self.kda.kda_conv_compact(self.conv3, self.conv_slot3, self.acc3, 3,
                                  dev_status=self.status)

    def slot_copy(self):
        c = self.c4
        self.kda.kda_slot_copy([self.pool4], c["clear"], c["src"], c["dst_offsets"], c["dst"],
                               self.ws4, dev_status=self.status)

    # name -> (callable, kernel launches), for the parts that were built
    def calls(self):
        part = {"prefill": "prefill", "decode": "decode", "verify": "spec", "commit": "spec",
                "conv_compact": "spec", "slot_copy": "copy"}
        every = [("prefill", self.prefill, 3), ("decode", self.decode, 1),
                 ("verify", self.verify, 1), ("commit", self.commit, 1),
                 ("slot_copy", self.slot_copy, 2)]
        return [c for c in every if part[c[0]] in self.parts]

    # entry points measured on their own, outside the step (profile cases)
    def extra_calls(self):
        return [("conv_compact", self.conv_compact, 1)] if "spec" in self.parts else []


def run_device(step, steps, warmup, rank, world):
    import torch

    calls = step.calls()
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for _, fn, _ in calls:
            step.flush.zero_()
            fn()
    torch.cuda.synchronize()
    times = {name: [] for name, _, _ in calls}
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    evs = []
    for _ in range(steps):
        row = []
        for name, fn, _ in calls:
            step.flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            row.append((name, a, b))
        evs.append(row)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop() if sampler else None
    for row in evs:
        for name, a, b in row:
            times[name].append(a.elapsed_time(b) * 1e-3)
    launches = steps * sum(n for _, _, n in calls)
    return times, wall, clocks, launches


def run_state_bf16(step, steps, warmup):
    """decode, verify and the fused accept + commit on bf16 copies of their state pools
    (KDA_STATE_BF16: 32 KiB per head), timed like the step's calls (L2 flushed before each
    call, CUDA events on the launching stream).  Returns mean seconds per call."""
    import torch

    kda = step.kda
    pool2, pool3 = step.pool2.to(torch.bfloat16), step.pool3.to(torch.bfloat16)
    d, s = step.dec, step.spec

    def decode():
        kda.kda_recurrent_decode(d["q"], d["k"], d["v"], d["beta"], d["gate"], pool2, step.slot2,
                                 step.out2, dev_status=step.status)

    def verify():
        kda.kda_spec_verify(s["q"], s["k"], s["v"], s["beta"], s["gate"], pool3, step.ckpt3,
                            step.rec_u, step.rec_kg, step.out3, K=7, dev_status=step.status)

    def commit():
        kda.kda_spec_accept_commit(pool3, step.ckpt3, step.tok3, step.smp3, step.rec_u,
                                   step.rec_kg, num_accepted=step.acc3, next_token=step.next3,
                                   dev_status=step.status)

    calls = [("decode", decode), ("verify", verify), ("commit", commit)]
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for _, fn in calls:
            step.flush.zero_()
            fn()
    torch.cuda.synchronize()
    evs = []
    for _ in range(steps):
        for name, fn in calls:
            step.flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((name, a, b))
    torch.cuda.synchronize()
    t = {name: [] for name, _ in calls}
    for name, a, b in evs:
        t[name].append(a.elapsed_time(b) * 1e-3)
    return {k: statistics.mean(v) for k, v in t.items()}


def run_spec_graph(step, steps, warmup):
    """The spec step (verify, then the fused accept + commit + conv windows) captured once in a
    CUDA graph and replayed: the step as a serving loop runs it, without per-launch host
    overhead.  L2 is flushed before each replay (outside the graph); CUDA events around the
    replay.  Returns mean seconds per replay."""
    import torch

    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        step.verify()
        step.commit()
    torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    for _ in range(warmup):
        step.flush.zero_()
        g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        step.flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(main)
        g.replay()
        b.record(main)
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e-3)
    return statistics.mean(ts)


def run_prefill_long(step, reps):
    """One long sequence (131 072 tokens, H = 16, snapshots every 64 chunks, final state to a
    slot): the chunk recurrence leaves one (sequence, head) unit per head, so 16 SMs carry it.
    Timed like the step's calls (L2 flushed, CUDA events), outside the timed step.  Returns
    (mean seconds, tokens, algorithmic bytes)."""
    import torch

    c = W.long_prefill_131072_h16()
    dev = step.dev
    t = {n: to_dev(c[n], "bf16", dev) for n in ("q", "k", "v", "beta", "gate")}
    T, H = c["T"], c["H"]
    pool = torch.zeros(1, H, D, D, device=dev)
    cu = i32(c["cu_seqlens"], dev)
    fin = i32([0], dev)
    tr = i32(c["track"], dev)
    snap = torch.empty(1, c["track"].shape[1], H, D, D, device=dev)
    out = torch.empty(T, H, D, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(step.kda.kda_chunk_prefill_workspace_size(T, 1, H), 16),
                     dtype=torch.uint8, device=dev)

    def call():
        step.kda.kda_chunk_prefill(t["q"], t["k"], t["v"], t["beta"], t["gate"], cu, out,
                                   state_pool=pool, final_slot=fin, track_chunk_idx=tr,
                                   track_state=snap, workspace=ws, dev_status=step.status)

    call()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        step.flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e-3)
    n_states = 1 + int((c["track"] >= 0).sum())  # final state + snapshots (no initial state)
    return statistics.mean(ts), T, T * H * 1282 + n_states * H * STATE_BYTES


def run_prefill_tp_slice(step, reps):
    """Four sequences of 32 768 tokens at H = 4 (a tensor-parallel slice of 32 heads): 16
    (sequence, head) units, swept as chunk segments at once.  Seeded inputs with the workload
    recipe, initial and final states in slots, one snapshot per sequence; timed like the long
    prefill.  Returns (mean seconds, tokens, algorithmic bytes)."""
    import torch

    c = W.tp_slice_prefill_4x32768_h4()
    dev = step.dev
    t = {n: to_dev(c[n], "bf16", dev) for n in ("q", "k", "v", "beta", "gate")}
    T, H, N = c["T"], c["H"], c["N"]
    pool = torch.from_numpy(c["pool"]).to(dev)
    cu, sl, tr = i32(c["cu_seqlens"], dev), i32(c["init_slot"], dev), i32(c["track"], dev)
    snap = torch.empty(N, 1, H, D, D, device=dev)
    out = torch.empty(T, H, D, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(step.kda.kda_chunk_prefill_workspace_size(T, N, H), 16), dtype=torch.uint8, device=dev)

    def call():
        step.kda.kda_chunk_prefill(t["q"], t["k"], t["v"], t["beta"], t["gate"], cu, out,
                                   state_pool=pool, init_slot=sl, final_slot=sl, track_chunk_idx=tr,
                                   track_state=snap, workspace=ws, dev_status=step.status)

    call()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        step.flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e-3)
    n_states = 2 * N + int((c["track"] >= 0).sum())  # initial + final states and snapshots
    return statistics.mean(ts), T, T * H * 1282 + n_states * H * STATE_BYTES


def run_e2e(step, steps, warmup):
    """Prefill through the public call with host buffers, streamed per sequence: the pinned
    H2D copies of a sequence's inputs (one stream, longest sequence first), its
    kda_chunk_prefill call (one stream and one workspace per sequence, so sequences overlap on
    the GPU and each takes the two-phase path) and the
    D2H copy of its output rows (one stream) overlap with the other sequences' copies and
    compute; everything is inside the timed region.  The step is captured once in a CUDA graph
    and replayed for every timed step.  Every sequence is independent, so the outputs, final
    states and snapshots are those of the one-call prefill."""
    import torch

    c1 = step.c1
    cu = c1["cu_seqlens"]
    N = int(c1["N"])
    order = sorted(range(N), key=lambda n: -(int(cu[n + 1]) - int(cu[n])))
    dev_in = step.pre
    host_in = step.pre_host
    # every sequence's [0, length] in one pinned block and one copy (rows padded to 16 bytes:
    # the entry points take 16-byte aligned arrays)
    cu_host = torch.tensor([[0, int(cu[n + 1]) - int(cu[n]), 0, 0] for n in range(N)], dtype=torch.int32).pin_memory()
    cu_dev_all = torch.empty(N, 4, dtype=torch.int32, device=step.dev)
    cu_dev = [cu_dev_all[n, :2] for n in range(N)]
    # per-sequence slot / snapshot index arrays (own 16-byte-aligned allocations), resident like
    # the pool, as in the one-call prefill
    slot_n = [step.slots1[n:n + 1].clone() for n in range(N)]
    track_n = [step.track1[n:n + 1].clone() for n in range(N)]
    # one workspace per sequence (the calls run concurrently): the two-phase path
    H = int(c1["H"])
    ws_n = [torch.empty(max(16, step.kda.kda_chunk_prefill_workspace_size(int(cu[n + 1]) - int(cu[n]), 1, H)),
                        dtype=torch.uint8, device=step.dev) for n in range(N)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values()) + 16 * N
    d2h = step.out1.numel() * step.out1.element_size()
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    s_cmp = [torch.cuda.Stream() for _ in range(N)]
    main = torch.cuda.current_stream()

    def once():
        cur = torch.cuda.current_stream()  # the capture stream while the step is captured
        start = torch.cuda.Event()
        start.record(cur)
        s_h2d.wait_event(start)
        # every input copy is queued before any prefill call, so that the host's work on the
        # calls never leaves the host link idle; each call waits only for its own sequence's rows
        ready = {}
        with torch.cuda.stream(s_h2d):
            cu_dev_all.copy_(cu_host, non_blocking=True)
            for n in order:
                a, b = int(cu[n]), int(cu[n + 1])
                for name, t in host_in.items():
                    dev_in[name][a:b].copy_(t[a:b], non_blocking=True)
                ready[n] = torch.cuda.Event()
                ready[n].record(s_h2d)
        for n in order:
            a, b = int(cu[n]), int(cu[n + 1])
            s_cmp[n].wait_event(ready[n])
            with torch.cuda.stream(s_cmp[n]):
                step.kda.kda_chunk_prefill(
                    dev_in["q"][a:b], dev_in["k"][a:b], dev_in["v"][a:b], dev_in["beta"][a:b],
                    dev_in["gate"][a:b], cu_dev[n], step.out1[a:b], state_pool=step.pool1,
                    init_slot=slot_n[n], final_slot=slot_n[n],
                    track_chunk_idx=track_n[n], track_state=step.snap1[n:n + 1],
                    workspace=ws_n[n], dev_status=step.status, stream=s_cmp[n])
                done = torch.cuda.Event()
                done.record(s_cmp[n])
            s_d2h.wait_event(done)
            with torch.cuda.stream(s_d2h):
                step.out1_host[a:b].copy_(step.out1[a:b], non_blocking=True)
        cur.wait_stream(s_d2h)

    for _ in range(warmup):
        step.flush.zero_()
        once()
    torch.cuda.synchronize()
    # the step (copies in, calls, copies out) captured once and replayed, as a serving loop
    # would: host-side pauses between the issue of its operations then cannot stretch the
    # timed region, which still covers every copy and every call of the step
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        once()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        step.flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(main)
        graph.replay()
        b.record(main)
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e-3)
    # the host link's own rate on this machine, one direction at a time (256 MiB pinned copies)
    link = {}
    dev_buf, host_buf = step.out1.view(-1)[: 1 << 27], step.out1_host.view(-1)[: 1 << 27]
    for name, dst, src in (("h2d_gbs", dev_buf, host_buf), ("d2h_gbs", host_buf, dev_buf)):
        best = 0.0
        for _ in range(3):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(main)
            dst.copy_(src, non_blocking=True)
            b.record(main)
            b.synchronize()
            best = max(best, src.numel() * src.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9)
        link[name] = best
    return ts, h2d, d2h, link


# --------------------------------------------------------------------------
# CPU oracle on a bounded sample of the prefill workload


_BATCHED_PREFILL = None


def _batched_prefill():
    global _BATCHED_PREFILL
    if _BATCHED_PREFILL is None:
        _BATCHED_PREFILL = W.batched_prefill_8seq_h32()
    return _BATCHED_PREFILL


def cpu_oracle_sample(heads=tuple(range(8)), threads=None):
    import oracle

    c = _batched_prefill()
    H = c["H"]
    hs = list(heads)
    wid = lambda n: W.widen(c[n], "bf16")[:, hs]  # noqa: E731
    S0 = c["pool"][c["init_slot"]][:, hs].astype(np.float64)
    cores = threads or (os.cpu_count() or 1)
    args = (wid("q"), wid("k"), wid("v"), W.widen(c["beta"], "bf16")[:, hs], wid("gate"))
    t0 = time.perf_counter()
    oracle.prefill(*args, c["cu_seqlens"], S0=S0, track=c["track"], n_threads=cores)
    dt = time.perf_counter() - t0
    tok_heads = c["T"] * len(hs)
    value = tok_heads / H / dt  # full-width (all H heads) tokens per second
    sample = (f"fp64 oracle prefill on heads {hs} of {H} for all {c['N']} sequences "
              f"({c['T']} tokens), {dt:.2f} s wall; value scaled to all heads")
    return {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": sample}


# --------------------------------------------------------------------------
# distributed plumbing (replicas: no collective on the data path)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------


def config_block():
    lengths = W.batched_prefill_lengths()
    return {"workload": (f"batched chunk prefill: 8 packed seqs, lengths {lengths} "
                         f"(sum {sum(lengths)}), H=32, d_k=d_v=128, chunk=64, bf16 in/out, "
                         "fp32 state; step also runs decode 256xH32, spec verify + fused "
                         "accept/commit + q/k/v conv-window compaction "
                         "64xK7xH32, slot copy 256x8 + 512 clears of 1 MiB states"),
            "global_batch": 8, "seq_len": max(lengths), "tokens": sum(lengths),
            "l2": "flushed (256 MiB write) before every timed call",
            "parallelism": "replicas (one independent copy per GPU)"}


def main_reference(args, rank, world):
    if rank != 0:
        return 0
    steps, warmup = max(1, args.steps), max(0, args.warmup)
    # each step is the oracle on a few heads of the whole batch (~0.15 s of wall time per head
    # on 16 cores), so that the run stays within a couple of minutes for any K + W up to ~200
    n_heads = 4 if steps + warmup <= 60 else 2
    vals = []
    for _ in range(warmup):
        cpu_oracle_sample(heads=tuple(range(n_heads)))
    cb = None
    for _ in range(steps):
        cb = cpu_oracle_sample(heads=tuple(range(n_heads)))
        vals.append(cb["value"])
    value = statistics.mean(vals)
    cb["value"] = value
    cb["sample"] += f"; mean over {steps} steps"
    toks = sum(W.batched_prefill_lengths())
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": 1, "steps": steps, "warmup": warmup,
            "ms_per_step": toks / value * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_block(),
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_profile_case(name, reps):
    """One entry point on its workload, for an ncu capture (`--profile NAME`).

    prefill runs a reduced batch (8 sequences x 2048 tokens, H=16: 168 MB of
    activations, above L2) so that a full-set capture ends quickly, through the
    two-phase kernels (prefill) or the single-pass kernel (prefill_single); the
    other entry points run their serving workloads."""
    import torch

    import serving_kda_chunk_gb300 as kda

    dev = torch.device("cuda", 0)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    if name in ("prefill", "prefill_single"):
        # "prefill": the two-phase kernels (the workspace the benchmark passes); "prefill_single":
        # the single-pass kernel (a workspace too small for the two-phase plan)
        c = W.prefill_case(11, [2048] * 8, 16, pool_slots=8)
        t = {n: to_dev(c[n], "bf16", dev) for n in ("q", "k", "v", "beta", "gate")}
        pool = torch.from_numpy(c["pool"]).to(dev)
        sl, tr, cu = i32(c["init_slot"], dev), i32(c["track"], dev), i32(c["cu_seqlens"], dev)
        snap = torch.empty(8, 1, 16, D, D, device=dev)
        out = torch.empty(c["T"], 16, D, dtype=torch.bfloat16, device=dev)
        need = kda.kda_chunk_prefill_workspace_size(c["T"], 8, 16)
        ws = torch.empty(need if name == "prefill" else 64, dtype=torch.uint8, device=dev)

        def fn():
            kda.kda_chunk_prefill(t["q"], t["k"], t["v"], t["beta"], t["gate"], cu, out,
                                  state_pool=pool, init_slot=sl, final_slot=sl,
                                  track_chunk_idx=tr, track_state=snap, workspace=ws)
    elif name == "prefill_long":
        # one sequence of 32 768 tokens (512 chunks), H = 16: the long-sequence segment scan on a
        # reduced case (1.1 GB of workspace) so that a capture of its kernels ends quickly
        c = W.prefill_case(13, [32768], 16, pool_slots=1, track=[[0, 64, 511]])
        t = {n: to_dev(c[n], "bf16", dev) for n in ("q", "k", "v", "beta", "gate")}
        pool = torch.from_numpy(c["pool"]).to(dev)
        sl, tr, cu = i32(c["init_slot"], dev), i32(c["track"], dev), i32(c["cu_seqlens"], dev)
        snap = torch.empty(1, 3, 16, D, D, device=dev)
        out = torch.empty(c["T"], 16, D, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(kda.kda_chunk_prefill_workspace_size(c["T"], 1, 16), dtype=torch.uint8, device=dev)

        def fn():
            kda.kda_chunk_prefill(t["q"], t["k"], t["v"], t["beta"], t["gate"], cu, out,
                                  state_pool=pool, init_slot=sl, final_slot=sl,
                                  track_chunk_idx=tr, track_state=snap, workspace=ws)
    elif name == "slot_copy_small":
        # the fused copy kernel on a reduced pool (512 slots of 1 MiB states, 32 parents x 8
        # children + 64 clears: 352 MiB moved, above L2) so that a multi-pass capture holds
        # well under a few GB
        sc = W.slot_copy_case(12, 512, 32, 8, 64)
        pool = torch.empty(512, 16, D, D, device=dev)
        pool.normal_(0.0, 0.1, generator=torch.Generator(device=dev).manual_seed(12))
        args = [i32(sc[n], dev) for n in ("clear", "src", "dst_offsets", "dst")]
        ws = torch.empty(kda.kda_slot_copy_workspace_size(512), dtype=torch.uint8, device=dev)

        def fn():
            kda.kda_slot_copy([pool], *args, ws)
    elif name == "verify_bf16":
        # verify on a bf16 copy of the checkpoint pool (KDA_STATE_BF16): the checkpoint is used
        # as the MMA's shared-memory operand where it lands
        step = Step(dev, parts=("spec",), compact_decode_pool=True)
        pool3 = step.pool3.to(torch.bfloat16)
        s3 = step.spec

        def fn():
            kda.kda_spec_verify(s3["q"], s3["k"], s3["v"], s3["beta"], s3["gate"], pool3, step.ckpt3,
                                step.rec_u, step.rec_kg, step.out3, K=7, dev_status=step.status)
    else:
        part = {"decode": "decode", "verify": "spec", "commit": "spec", "conv_compact": "spec",
                "slot_copy": "copy"}[name]
        step = Step(dev, parts=(part,), compact_decode_pool=True)
        fn = dict((n, f) for n, f, _ in step.calls() + step.extra_calls())[name]
        if name in ("commit", "conv_compact"):
            step.verify()  # records for the commit to read
    times = []
    for _ in range(reps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1e3)
    print(json.dumps({"profile": name, "us_per_call": times}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kda", choices=["kda", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=["prefill", "prefill_single", "prefill_long", "decode", "verify", "verify_bf16", "commit",
                                          "conv_compact", "slot_copy", "slot_copy_small"],
                    help="run one entry point a few times (for an ncu capture) and exit")
    args = ap.parse_args()
    if args.profile:
        return run_profile_case(args.profile, max(args.steps, 1))
    rank, world, local = dist_setup()
    if args.impl == "reference":
        rc = main_reference(args, rank, world)
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return rc

    import torch

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    step = Step(dev)
    times, wall, clocks, launches = run_device(step, args.steps, args.warmup, rank, world)
    e2e_steps, h2d, d2h, link = run_e2e(step, max(1, min(args.steps, 5)), min(args.warmup, 3))
    e2e_t = statistics.mean(e2e_steps)
    t16 = run_state_bf16(step, max(1, min(args.steps, 5)), min(args.warmup, 3))
    t_graph = run_spec_graph(step, max(1, min(args.steps, 5)), min(args.warmup, 3))
    t_long, tok_long, b_long = run_prefill_long(step, 2)
    t_tp, tok_tp, b_tp = run_prefill_tp_slice(step, 3)

    hbm, tc, peak_kind = load_peaks()
    mean = {k: statistics.mean(v) for k, v in times.items()}
    lengths = step.c1["lengths"]
    toks = sum(lengths)
    t_pre = max_over_ranks(mean["prefill"], world)
    value = sum_over_ranks(toks, world) / t_pre
    e2e_val = sum_over_ranks(toks, world) / max_over_ranks(e2e_t, world)
    pb, pf = prefill_work(lengths, 32, 1)
    achieved = pb / mean["prefill"] / 1e9
    traffic = prefill_traffic(toks * 32)
    t_hbm, t_tc = pb / (hbm * 1e9), pf / (tc * 1e12)
    dec_b = decode_work(256, 32)
    ver_b = verify_work(64, 7, 32)
    conv_b = sum(3 * 2 * 3 * 4096 * 2 for a in step.acc3.cpu().tolist() if a > 0)
    com_b = commit_work(step.acc3.cpu().tolist(), 32, 7) + conv_b
    cp_b = STATE_BYTES * 16 * (sum(step.n4))
    parts = {
        "prefill": {"us": mean["prefill"] * 1e6, "tokens_per_s": toks / mean["prefill"],
                    "bytes": pb, "flops": pf, "hbm_frac": t_hbm / mean["prefill"],
                    "tensor_frac": t_tc / mean["prefill"]},
        "decode": {"us": mean["decode"] * 1e6, "bytes": dec_b,
                   "hbm_frac": dec_b / (hbm * 1e9) / mean["decode"]},
        "verify": {"us": mean["verify"] * 1e6, "bytes": ver_b,
                   "hbm_frac": ver_b / (hbm * 1e9) / mean["verify"]},
        "commit": {"us": mean["commit"] * 1e6, "bytes": com_b,
                   "mean_accepted": float(step.acc3.float().mean().item()),
                   "hbm_frac": com_b / (hbm * 1e9) / mean["commit"]},
        "verify_commit_us_per_step": (mean["verify"] + mean["commit"]) * 1e6,
        "verify_commit_graph_us": t_graph * 1e6,
        "prefill_long": {"us": t_long * 1e6, "tokens_per_s": tok_long / t_long, "bytes": b_long,
                         "hbm_frac": b_long / (hbm * 1e9) / t_long,
                         "note": "1 x 131072 tokens, H=16: the prep on every SM, then 10 chunk segments swept at once (the middle segments' state maps and offsets, the start states chained, every segment swept from its start)"},
        "prefill_tp_slice": {"us": t_tp * 1e6, "tokens_per_s": tok_tp / t_tp, "bytes": b_tp,
                             "hbm_frac": b_tp / (hbm * 1e9) / t_tp,
                             "note": "4 x 32768 tokens, H=4 (a tensor-parallel slice of 32 heads): 16 (sequence, head) units, each swept as chunk segments at once"},
        "slot_copy": {"us": mean["slot_copy"] * 1e6, "bytes": cp_b,
                      "hbm_frac": cp_b / (hbm * 1e9) / mean["slot_copy"]},
    }
    sb16 = STATE_BYTES // 2
    w16 = {"decode": decode_work(256, 32, sb16), "verify": verify_work(64, 7, 32, sb16),
           "commit": commit_work(step.acc3.cpu().tolist(), 32, 7, sb16)}
    parts["state_bf16"] = {
        name: {"us": t16[name] * 1e6, "bytes": w16[name],
               "hbm_frac": w16[name] / (hbm * 1e9) / t16[name]} for name in w16}
    parts["state_bf16"]["note"] = ("same calls on bf16 copies of the pools (KDA_STATE_BF16), "
                                   "outside the timed step")
    step_s = sum(mean.values())
    status = int(step.status.item())
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_oracle_sample()
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; bf16 inputs, fp32 state)", "config": config_block(),
        "roofline": {"bound": "hbm", "kernel": "kda_chunk_prefill (plan + prep + sweep)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": traffic,
                     "traffic_over_algorithmic": (traffic / pb) if traffic else None,
                     "traffic_source": PREFILL_TRAFFIC["capture"],
                     "peak_source": f"{peak_kind} hbm_gbs (burst copy)"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "link_measured": link,
                # the link is full duplex: the slower direction bounds the step
                "link_bound_tokens_per_s": toks / max(h2d / (link["h2d_gbs"] * 1e9),
                                                      d2h / (link["d2h_gbs"] * 1e9)),
                "ms_per_step_each": [round(t * 1e3, 3) for t in e2e_steps]},
        "gpu_launches": launches,
        "clocks": clocks,
        "parts": parts,
        "dev_status": status,
        "wall_s_timed": wall,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
