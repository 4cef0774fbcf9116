#!/usr/bin/env python
"""Benchmark of the quantized KV-cache decode step on GB300 (one JSON line).

A step is one decode step of the whole hot path for every layer of the
workload: quantize-on-append of the new token of every sequence (bf16 residual
write, group spill or FP8 encode), then fused decode attention over the whole
cache (split pass + log-sum-exp combine).  Inputs are seeded synthetic tensors
already resident in HBM; the cache is built before the timed region.

Metric: effective KV GB/s = algorithmic bytes of one step (codes + scales and
zero-points + bf16 sink/residual + q + out + lse + append traffic, every KV head
read once) / step time.  Also reported: % of the measured HBM peak, tokens/s
(sequences decoded per second), and the same metric end to end ("e2e"): every
step's inputs copied in from pinned host memory and its results copied back,
on a copy stream that overlaps them with the neighbouring steps' kernels, all
inside the timed region.

  python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl reference]

Under torchrun (N > 1) every rank runs its own copy of the workload on its own
GPU (the path shards by sequence with no exchange: weak scaling); rank 0 prints.
"""
from __future__ import annotations

import os

# the CPU oracle baseline is timed single-threaded (set before numpy loads BLAS)
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import argparse
import dataclasses
import datetime
import json
import math
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_kv_cache_decode_gb300 import inputs as I  # noqa: E402

DEFAULT_WORKLOAD = "paged_mixed_int8_int4_64l"
# where the raw nvidia-smi clock samples of the timed region are written (the JSON line
# carries their summary)
OUT_DIR = os.environ.get("KVQ_BENCH_OUT", os.path.join(ROOT, "bench_out"))
L2_BYTES = 129 * 2 ** 20


# --------------------------------------------------------------------------- #
# byte accounting (algorithmic bytes; the roofline numerator)
# --------------------------------------------------------------------------- #


def is_fp8(fmt):
    return fmt.fmt in ("fp8_e4m3", "fp8_e5m2")


def split_tokens(T, fmt):
    n_sink = min(T, fmt.S)
    n = T - n_sink
    if is_fp8(fmt):
        return n_sink, n, 0
    if fmt.fmt == "bf16":  # skip layer: nothing quantized
        return n_sink, 0, n
    qn = max(0, (n - fmt.R) // fmt.G) * fmt.G
    return n_sink, qn, n - qn


def attention_bytes(fmt, T, H, d=128):
    """Bytes one (sequence, kv head) must read for attention over T tokens."""
    bits = I.FORMAT_BITS[fmt.fmt]
    n_sink, qn, r = split_tokens(T, fmt)
    b = 2 * qn * d * bits // 8
    if not is_fp8(fmt) and qn:
        b += (qn // fmt.G) * d * 8 + qn * (d // fmt.Gv) * 8
        b += qn * 4 * (fmt.k_outliers + fmt.v_outliers)  # dense-and-sparse entries
    b += (n_sink + r) * d * 2 * 2
    return b * H


def append_bytes(fmt, T_before, n, H, d=128):
    """Bytes moved by appending n tokens to one sequence (all heads)."""
    bits = I.FORMAT_BITS[fmt.fmt]
    b = 2 * n * d * 2  # read new K, V
    if is_fp8(fmt):
        return H * (b + 2 * n * d)
    _, q0, _ = split_tokens(T_before, fmt)
    n_sink1, q1, r1 = split_tokens(T_before + n, fmt)
    spilled = q1 - q0
    b += 2 * n * d * 2  # ring write (upper bound: every new token)
    b += spilled * 2 * d * 2  # spilled tokens read back (bf16 K, V)
    b += 2 * spilled * d * bits // 8 + (spilled // fmt.G) * d * 8 + spilled * (d // fmt.Gv) * 8
    b += spilled * 4 * (getattr(fmt, "k_outliers", 0) + getattr(fmt, "v_outliers", 0))
    return H * b


def step_bytes(w, lens_after, n_app):
    total = 0
    for l, fmt in enumerate(w.layer_formats):
        for T in lens_after:
            total += attention_bytes(fmt, int(T), w.num_kv_heads)
            total += append_bytes(fmt, int(T) - n_app, n_app, w.num_kv_heads)
        B = len(lens_after) * w.n_query    # query rows
        total += B * w.num_q_heads * 128 * 2  # q
        total += B * w.num_q_heads * 128 * 2  # out (bf16)
        total += B * w.num_q_heads * 4        # lse
    return total


# --------------------------------------------------------------------------- #
# multi-rank aggregation (weak scaling: every rank runs its own replica)
# --------------------------------------------------------------------------- #


def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step: float, ms_per_step_max: float, world: int) -> float:
    """Whole-job GB/s: the bytes all ranks processed per step over the slowest rank's step time."""
    return bytes_per_rank_step * world / (ms_per_step_max * 1e-3) / 1e9


# --------------------------------------------------------------------------- #
# clocks
# --------------------------------------------------------------------------- #


class ClockSampler:
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str):
        self.path = path
        self.proc = None
        try:
            self.f = open(path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self, t0: float, t1: float):
        """Median SM clock and active throttle reasons of the samples taken in [t0, t1] (epoch s)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(p[2]), float(p[3]), p[6:10]))
                except ValueError:
                    continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed"
        if not inside:
            inside, window = rows, "warmup+timed"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[3][i].lower().startswith("active")})
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# --------------------------------------------------------------------------- #
# the GPU workload
# --------------------------------------------------------------------------- #


class Layer:
    """One layer's cache (one replica) with its step inputs and outputs."""

    def __init__(self, kvq, torch, w, l, fmt, lens_before, n_app, dev, seed_offset):
        self.kvq, self.torch = kvq, torch
        B, H, Hq = len(lens_before), w.num_kv_heads, w.num_q_heads
        self.B, self.H, self.Hq, self.fmt = B, H, Hq, fmt
        lens_after = [int(t) + n_app for t in lens_before]
        fp8 = is_fp8(fmt)
        G = 1 if fp8 else fmt.G
        qmax = [split_tokens(t, fmt)[1] for t in lens_after]
        if fmt.fmt == "bf16":
            rows = max([1] + [t - min(t, fmt.S) for t in lens_after])
            self.cfg = kvq.make_config("bf16", H, 0, 0, 0, fmt.S, capacity_tokens=rows)
        elif w.paged:
            P = w.block_tokens
            nblk = [math.ceil(q / P) for q in qmax]
            mbps = max(nblk + [1])
            self.cfg = kvq.make_config(fmt.fmt, H, G, fmt.Gv, fmt.R, fmt.S, paged=True, block_tokens=P,
                                       num_blocks=max(1, sum(nblk)), max_blocks_per_seq=mbps, rope_base=fmt.rope_base,
                                       k_outliers=fmt.k_outliers, v_outliers=fmt.v_outliers)
        else:
            unit = 16 if fp8 else max(16, G)
            cap = max(unit, math.ceil(max(qmax) / unit) * unit)
            self.cfg = kvq.make_config(fmt.fmt, H, G, fmt.Gv, fmt.R, fmt.S, capacity_tokens=cap,
                                       rope_base=fmt.rope_base, k_outliers=fmt.k_outliers, v_outliers=fmt.v_outliers)
        self.cache = kvq.CacheLayer(self.cfg, B, device=dev, zero=False)
        if w.paged:
            perm = torch.from_numpy(I.block_permutation(w, max(1, sum(nblk)), l)).to(dev)
            table = torch.full((B, mbps), -1, dtype=torch.int32, device=dev)
            k = 0
            for b, nb in enumerate(nblk):
                table[b, :nb] = perm[k:k + nb]
                k += nb
            self.cache.block_table.copy_(table)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.lens_before = torch.tensor(lens_before, dtype=torch.int32, device=dev)
        self.lens_after = torch.tensor(lens_after, dtype=torch.int32, device=dev)
        self.n_app = n_app
        # build: the cache holds lens_before tokens; the step appends n_app more
        Tmax = max(lens_after)
        uniform = len(set(lens_after)) == 1
        if uniform:
            k, v = I.device_kv_bf16(w, l, Tmax, dev, batch=B, seed_offset=seed_offset)
            self._calibrate(fp8, fmt.fmt, k, v)
            Tb = lens_before[0]
            if Tb > 0:
                zero = torch.zeros(B, dtype=torch.int32, device=dev)
                kvq.quantize_append(self.cfg, self.cache.struct(), k[:, :, :Tb].contiguous(),
                                    v[:, :, :Tb].contiguous(), Tb, zero, B, self.status)
            self.k_new = k[:, :, Tb:Tb + n_app].contiguous()
            self.v_new = v[:, :, Tb:Tb + n_app].contiguous()
            del k, v
        else:
            if fp8:
                raise NotImplementedError("per-tensor FP8 calibration over ragged batches")
            self.k_new = torch.empty((B, H, n_app, 128), dtype=torch.bfloat16, device=dev)
            self.v_new = torch.empty_like(self.k_new)
            zero1 = torch.zeros(1, dtype=torch.int32, device=dev)
            for b in range(B):
                wb = dataclasses.replace(w, batch=1)
                k, v = I.device_kv_bf16(wb, l, lens_after[b], dev, batch=1, seed_offset=seed_offset + 7 * b)
                Tb = lens_before[b]
                kvq.quantize_append(self.cfg, self.cache.seq_struct(b), k[:, :, :Tb].contiguous(),
                                    v[:, :, :Tb].contiguous(), Tb, zero1, 1, self.status)
                self.k_new[b] = k[0, :, Tb:Tb + n_app]
                self.v_new[b] = v[0, :, Tb:Tb + n_app]
                del k, v
        self.q = I.device_q_bf16(w, l, dev, batch=B, seed_offset=seed_offset)
        self.nq = w.n_query
        qrows = (B, Hq) if self.nq == 1 else (B, self.nq, Hq)
        self.out = torch.empty(qrows + (128,), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(qrows, dtype=torch.float32, device=dev)
        self.wsb = kvq.decode_workspace_size_multi(self.cfg, B, self.nq, Hq)
        self.ws = torch.zeros(self.wsb, dtype=torch.uint8, device=dev)
        self.struct = self.cache.struct()
        self.scale = 1.0 / math.sqrt(128)

    def _calibrate(self, fp8, name, k, v):
        if fp8:
            self.kvq.fp8_calibrate(k, k.numel(), self.cache.k_tensor_scale, fmt=name)
            self.kvq.fp8_calibrate(v, v.numel(), self.cache.v_tensor_scale, fmt=name)

    def append(self, stream=None):
        self.kvq.quantize_append(self.cfg, self.struct, self.k_new, self.v_new, self.n_app, self.lens_before,
                                 self.B, self.status, stream)

    # FP8 layers without sink tokens take the step as one call and one launch
    # (kvq_append_decode_attention: the decode writes the token's codes itself)
    @property
    def fused(self):
        return is_fp8(self.fmt) and self.fmt.S == 0 and self.nq == 1 and self.n_app == 1

    def step_calls(self, stream=None):
        if self.fused:
            self.append_decode(stream)
        else:
            self.append(stream)
            self.decode(stream)

    def append_decode(self, stream=None):
        self.kvq.append_decode_attention(self.cfg, self.struct, self.k_new, self.v_new, self.lens_before, self.B,
                                         self.q, self.Hq, self.scale, self.out, True, self.lse, self.ws, self.wsb,
                                         self.status, stream)

    def decode(self, stream=None):
        # one launch: split pass with the log-sum-exp merge fused in (last CTA per pair)
        if self.nq == 1:
            self.kvq.decode_attention(self.cfg, self.struct, self.q, self.Hq, self.lens_after, self.B, self.scale,
                                      self.out, True, self.lse, self.ws, self.wsb, self.status, stream)
        else:  # the last nq appended tokens' queries, causal among them
            self.kvq.decode_attention_multi(self.cfg, self.struct, self.q, self.nq, self.Hq, self.lens_after, self.B,
                                            self.scale, self.out, True, self.lse, self.ws, self.wsb, self.status,
                                            stream)


def count_launches(w):
    # per layer: append (1 kernel) and decode (1 kernel, merge fused); FP8 layers without sink
    # tokens (one token, one query per step): one kernel, the append folded into the decode
    n = 0
    for f in w.layer_formats:
        n += 1 if (is_fp8(f) and f.S == 0 and w.n_query == 1 and max(1, w.append_tokens) == 1) else 2
    return n


def run_gpu(args, w, rank, world):
    import torch
    from quantized_kv_cache_decode_gb300 import kvq
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    n_app = max(1, w.append_tokens)
    lens_after = lens_after_step(w)
    lens_before = [int(t) - n_app for t in lens_after]
    sbytes = step_bytes(w, lens_after, n_app)
    replicas = args.replicas or max(1, min(4, math.ceil(3 * L2_BYTES / sbytes)))
    reps = []
    for rep in range(replicas):
        ids = getattr(w, "layer_ids", range(len(w.layer_formats)))
        reps.append([Layer(kvq, torch, w, l, f, lens_before, n_app, dev, seed_offset=1000 * rep + 17 * rank)
                     for l, f in zip(ids, w.layer_formats)])
    torch.cuda.synchronize()
    for rep in reps:
        for lay in rep:
            assert lay.status.item() == 0, f"device status {lay.status.item()} while building"
    dist = world > 1

    def barrier():
        if dist:
            torch.distributed.barrier()

    # The timed loop calls the library directly (append, then decode, per layer) with
    # events around each decode launch; the host issues a step's calls in well under the
    # step's device time, so the launches queue up and run back to back (measured on
    # GB300: 2.5 us per step less than replaying one CUDA graph per call).  --graphs
    # captures each layer's append and decode once into two graphs and replays them.
    for rep in reps:  # first calls outside capture (launch settings, shared-memory limits)
        for lay in rep:
            lay.step_calls()
    torch.cuda.synchronize()
    graphs = None
    if args.graphs:
        graphs = []
        for rep in reps:
            gl = []
            for lay in rep:
                ga, gd = (None if lay.fused else torch.cuda.CUDAGraph()), torch.cuda.CUDAGraph()
                if ga is not None:
                    with torch.cuda.graph(ga, capture_error_mode="relaxed"):
                        lay.append()
                with torch.cuda.graph(gd, capture_error_mode="relaxed"):
                    lay.append_decode() if lay.fused else lay.decode()
                gl.append((ga, gd))
            graphs.append(gl)
        torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step(i, ev=None):
        rep = reps[i % replicas]
        for j, lay in enumerate(rep):
            # events around the decode launch (fused layers: the one launch of the step)
            if graphs is not None:
                if graphs[i % replicas][j][0] is not None:
                    graphs[i % replicas][j][0].replay()
            elif not lay.fused:
                lay.append()
            if ev is not None:
                ev[0][j].record(stream)
            if graphs is not None:
                graphs[i % replicas][j][1].replay()
            elif lay.fused:
                lay.append_decode()
            else:
                lay.decode()
            if ev is not None:
                ev[1][j].record(stream)

    # the clock sampler starts first; the warm-up steps then run right before the timed ones, so
    # the GPU is not left idle (and its clocks low) between them
    clk = ClockSampler(dev.index if dev.index is not None else 0, os.path.join(OUT_DIR, f"clocks_rank{rank}.csv")) \
        if rank == 0 else None
    time.sleep(0.15 if clk else 0)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    # ---- timed region: exactly K steps, back to back (no event between two kernels: the library's
    # kernels are programmatically dependent launches, and an event in the stream would stop a
    # kernel from being scheduled during the tail of the one before it) ----
    K = args.steps
    nl = len(w.layer_formats)
    KP = min(K, 50)  # steps of the kernel pass (CUDA events around each decode launch)
    evs = [([torch.cuda.Event(enable_timing=True) for _ in range(nl)],
            [torch.cuda.Event(enable_timing=True) for _ in range(nl)]) for _ in range(KP)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    if args.profile_range:  # ncu --profile-from-start off then sees only the timed steps
        torch.cuda.profiler.start()
    t_start.record(stream)
    for i in range(K):
        step(args.warmup + i)
    t_end.record(stream)
    torch.cuda.synchronize()
    if args.profile_range:
        torch.cuda.profiler.stop()
    # ---- kernel pass: KP more steps with CUDA events around each decode launch (the roofline's
    # per-launch durations), right after the timed steps and inside the clock-sampled window ----
    for i in range(KP):
        step(args.warmup + K + i, evs[i])
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier()
    ms = t_start.elapsed_time(t_end)
    kern_ms = [[evs[i][0][j].elapsed_time(evs[i][1][j]) for j in range(nl)] for i in range(KP)]  # [step][layer]
    ms = max_over_ranks(ms, dev)
    ms_step = ms / K
    # ---- end to end through the public API, host buffers, copies inside the timed region ----
    E = args.e2e_steps or K
    rep0 = reps[0]

    def packed(tensors):
        # one device buffer holding the tensors (256-byte aligned slices); the returned
        # views replace them, so a step's inputs (outputs) move in one copy per layer
        sizes = [t.numel() * t.element_size() for t in tensors]
        offs, o = [], 0
        for n in sizes:
            offs.append(o)
            o += (n + 255) // 256 * 256
        buf = torch.empty(o, dtype=torch.uint8, device=dev)
        views = []
        for t, off, n in zip(tensors, offs, sizes):
            v = buf[off:off + n].view(t.dtype).view(t.shape)
            v.copy_(t)
            views.append(v)
        return buf, views, sum(sizes)

    # Two sets of device buffers, used by alternate steps, each holding the inputs (outputs) of all
    # the step's layers in one buffer: a step moves its inputs in with one copy and its results out
    # with one copy.  The copies run on their own stream, so the inputs of step i + 1 move to the
    # device while step i computes and the results of step i move back while step i + 1 computes;
    # every step's copies still lie inside the timed region.  The compute stream waits for them
    # once per step (its kernels then run back to back).
    sets = []  # [set] = (input buffer, output buffer, [layer] = (q, k_new, v_new, out, lse))
    for sidx in range(2):
        bi, vi, h2d = packed([t for lay in rep0 for t in (lay.q, lay.k_new, lay.v_new)])
        bo, vo, d2h = packed([t for lay in rep0 for t in (lay.out, lay.lse)])
        sets.append((bi, bo, [tuple(vi[3 * j:3 * j + 3]) + tuple(vo[2 * j:2 * j + 2]) for j in range(len(rep0))]))
    h_in = sets[0][0].cpu().pin_memory()
    h_out = [torch.empty(sets[s][1].shape, dtype=torch.uint8).pin_memory() for s in range(2)]
    copy_stream = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # a set's inputs are on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]  # a set's step has finished computing
    ev_out = [torch.cuda.Event() for _ in range(2)]   # a set's results are on the host
    compute = torch.cuda.current_stream()

    def copy_in(sidx):  # on the copy stream: the inputs of the next step that uses set sidx
        copy_stream.wait_event(ev_done[sidx])  # the set's last step has read its inputs
        sets[sidx][0].copy_(h_in, non_blocking=True)
        ev_in[sidx].record(copy_stream)

    def e2e_steps(n):
        # step i computes on set i % 2; after its kernels are queued, the copy stream moves the
        # inputs of step i + 1 in (they wait only for step i - 1, so they overlap step i's
        # kernels) and then step i's results out
        torch.cuda.set_stream(copy_stream)
        copy_in(0)
        for i in range(n):
            sidx = i % 2
            bi, bo, views = sets[sidx]
            torch.cuda.set_stream(compute)
            compute.wait_event(ev_in[sidx])
            compute.wait_event(ev_out[sidx])  # the set's last results have left its output buffer
            for lay, v in zip(rep0, views):
                lay.q, lay.k_new, lay.v_new, lay.out, lay.lse = v
                lay.step_calls(compute)
            ev_done[sidx].record(compute)
            torch.cuda.set_stream(copy_stream)
            if i + 1 < n:
                copy_in(1 - sidx)
            copy_stream.wait_event(ev_done[sidx])
            h_out[sidx].copy_(bo, non_blocking=True)
            ev_out[sidx].record(copy_stream)
        torch.cuda.set_stream(compute)

    e2e_steps(min(3, E))
    torch.cuda.synchronize()
    barrier()
    e0 = time.perf_counter()
    e2e_steps(E)
    torch.cuda.synchronize()
    e_ms = (time.perf_counter() - e0) * 1e3 / E
    e_ms = max_over_ranks(e_ms, dev)
    clocks = None
    if clk:
        clk.stop()
        clocks = clk.summary(wall0, wall1)
    for rep in reps:
        for lay in rep:
            assert lay.status.item() == 0, f"device status {lay.status.item()}"
    return dict(ms_step=ms_step, kern_ms=np.array(kern_ms), sbytes=sbytes,
                replicas=replicas, e2e_ms=e_ms, h2d=h2d, d2h=d2h, clocks=clocks, wall_ms=(wall1 - wall0) * 1e3,
                lens_after=lens_after, n_app=n_app)


# --------------------------------------------------------------------------- #
# CPU oracle (baseline and the reference arm)
# --------------------------------------------------------------------------- #


def lens_after_step(w):
    return I.seq_lens(w) + w.append_tokens if w.seq_len_range is not None else np.full(w.batch, w.seq_len)


def oracle_pairs(w, layer, pairs):
    """Host inputs and prebuilt oracle caches of the given (sequence, kv head) pairs of one layer."""
    from oracle import kvq_oracle as O
    fmt = w.layer_formats[layer]
    lens_after = lens_after_step(w)
    n_app = max(1, w.append_tokens)
    spec = O.Spec(fmt.fmt, d=128, G=1 if is_fp8(fmt) else fmt.G, Gv=fmt.Gv,
                  R=0 if is_fp8(fmt) else fmt.R, S=fmt.S, rope_base=fmt.rope_base, k_outliers=fmt.k_outliers,
                  v_outliers=fmt.v_outliers)
    q = O.bf16_to_f32(I.q_bf16(w, layer))
    items = []
    for b, h in pairs:
        T = int(lens_after[b])
        k, v = I.kv_bf16(w, layer, b, h, T)
        kf, vf = O.bf16_to_f32(k), O.bf16_to_f32(v)
        ks = O.fp8_tensor_scale(kf, spec.fmt) if spec.is_fp8 else None
        vs = O.fp8_tensor_scale(vf, spec.fmt) if spec.is_fp8 else None
        hc = O.build_head_cache(kf[:T - n_app], vf[:T - n_app], spec, ks, vs)
        qh = q[b, h * w.gqa:(h + 1) * w.gqa] if w.n_query == 1 else q[b, :, h * w.gqa:(h + 1) * w.gqa]
        items.append((b, h, T, hc, kf[T - n_app:], vf[T - n_app:], qh.reshape(-1, 128)))
    return O, items, n_app


def oracle_step(O, items, n_query=1):
    """One oracle decode step over the sample: append the new tokens, attend for the g heads
    (of each of the n_query query tokens, over its causal prefix)."""
    import copy
    for (b, h, T, hc, kn, vn, qh) in items:
        c = copy.copy(hc)
        for t in range(len(kn)):
            O.append_token(c, kn[t], vn[t])
        kh, vh = O.dequantized_f64(c)
        per = qh.shape[0] // n_query  # query heads of the pair (rows: query token major)
        for j in range(qh.shape[0]):
            n = T - n_query + j // per + 1
            O.attend_head(qh[j], kh[:n], vh[:n], 1.0 / math.sqrt(128))


def sample_bytes(w, layer, items, n_app):
    fmt = w.layer_formats[layer]
    tot = 0
    for (b, h, T, hc, kn, vn, qh) in items:
        tot += attention_bytes(fmt, T, 1) + append_bytes(fmt, T - n_app, n_app, 1)
        tot += qh.shape[0] * (128 * 2 * 2 + 4)
    return tot


def sample_pairs(w, layer, token_budget):
    """(sequence, kv head) pairs of one layer in a seeded random order (so the sample follows the
    workload's length mix), as many as hold about ``token_budget`` cached tokens (at least one)."""
    lens_after = lens_after_step(w)
    rng = np.random.default_rng(w.seed * 31 + layer)
    order = rng.permutation(w.batch * w.num_kv_heads)
    out, tok = [], 0
    for u in order:
        b, h = divmod(int(u), w.num_kv_heads)
        out.append((b, h))
        tok += int(lens_after[b])
        if tok >= token_budget:
            break
    return out


def _oracle_worker(wname, layer, pairs, barrier, results):
    """One CPU worker (its own process, one numpy thread): build its pairs' oracle caches, wait for
    every worker, then time one oracle step over them."""
    w = I.WORKLOADS[wname]()
    O, items, n_app = oracle_pairs(w, layer, pairs)
    barrier.wait()
    t0 = time.time()
    oracle_step(O, items, w.n_query)
    t1 = time.time()
    results.put((sample_bytes(w, layer, items, n_app), t0, t1, len(items)))


def time_oracle_parallel(w, layer, pairs, workers):
    """GB/s of the oracle over ``pairs`` spread over ``workers`` processes (spawned, so safe after the
    GPU run): the sample's bytes over the span from the first worker's start to the last one's end."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    workers = max(1, min(workers, len(pairs)))
    # deal the pairs so each worker gets a similar number of tokens (longest first)
    lens_after = lens_after_step(w)
    order = sorted(pairs, key=lambda bh: -int(lens_after[bh[0]]))
    shares, load = [[] for _ in range(workers)], [0] * workers
    for bh in order:
        i = int(np.argmin(load))
        shares[i].append(bh)
        load[i] += int(lens_after[bh[0]])
    barrier = ctx.Barrier(workers)
    results = ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(w.name, layer, sh, barrier, results)) for sh in shares]
    for p in procs:
        p.start()
    got = [results.get() for _ in procs]
    for p in procs:
        p.join()
    nbytes = sum(g[0] for g in got)
    span = max(g[2] for g in got) - min(g[1] for g in got)
    return nbytes / span / 1e9, span, sum(g[3] for g in got)


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            txt = f.read()
        for key in ("model name", "Model"):
            for line in txt.splitlines():
                if line.split(":")[0].strip() == key:
                    return f"{key}: {line.split(':', 1)[1].strip()}"
        # Arm cores name themselves only by implementer and part number (MIDR fields)
        fields = {}
        for line in txt.splitlines():
            k, _, v = line.partition(":")
            fields.setdefault(k.strip(), v.strip())
        arm_parts = {"0xd40": "Arm Neoverse V1", "0xd49": "Arm Neoverse N2", "0xd4f": "Arm Neoverse V2 (as in NVIDIA Grace)",
                     "0xd0c": "Arm Neoverse N1", "0xd8e": "Arm Neoverse N3", "0xd84": "Arm Neoverse V3"}
        part = fields.get("CPU part")
        if part:
            name = arm_parts.get(part.lower()) if fields.get("CPU implementer", "").lower() == "0x41" else None
            return f"{name} (CPU part {part})" if name else f"CPU part: {part}"
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def parity_layers(w):
    """The layers the oracle is timed on: all of a one-layer workload, else the first, a middle and the
    last layer (for the paged mix: INT8, INT4, INT8)."""
    n = len(w.layer_formats)
    return sorted({0, n // 2 - 1 if n > 2 else 0, n - 1})


def cpu_baseline(w, token_budget=400000):
    """The oracle on the host cores, 1 thread and every core, on a bounded sample of each parity layer;
    the whole-step figure is extrapolated from the per-format rates (stated as such)."""
    nproc = os.cpu_count() or 1
    legs = []
    lens_after = lens_after_step(w)
    n_app = max(1, w.append_tokens)
    for workers in (1, nproc):
        per_layer = []
        rate = {}
        for layer in parity_layers(w):
            fmt = w.layer_formats[layer].fmt
            pairs = sample_pairs(w, layer, token_budget * workers)
            gbs, span, n = time_oracle_parallel(w, layer, pairs, workers)
            per_layer.append({"layer": layer, "format": fmt, "pairs": n, "of_pairs": w.batch * w.num_kv_heads,
                              "GB_per_s": round(gbs, 5), "timed_s": round(span, 2)})
            rate.setdefault(fmt, []).append(gbs)
        # every layer of the step at its format's measured rate
        t = 0.0
        tot = 0
        for f in w.layer_formats:
            lb = sum(attention_bytes(f, int(T), w.num_kv_heads) +
                     append_bytes(f, int(T) - n_app, n_app, w.num_kv_heads) for T in lens_after)
            lb += len(lens_after) * w.n_query * w.num_q_heads * (128 * 2 * 2 + 4)
            tot += lb
            t += lb / (float(np.mean(rate[f.fmt])) * 1e9)
        legs.append({"cores": workers, "value": round(tot / t / 1e9, 5), "unit": "GB/s", "step_s": round(t, 2),
                     "extrapolated": len(w.layer_formats) > len(parity_layers(w)), "per_layer": per_layer})
    best = legs[-1]
    layers = ", ".join(str(x) for x in parity_layers(w))
    return {"value": best["value"], "unit": "GB/s", "cores": best["cores"], "kind": "oracle",
            "sample": f"layer(s) {layers}: a seeded random sample of (sequence, kv head) pairs holding about "
                      f"{token_budget} cached tokens per worker, append + attention, numpy fp64, one thread per "
                      f"worker process; " + ("whole-step figure extrapolated from the per-format rates"
                                             if best["extrapolated"] else "the whole step is that layer"),
            "cpu_model": cpu_model(), "nproc": nproc, "legs": legs}


def run_reference(args, w, rank, world):
    if rank != 0:
        return None
    # a step = the oracle (one thread) over a bounded sample of layer 0's pairs, sized to ~1 s
    first = sample_pairs(w, 0, 1)
    O, items, n_app = oracle_pairs(w, 0, first)
    t0 = time.perf_counter()
    oracle_step(O, items, w.n_query)
    per_tok = max(1e-9, (time.perf_counter() - t0) / items[0][2])
    pairs = sample_pairs(w, 0, int(1.0 / per_tok))
    O, sample, n_app = oracle_pairs(w, 0, pairs)
    for _ in range(args.warmup):
        oracle_step(O, sample, w.n_query)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(O, sample, w.n_query)
    dt = (time.perf_counter() - t0) / args.steps
    gbs = sample_bytes(w, 0, sample, n_app) / dt / 1e9
    return gbs, dt, len(sample)


# --------------------------------------------------------------------------- #


def _code_only(text: str) -> str:
    """C/C++/CUDA source without its comments and blank space (string literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"' or c == "'":  # literal: copy through its closing quote
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_sources_sha256() -> str:
    """Hash of the code of the library's CUDA sources, comments and blank space left out (decides
    whether a recorded ncu traffic figure still applies: a comment edit does not change a kernel)."""
    import hashlib
    h = hashlib.sha256()
    src = os.path.join(ROOT, "quantized_kv_cache_decode_gb300", "csrc")
    for name in sorted(os.listdir(src)):
        if name.endswith((".cu", ".cuh", ".h", ".cpp")):
            with open(os.path.join(src, name), encoding="utf-8") as f:
                h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(I.WORKLOADS))
    ap.add_argument("--replicas", type=int, default=0, help="cache copies cycled to defeat L2 (0: auto)")
    ap.add_argument("--e2e-steps", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graphs", action="store_true",
                    help="replay per-layer CUDA graphs of the library calls instead of calling the library directly")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers of the workload (profiling captures; 0: all)")
    ap.add_argument("--only-layers", default="",
                    help="comma-separated layer indices to run (profiling captures of chosen layers)")
    ap.add_argument("--profile-range", action="store_true",
                    help="bracket the timed steps with cudaProfilerStart/Stop (for ncu --profile-from-start off)")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    w = I.WORKLOADS[args.workload]()
    if args.layers:
        w.layer_formats = w.layer_formats[:args.layers]
    if args.only_layers:
        ids = [int(x) for x in args.only_layers.split(",")]
        w.layer_formats = [w.layer_formats[i] for i in ids]
        w.layer_ids = ids
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    config = {"workload": w.name, "layers": len(w.layer_formats), "batch": w.batch, "q_heads": w.num_q_heads,
              "kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
              "seq_len": w.seq_len if w.seq_len else f"log-uniform {tuple(w.seq_len_range)}",
              "formats": sorted({f.fmt for f in w.layer_formats}), "append_tokens_per_step": max(1, w.append_tokens), "query_tokens_per_step": w.n_query,
              "paged": w.paged}
    metric = "effective KV GB/s (quantized decode step)"

    if args.impl == "reference":
        r = run_reference(args, w, rank, world)
        if rank == 0:
            gbs, dt, n = r
            cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                   "sample": f"layer 0, {n} (sequence, kv head) pairs per step (seeded random order), "
                             f"append + attention, numpy fp64, one thread", "cpu_model": cpu_model()}
            line = {"impl": "reference", "metric": metric, "value": round(gbs, 4), "unit": "GB/s",
                    "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                    "data": "synthetic", "config": config, "cpu_baseline": cpu,
                    "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}
            print(json.dumps(line))
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", int(os.environ["LOCAL_RANK"])))
    os.makedirs(OUT_DIR, exist_ok=True)
    r = run_gpu(args, w, rank, world)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return
    gbs = job_throughput(r["sbytes"], r["ms_step"], world)
    # roofline of the decode kernel: algorithmic bytes of each layer's launch (codes, scales and
    # zero-points, bf16 sink/residual, q, bf16 out, lse) over that launch's CUDA-event duration
    B = len(r["lens_after"])
    # a fused layer's launch (FP8, no sink tokens) also reads the step's K, V rows (bf16) and
    # writes their codes (1 byte each)
    fused = [is_fp8(f) and f.S == 0 and w.n_query == 1 and max(1, w.append_tokens) == 1 for f in w.layer_formats]
    layer_bytes = np.array([sum(attention_bytes(f, int(T), w.num_kv_heads) for T in r["lens_after"]) +
                            B * w.n_query * w.num_q_heads * (128 * 2 * 2 + 4) +
                            (B * w.num_kv_heads * 128 * (2 * 2 + 2) if fz else 0)
                            for f, fz in zip(w.layer_formats, fused)], float)
    km = r["kern_ms"]  # [steps][layers] ms
    kern_gbs = layer_bytes.sum() / (km.sum(axis=1).mean() * 1e-3) / 1e9
    by_format = {}
    for fname in sorted({f.fmt for f in w.layer_formats}):
        idx = [j for j, f in enumerate(w.layer_formats) if f.fmt == fname]
        t = km[:, idx]
        a = layer_bytes[idx].sum() / (t.sum(axis=1).mean() * 1e-3) / 1e9
        by_format[fname] = {"layers": len(idx), "achieved": round(a, 1), "frac": round(a / hbm_peak, 4),
                            "bytes_per_launch": int(layer_bytes[idx].mean()),
                            "mean_launch_us": round(float(t.mean()) * 1e3, 2),
                            "median_launch_us": round(float(np.median(t)) * 1e3, 2)}
    # DRAM bytes per decode launch from an ncu capture, used only while the kernel sources are
    # the ones the capture ran (their hash is recorded beside the figure)
    traffic = None
    tpath = os.path.join(ROOT, "profiles", f"traffic_{w.name}.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            rec = json.load(f)
        if rec.get("kernel_sources_sha256") == kernel_sources_sha256():
            per_fmt = rec.get("bytes_per_launch_by_format")
            if per_fmt:  # the step's launches, averaged, each at its format's captured figure
                if all(f.fmt in per_fmt for f in w.layer_formats):
                    traffic = int(np.mean([per_fmt[f.fmt] for f in w.layer_formats]))
            else:
                traffic = rec.get("bytes_per_launch")
    line = {
        "metric": metric, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(r["ms_step"], 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16/f32 (fp8/int codes)", "data": "synthetic",
        "config": {**config, "l2": f"{r['replicas']} rotating cache copies, {r['replicas'] * r['sbytes'] / 1e6:.0f} MB"
                   f" cycled (L2 {L2_BYTES / 2 ** 20:.0f} MiB)", "bytes_per_step": r["sbytes"],
                   "launch": "direct library calls" if not args.graphs else
                   "per-layer CUDA graphs of the library calls (append, decode), replayed"},
        "pct_hbm_peak": round(100 * gbs / world / hbm_peak, 2),
        "tokens_per_s": round(len(r["lens_after"]) * world / (r["ms_step"] * 1e-3), 1),
        "roofline": {"bound": "hbm", "achieved": round(kern_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(kern_gbs / hbm_peak, 4), "traffic": traffic,
                     "kernel": "decode_kernel (fused merge; FP8 without sinks: the append folded in)", "peak_source": peak_src,
                     "bytes_per_launch": int(layer_bytes.mean()),
                     "mean_launch_us": round(float(km.mean()) * 1e3, 2),
                     "median_launch_us": round(float(np.median(km)) * 1e3, 2),
                     "min_launch_us": round(float(np.min(km)) * 1e3, 2),
                     "max_launch_us": round(float(np.max(km)) * 1e3, 2),
                     "launches_timed": int(km.size), "by_format": by_format,
                     "timing": "CUDA events around each decode launch over a kernel pass of min(K, 50) steps run "
                               "right after the K timed steps (which run back to back without events)"},
        "e2e": {"value": round(job_throughput(r["sbytes"], r["e2e_ms"], world), 2), "unit": "GB/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "ms_per_step": round(r["e2e_ms"], 4)},
        "gpu_launches": count_launches(w) * args.steps,
        "clocks": r["clocks"],
        "wall_ms_timed": round(r["wall_ms"], 2),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line))


if __name__ == "__main__":
    main()
