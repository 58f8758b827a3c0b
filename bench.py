"""Throughput of packed blockwise attention on GB300, as one JSON line.

A step is one sp_packed_attention call (set-up kernel + persistent attention
kernel) over the whole chunk schedule of the benchmark workload: the Llama-style
GQA layer (32 query / 8 key-value heads, d = 128, 32K tokens in one document,
causal, 8 virtual ranks in zigzag order), bf16 inputs resident in HBM.
FLOP = 4 * d * Hq * (valid query-key pairs).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun the virtual sequence-parallel ranks are split over the GPUs
(default, `--split ranks`): GPU g runs the schedule items of the virtual ranks
r with r mod N = g (their Q chunks against the K/V chunks their steps visit),
with K and V resident on every GPU before the timed region, so no data crosses
GPUs inside it; `value` is the whole workload's FLOP over the slowest GPU's
time (strong scaling). `--split replicas` runs an independent full copy per GPU
(weak scaling). The timed region is bracketed by a barrier and device
synchronisation, and its maximum over ranks is reported. With N = 1 the line
also carries `per_workload`: forward (and backward) time of every workload.
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "packed causal attention TFLOP/s (valid pairs) on 1 GB300 and % of bf16 peak"
L2_BYTES = 129 * 1024 * 1024
WORKLOAD_INDEX = 1  # the Llama-style layer the metric is quoted on


def valid_pairs(cu, causal: bool) -> int:
    lens = np.diff(np.asarray(cu, dtype=np.int64))
    if causal:
        return int(np.sum(lens * (lens + 1) // 2))
    return int(np.sum(lens * lens))


def sched_name(kind: int) -> str:
    return {0: "ring", 1: "zigzag", 2: "tasp"}[kind]


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]), "hbm_gbs": float(p["hbm_gbs"]),
                "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "source": "fallback"}


def fwd_kernel_name(w):
    """The forward kernel the library runs for a workload: CTA pairs (two query
    heads of one key/value head per cluster) when d = 128 and Hq / Hkv is even,
    else one CTA per unit."""
    if w.d == 128 and (w.Hq // w.Hkv) % 2 == 0:
        return "attn_tc_pair_kernel<0> (cluster of 2, tcgen05 cta_group::2)"
    return f"attn_tc_kernel<{w.d},0>"


def kernel_traffic():
    """DRAM bytes per launch of the attention kernel from the committed ncu
    summary, if it was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "attn_tc_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        for src in rec["kernel_sources"]:
            h.update(open(os.path.join(ROOT, src), "rb").read())
        if rec.get("kernel_sources_sha256") == h.hexdigest():
            return float(rec["traffic_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def dist_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_gather(x: float, world: int) -> list:
    """Every rank's value of x, in rank order."""
    if world == 1:
        return [x]
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    out = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(out, t)
    return [float(o.item()) for o in out]


# ------------------------------------------------------------------ CPU oracle

def oracle_sample(w, cu, seconds: float, seed: int = 0):
    """Runs the fp64 oracle on random query rows of workload w (all heads),
    growing the sample until it has run for about `seconds`. Inputs are drawn
    on the CPU with the workload's generator for the keys the rows need.
    Returns (flop, elapsed_s, n_rows, threads)."""
    import torch
    import oracle
    from sequence_blockwise_gb300 import workloads as wl
    rng = np.random.default_rng(seed)
    oracle.build()
    # Inputs: the same seeded recipe on the CPU.
    q, k, v = wl.make_qkv(w, "cpu")
    conv = (lambda t: wl.bf16_bits(t)) if w.dtype == "bf16" else (lambda t: t.numpy())
    kh, vh = conv(k), conv(v)
    threads = os.cpu_count() or 1
    flop, elapsed, nrows = 0, 0.0, 0
    batch = 16
    while elapsed < seconds:
        rows = np.sort(rng.integers(0, w.T, size=batch)).astype(np.int32)
        qr = conv(q[torch.from_numpy(rows.astype(np.int64))])
        lens = np.diff(cu)
        doc = np.searchsorted(cu, rows, side="right") - 1
        keys = (rows - cu[doc] + 1) if w.causal else lens[doc]
        t0 = time.perf_counter()
        oracle.attn(qr, kh, vh, cu, w.causal, rows=rows, q_rows_only=True, threads=threads)
        elapsed += time.perf_counter() - t0
        flop += int(4 * w.d * w.Hq * int(np.sum(keys)))
        nrows += batch
        batch = min(batch * 2, 1024)
    return flop, elapsed, nrows, threads


# ------------------------------------------------------------------ SP split

def split_items(items, world: int, gpu: int):
    """The schedule items GPU `gpu` of `world` runs: those of the virtual ranks
    r with r mod world == gpu (each virtual rank's Q chunk and its chunk-visit
    steps stay on one GPU, as a sequence-parallel rank's do). Returns the item
    rows in schedule order."""
    items = np.asarray(items)
    return np.ascontiguousarray(items[(items[:, 0] % world) == gpu])


def row_intervals(items):
    """The union of the items' Q ranges as sorted, disjoint [a, b) intervals:
    the output rows a GPU writes."""
    spans = sorted({(int(it[3]), int(it[4])) for it in np.asarray(items)})
    out = []
    for a, b in spans:
        if out and a <= out[-1][1]:
            out[-1][1] = max(out[-1][1], b)
        else:
            out.append([a, b])
    return [(a, b) for a, b in out]


def owned_chunks(kind: int, P: int, T: int, rank: int):
    """The Q chunks virtual rank `rank` owns (equal chunking): RING and TASP,
    chunk r of P (the first T mod P get one more token); ZIGZAG, chunks r and
    2P-1-r of 2P equal chunks."""
    if kind == 1:  # zigzag
        c = T // (2 * P)
        return sorted([(rank * c, (rank + 1) * c), ((2 * P - 1 - rank) * c, (2 * P - rank) * c)])
    base, extra = divmod(T, P)
    a = rank * base + min(rank, extra)
    return [(a, a + base + (1 if rank < extra else 0))]


# ------------------------------------------------------------------ tile work

def tile_work(items, cu, causal: bool, T: int, rows_per_unit: int = 256):
    """Executed (query, key) tile area of the tensor-core forward for one query
    head, from the same walk the kernels do: items grouped by (rank, Q range);
    each unit is two 128-row Q tiles; an item's key range is clipped to the keys
    some row of the unit may attend (its rows' documents; up to its last row
    when causal) and walked in 128-key tiles from the clipped start; when some
    group holds items that are not whole 128-key tiles long, every group walks
    its items in key order and joins contiguous clipped ranges; a (Q tile, key
    tile) pair costs 128 x 128 unless it holds no valid pair for the tile's rows
    (skipped). Divided by the valid pairs, this is the forward's tile work."""
    items = np.asarray(items)
    cu = np.asarray(cu, dtype=np.int64)
    doc = lambda t: int(np.searchsorted(cu, t, side="right") - 1)
    groups, start = [], 0
    for i in range(1, len(items) + 1):
        if i == len(items) or tuple(items[i, [0, 3, 4]]) != tuple(items[start, [0, 3, 4]]):
            groups.append((start, i))
            start = i
    ordered = any(((items[a:b, 6] - items[a:b, 5]) % 128 != 0).any() and b - a <= 2048 for a, b in groups)
    work = 0
    for a, b in groups:
        g = items[a:b]
        if ordered and ((g[:, 6] - g[:, 5]) % 128 != 0).any() and b - a <= 2048:
            g = g[np.argsort(g[:, 5], kind="stable")]
        q_lo, q_hi = int(g[0, 3]), int(g[0, 4])
        for q0 in range(q_lo, q_hi, rows_per_unit):
            tiles = []
            for i in range(2):
                qa, qb = q0 + 128 * i, min(q0 + 128 * (i + 1), q_hi)
                if qa < qb:
                    tiles.append((qa, qb, int(cu[doc(qa)]), int(cu[doc(qb - 1) + 1])))
            if not tiles:
                continue
            lo, hi = tiles[0][2], tiles[-1][3]
            if causal:
                hi = min(hi, tiles[-1][1])
            ranges, j = [], 0
            while j < len(g):
                k0, k1 = max(int(g[j, 5]), lo), min(int(g[j, 6]), hi)
                j += 1
                while ordered and k0 < k1 and j < len(g):
                    n0, n1 = max(int(g[j, 5]), lo), min(int(g[j, 6]), hi)
                    if n0 != k1 or n1 <= n0:
                        break
                    k1 = n1
                    j += 1
                if k0 < k1:
                    ranges.append((k0, k1))
            for k0, k1 in ranges:
                ka = np.arange(k0, k1, 128, dtype=np.int64)
                kb = np.minimum(ka + 128, k1)
                for qa, qb, ds, de in tiles:
                    skip = (de <= ka) | (kb <= ds)
                    if causal:
                        skip |= ka > qb - 1
                    work += int((~skip).sum()) * 128 * 128
    return work


# ------------------------------------------------------------------ GPU arm

def run_ours(args, world, rank, local):
    import torch
    import sequence_blockwise_gb300 as sb
    from sequence_blockwise_gb300 import workloads as wl

    w = wl.WORKLOADS[WORKLOAD_INDEX]
    cu = wl.cu_seqlens(w)
    pairs = valid_pairs(cu, w.causal)
    flop = 4.0 * w.d * w.Hq * pairs
    dev = torch.device("cuda", local)
    q, k, v = wl.make_qkv(w, dev)
    att = sb.PackedAttention(cu, w.causal, w.kind, w.P, w.Hq, seed=w.seed, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.Hq, w.T), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # Sequence-parallel split (default): GPU g runs the items of the virtual
    # ranks r with r mod N = g, i.e. their Q chunks against the K/V chunks their
    # schedule visits; K and V are resident on every GPU before the timed
    # region, so nothing crosses GPUs inside it. With N = 1 that is the whole
    # schedule. --split replicas runs an independent full copy per GPU.
    split = "replicas" if (world > 1 and args.split == "replicas") else "ranks"
    my_items = split_items(att.items, world, rank) if split == "ranks" else att.items
    n_my = int(len(my_items))
    my_intervals = row_intervals(my_items) if n_my else []
    my_flop = 4.0 * w.d * w.Hq * sum(valid_pairs_range(cu, w.causal, it) for it in my_items)
    my_items_dev = torch.from_numpy(np.ascontiguousarray(my_items)).to(dev) if n_my else None
    my_ws = torch.empty(sb.sp_packed_attention_workspace_size(max(n_my, 1)), dtype=torch.uint8, device=dev)
    launches_per_step = 2 if n_my else 0  # set-up kernel + persistent attention kernel

    def step():
        if n_my:
            sb.sp_packed_attention(q, k, v, o, lse, att.cu_dev, w.causal, my_items_dev, my_ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    sb.sp_check_device_status(stream)

    # ---- device-resident timed region
    clocks = ClockSampler(local)
    time.sleep(0.3)
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    dist_barrier(world)
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    per = [a.elapsed_time(b) for a, b in ev]
    sb.sp_check_device_status(stream)
    gpu_ms = dist_gather(total_ms / args.steps, world)
    total_ms = dist_max(total_ms, world)
    ms_step = total_ms / args.steps
    job_flop = flop if split == "ranks" else world * flop
    value = job_flop * args.steps / (total_ms * 1e-3) / 1e12

    # ---- end to end through the C-ABI with host buffers: every step copies its
    # inputs (Q, K, V, cu_seqlens, items) from pinned host memory and reads its O
    # and LSE back into pinned host memory. Steps are pipelined as a serving
    # loop would run them: step i+1's inputs travel on one copy stream and step
    # i-1's outputs on another while step i computes, with two sets of device
    # buffers.
    qh = q.cpu().pin_memory()
    kh = k.cpu().pin_memory()
    vh = v.cpu().pin_memory()
    cu_h = torch.from_numpy(cu).pin_memory()
    it_h = torch.from_numpy(att.items).pin_memory()
    oh = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
    lh = [torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True) for _ in range(2)]
    qd = [torch.empty_like(q) for _ in range(2)]
    kd = [torch.empty_like(k) for _ in range(2)]
    vd = [torch.empty_like(v) for _ in range(2)]
    od = [torch.empty_like(o) for _ in range(2)]
    ld = [torch.empty_like(lse) for _ in range(2)]
    cud = [torch.empty_like(att.cu_dev) for _ in range(2)]
    itd = [torch.empty_like(att.items_dev) for _ in range(2)]  # holds this GPU's items at the front
    it_h = torch.from_numpy(np.ascontiguousarray(my_items)).pin_memory() if n_my else it_h
    row_bytes = w.Hq * w.d * q.element_size()
    my_rows = sum(b - a for a, b in my_intervals)
    # Per step: this GPU's Q rows, all of K and V, cu_seqlens and its items in;
    # its O rows and the LSE out.
    h2d = (my_rows * row_bytes + kh.numel() * kh.element_size() + vh.numel() * vh.element_size() +
           cu_h.numel() * 4 + (it_h.numel() * 4 if n_my else 0))
    d2h = my_rows * row_bytes + lh[0].numel() * lh[0].element_size()
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n_steps, start_ev):
        s_in.wait_event(start_ev)
        for i in range(n_steps):
            sl = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[sl])  # step i-2 has finished reading this slot
                for a, b in my_intervals:
                    qd[sl][a:b].copy_(qh[a:b], non_blocking=True)
                kd[sl].copy_(kh, non_blocking=True)
                vd[sl].copy_(vh, non_blocking=True)
                cud[sl].copy_(cu_h, non_blocking=True)
                if n_my:
                    itd[sl][:n_my].copy_(it_h, non_blocking=True)
                ev_in[sl].record(s_in)
            stream.wait_event(ev_in[sl])
            if i >= 2:
                stream.wait_event(ev_out[sl])  # step i-2's outputs have left this slot
            if n_my:
                sb.sp_packed_attention(qd[sl], kd[sl], vd[sl], od[sl], ld[sl], cud[sl], w.causal,
                                       itd[sl][:n_my], my_ws, stream=stream)
            ev_comp[sl].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[sl])
                for a, b in my_intervals:
                    oh[sl][a:b].copy_(od[sl][a:b], non_blocking=True)
                lh[sl].copy_(ld[sl], non_blocking=True)
                ev_out[sl].record(s_out)
        for sl in range(min(2, n_steps)):
            stream.wait_event(ev_out[sl])

    warm = torch.cuda.Event()
    warm.record(stream)
    e2e_run(2, warm)
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps, e0)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    dist_barrier(world)
    e2e_ms = dist_max(e0.elapsed_time(e1), world)
    e2e_value = job_flop * args.steps / (e2e_ms * 1e-3) / 1e12
    sb.sp_check_device_status(stream)
    # The pipelined result equals the device-resident one on this GPU's rows.
    e2e_same = True
    if args.steps > 0:
        o_cpu, last = o.cpu(), oh[(args.steps - 1) % 2]
        e2e_same = all(bool(torch.equal(last[a:b], o_cpu[a:b])) for a, b in my_intervals)

    # ---- backward of the same call (dQ, dK, dV), timed on its own after the
    # forward's timed region; reported beside the headline, not in `value`.
    bwd = None
    if not args.no_backward and world == 1:
        dout = wl.random_normal((w.T, w.Hq, w.d), w.seed + 99, dev, "bf16")
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        att(q, k, v, o, lse, stream=stream)

        def bstep():
            att.backward(q, k, v, o, lse, dout, dq, dk, dv, stream=stream)

        for _ in range(max(args.warmup, 3)):
            bstep()
        torch.cuda.synchronize(dev)
        # The timed backward starts, like the headline's forward region, from a
        # GPU that has idled for a moment (the end-to-end region just before it
        # ran at the power cap), and its clocks are recorded beside it.
        time.sleep(1.0)
        bclocks = ClockSampler(local)
        time.sleep(0.3)
        bev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i in range(args.steps):
            bev[i][0].record(stream)
            bstep()
            bev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        bclk = bclocks.stop()
        sb.sp_check_device_status(stream)
        bper = [a.elapsed_time(b) for a, b in bev]
        b_ms = dist_max(sum(bper) / len(bper), world)
        bflop = 2.5 * flop  # QK^T and dO V^T recomputed, dV, dK, dQ: 10 d per pair and head
        bwd = {"ms_per_call": round(b_ms, 4), "tflops": round(bflop / (b_ms * 1e-3) / 1e12, 2),
               "flop_per_call": bflop, "flop_convention": "10*d*Hq*valid_pairs (2.5x forward)",
               "frac_of_peak": None, "launches_per_call": 3,
               "kernels": "bwd_rowdot_kernel, bwd_fused_kernel<128>, bwd_dq_convert_kernel",
               "clocks": bclk}
        del dout, dq, dk, dv

    # ---- secondary: the log-sum-exp merge kernel of the unfused API path,
    # bandwidth bound (12 bytes per O element + 12 per LSE word). Shape of the
    # 64K full-mask layer's partials over all rows at once, so that the three
    # fp32 O arrays (512 MB each) are far larger than L2.
    merge = None
    if not args.no_backward and world == 1:
        wm = wl.WORKLOADS[3]
        rows, Hm, dm = wm.T, wm.Hq, wm.d
        o_acc = torch.randn((rows, Hm, dm), dtype=torch.float32, device=dev)
        o_part = torch.randn((rows, Hm, dm), dtype=torch.float32, device=dev)
        l_acc = torch.randn((Hm, rows), dtype=torch.float32, device=dev)
        l_part = torch.randn((Hm, rows), dtype=torch.float32, device=dev)
        for _ in range(3):
            sb.sp_lse_merge(o_acc, l_acc, o_part, l_part, stream=stream)
        torch.cuda.synchronize(dev)
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_m = 10
        m0.record(stream)
        for _ in range(n_m):
            sb.sp_lse_merge(o_acc, l_acc, o_part, l_part, stream=stream)
        m1.record(stream)
        torch.cuda.synchronize(dev)
        sb.sp_check_device_status(stream)
        m_ms = m0.elapsed_time(m1) / n_m
        m_bytes = 12 * o_acc.numel() + 12 * l_acc.numel()
        merge = {"kernel": "lse_merge_kernel", "bound": "hbm", "achieved": round(m_bytes / (m_ms * 1e-3) / 1e9, 1),
                 "unit": "GB/s", "bytes_per_call": int(m_bytes), "ms_per_call": round(m_ms, 4),
                 "shape": f"partials [{rows}, {Hm}, {dm}] fp32 + LSE [{Hm}, {rows}] ({wm.name})"}
        del o_acc, o_part, l_acc, l_part

    peaks = read_peaks()
    if merge is not None:
        merge["peak"] = peaks["hbm_gbs"]
        merge["frac"] = round(merge["achieved"] / peaks["hbm_gbs"], 4)
    if bwd is not None:
        bwd["frac_of_peak"] = round(bwd["tflops"] / peaks["bf16_tflops"], 4)
    avg_launch_ms = sum(per) / len(per)
    achieved = my_flop / (avg_launch_ms * 1e-3) / 1e12 if avg_launch_ms > 0 else 0.0
    traffic = kernel_traffic()
    # Bytes one GPU's step touches: its Q and O rows, all of K and V, the LSE.
    my_rows = sum(b - a for a, b in my_intervals)
    io_bytes = (2 * my_rows * w.Hq * w.d + k.numel() + v.numel()) * 2 + lse.numel() * 4

    result = None
    if rank == 0:
        result = {
            "metric": METRIC,
            "value": round(value, 3),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": max(args.warmup, 3),
            "ms_per_step": round(ms_step, 4),
            "higher_is_better": True,
            "scaling": "strong" if split == "ranks" else "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) Q/K/V rounded to bf16; no dataset or weights)",
            "config": {
                "workload": w.name, "T": w.T, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                "causal": w.causal, "docs": int(len(cu) - 1), "schedule": sched_name(w.kind),
                "P_virtual": w.P, "n_items": int(len(att.items)), "valid_pairs": pairs,
                "flop_per_step": job_flop,
                "parallelism": (f"sp split x{world}: GPU g runs the virtual ranks r with r mod {world} = g "
                                "(their Q chunks and chunk-visit steps); K/V resident on every GPU; "
                                "no collective" if split == "ranks" else
                                f"weak x{world} (independent problems)"),
                "l2": f"inputs+outputs {io_bytes / 2**20:.0f} MiB > L2 129 MiB; no flush",
            },
            "pct_of_peak": round(100.0 * value / world / peaks["bf16_tflops"], 2),
            "split": {"mode": split, "gpu_ms_per_step": [round(x, 4) for x in gpu_ms],
                      "gpu_ms_max": round(max(gpu_ms), 4), "gpu_ms_sum": round(sum(gpu_ms), 4)},
            "roofline": {
                "bound": "tensor", "achieved": round(achieved, 2),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved / peaks["bf16_tflops"], 4),
                "peak_source": f"{peaks['source']} bf16 dense (burst)",
                "traffic": traffic,
                "kernel": fwd_kernel_name(w) + " (+ prep_kernel inside the timed call)",
                "avg_launch_ms": round(avg_launch_ms, 4),
            },
            "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms / args.steps, 4),
                    "pipelined": "inputs of step i+1 and outputs of step i-1 copied during step i",
                    "matches_device_resident_output": e2e_same},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "backward": bwd,
            "secondary_roofline": merge,
        }
    return result, w, cu


def per_workload_report(args, local):
    """Forward time of every workload on this GPU (and the backward's for the
    bf16 ones), each workload's full schedule in one sp_packed_attention call,
    timed over calls issued back to back between two CUDA events (per-call
    average, median of a few such runs). For the 64K full-mask
    layer also the API path: one sp_partial_attn per schedule item into fp32
    partials and an sp_lse_merge per further item of a Q range."""
    import torch
    import sequence_blockwise_gb300 as sb
    from sequence_blockwise_gb300 import workloads as wl
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peak = read_peaks()["bf16_tflops"]

    def timed(fn, n, warm, reps=3):
        # n calls back to back between two events, so that the launches queue
        # on the stream and the host's argument marshalling between calls does
        # not leave the GPU idle inside the timed region; per-call average,
        # median over `reps` such runs.
        for _ in range(warm):
            fn()
        torch.cuda.synchronize(dev)
        time.sleep(1.0)  # each timed region starts from an idle GPU, as the headline's does
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(n):
                fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b) / n)
        sb.sp_check_device_status(stream)
        return float(np.median(ts))

    out = []
    for w in wl.WORKLOADS:
        big = w.T >= 262144
        cu = wl.cu_seqlens(w)
        pairs = valid_pairs(cu, w.causal)
        flop = 4.0 * w.d * w.Hq * pairs
        q, k, v = wl.make_qkv(w, dev)
        att = sb.PackedAttention(cu, w.causal, w.kind, w.P, w.Hq, seed=w.seed, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.Hq, w.T), dtype=torch.float32, device=dev)
        sampler = ClockSampler(local)  # clocks while this workload's calls run
        f_ms = timed(lambda: att(q, k, v, o, lse, stream=stream), 2 if big else 5, 1 if big else 3,
                     reps=2 if big else 3)
        e = {"workload": w.name, "dtype": w.dtype, "schedule": sched_name(w.kind), "P_virtual": w.P,
             "n_items": int(len(att.items)), "items_cut_at_documents": True, "valid_pairs": pairs,
             "forward_ms": round(f_ms, 4),
             "forward_tflops": round(flop / (f_ms * 1e-3) / 1e12, 2),
             "forward_kernel": fwd_kernel_name(w) if w.dtype == "bf16" else f"attn_simt_kernel<{w.d}> (fp32)"}
        if w.dtype == "bf16":
            e["forward_frac_of_peak"] = round(flop / (f_ms * 1e-3) / 1e12 / peak, 4)
            e["tile_work_over_valid_pairs"] = round(tile_work(att.items, cu, w.causal, w.T) / pairs, 4)
            dout = wl.random_normal((w.T, w.Hq, w.d), w.seed + 99, dev, "bf16")
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            b_ms = timed(lambda: att.backward(q, k, v, o, lse, dout, dq, dk, dv, stream=stream),
                         1 if big else 3, 1 if big else 2, reps=2 if big else 3)
            e["backward_ms"] = round(b_ms, 4)
            e["backward_tflops"] = round(2.5 * flop / (b_ms * 1e-3) / 1e12, 2)
            e["backward_frac_of_peak"] = round(2.5 * flop / (b_ms * 1e-3) / 1e12 / peak, 4)
            del dout, dq, dk, dv
        else:
            e["forward_frac_of_peak"] = None  # fp32 on CUDA cores, launch bound at this size
        if w.name.startswith("noncausal"):
            items = att.items
            groups = {}
            for it in items:
                groups.setdefault((int(it[0]), int(it[3]), int(it[4])), []).append(it)
            rows = max(int(it[4] - it[3]) for it in items)
            acc = [torch.empty((rows, w.Hq, w.d), dtype=torch.float32, device=dev) for _ in range(2)]
            accl = [torch.empty((w.Hq, rows), dtype=torch.float32, device=dev) for _ in range(2)]

            def api():
                for (_, qa, qb), its in groups.items():
                    n = qb - qa
                    oa, la = acc[0][:n], accl[0][:, :n]
                    op, lp = acc[1][:n], accl[1][:, :n]
                    for j, it in enumerate(its):
                        dst_o, dst_l = (oa, la) if j == 0 else (op, lp)
                        sb.sp_partial_attn(q, k, v, dst_o, dst_l, qa, qb, int(it[5]), int(it[6]), att.cu_dev,
                                           w.causal, stream=stream)
                        if j > 0:
                            sb.sp_lse_merge(oa, la, op, lp, stream=stream)

            a_ms = timed(api, 2, 1)
            e["api_path"] = {"ms": round(a_ms, 4), "tflops": round(flop / (a_ms * 1e-3) / 1e12, 2),
                             "launches": int(len(items) + len(items) - len(groups)),
                             "what": "one sp_partial_attn per item (fp32 partials) + sp_lse_merge per "
                                     "further item of a Q range"}
            del acc, accl
        e["clocks"] = sampler.stop()
        out.append(e)
        del q, k, v, o, lse, att
        torch.cuda.empty_cache()
    return out


def kernel_only(args, local):
    """W warm-up and K timed steps of the device-resident path, nothing else:
    the command the ncu summaries under profiles/ were taken with."""
    import torch
    import sequence_blockwise_gb300 as sb
    from sequence_blockwise_gb300 import workloads as wl
    w = wl.WORKLOADS[WORKLOAD_INDEX]
    if args.workload:
        w = next(x for x in wl.WORKLOADS if x.name == args.workload)
    cu = wl.cu_seqlens(w)
    dev = torch.device("cuda", local)
    q, k, v = wl.make_qkv(w, dev)
    att = sb.PackedAttention(cu, w.causal, w.kind, w.P, w.Hq, seed=w.seed, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.Hq, w.T), dtype=torch.float32, device=dev)
    if args.pass_ == "backward":
        att(q, k, v, o, lse)
        dout = wl.random_normal((w.T, w.Hq, w.d), w.seed + 99, dev, "bf16")
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        run = lambda: att.backward(q, k, v, o, lse, dout, dq, dk, dv)
        mult = 2.5
    else:
        run = lambda: att(q, k, v, o, lse)
        mult = 1.0
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        run()
    e1.record()
    torch.cuda.synchronize(dev)
    sb.sp_check_device_status()
    ms = e0.elapsed_time(e1) / max(1, args.steps)
    flop = mult * 4.0 * w.d * w.Hq * valid_pairs(cu, w.causal)
    print(json.dumps({"kernel_only": True, "pass": args.pass_, "workload": w.name, "ms_per_step": ms,
                      "tflops": flop / (ms * 1e-3) / 1e12}), flush=True)


def balance_report(args, local):
    """Per-virtual-rank device time of each chunking policy: every rank's items
    run alone through sp_packed_attention (one persistent launch on the whole
    GPU), so the slowest rank is the compute critical path of one SP step on P
    GPUs (transfers not included). Packed workloads and the single causal
    document, with the policies the schedule kind allows; the packed ones both
    with the items as built and cut at document boundaries."""
    import torch
    import sequence_blockwise_gb300 as sb
    from sequence_blockwise_gb300 import workloads as wl
    dev = torch.device("cuda", local)
    # (workload, schedule kind, chunking policies, Ulysses ranks per group)
    cases = [(1, sb.SP_SCHED_ZIGZAG, [0], 1), (1, sb.SP_SCHED_RING, [0, 1], 1),
             (2, sb.SP_SCHED_TASP, [0, 1, 2], 1), (4, sb.SP_SCHED_TASP, [0, 1, 2], 1),
             (3, sb.SP_SCHED_RING, [0], 1), (3, sb.SP_SCHED_RING, [0], 8), (1, sb.SP_SCHED_ZIGZAG, [0], 4)]
    out = []
    for idx, kind, modes, U in cases:
        w = wl.WORKLOADS[idx]
        cu = wl.cu_seqlens(w)
        q, k, v = wl.make_qkv(w, dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.Hq, w.T), dtype=torch.float32, device=dev)
        cu_dev = torch.from_numpy(cu).to(dev)
        for mode, cut in [(m, c) for m in modes for c in ((False, True) if len(cu) > 2 else (False,))]:
            R = w.P // U
            bounds = None if mode == 0 else sb.sp_chunk_bounds(mode, R, w.T, cu, w.causal)
            if U > 1:
                items, heads = sb.sp_schedule_build_hier(kind, R, U, w.T, cu, w.causal, w.Hq, seed=w.seed,
                                                         bounds=bounds)
            else:
                items = sb.sp_schedule_build(kind, w.P, w.T, cu, w.causal, seed=w.seed, bounds=bounds)
                heads = np.tile(np.array([[0, w.Hq]], dtype=np.int32), (len(items), 1))
            if cut:
                items, heads = sb.sp_schedule_split_documents(items, cu, w.causal, heads=heads)
            ms, pairs = [], []
            for r in range(w.P):
                sel = items[:, 0] == r
                mine = np.ascontiguousarray(items[sel])
                hmine = np.ascontiguousarray(heads[sel])
                pr = sum(valid_pairs_range(cu, w.causal, it) * int(h[1] - h[0]) for it, h in zip(mine, hmine))
                pairs.append(pr)
                if len(mine) == 0:
                    ms.append(0.0)
                    continue
                it_dev = torch.from_numpy(mine).to(dev)
                hd_dev = torch.from_numpy(hmine).to(dev)
                ws = torch.empty(sb.sp_packed_attention_workspace_size(len(mine)), dtype=torch.uint8,
                                 device=dev)
                run = lambda: sb.sp_packed_attention_ex(q, k, v, o, lse, cu_dev, w.causal, it_dev, hd_dev, ws)
                run()
                torch.cuda.synchronize(dev)
                t = []
                for _ in range(3):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    run()
                    b.record()
                    torch.cuda.synchronize(dev)
                    t.append(a.elapsed_time(b))
                ms.append(float(np.median(t)))
            sb.sp_check_device_status()
            ms_a, pr_a = np.array(ms), np.array(pairs, dtype=np.float64)
            cuts = 0 if bounds is None else int(sum(1 for x in bounds[1:-1] if x not in set(cu.tolist())))
            out.append({"workload": w.name, "schedule": sched_name(kind) + (f" {R}x{U} (head split)" if U > 1 else ""),
                        "P_virtual": w.P,
                        "chunking": ["equal", "balanced", "balanced_doc"][mode],
                        "split_at_documents": cut, "n_items": int(len(items)),
                        "bounds_inside_documents": cuts,
                        "pairs_max_over_mean": round(float(pr_a.max() / pr_a.mean()), 4),
                        "rank_ms_max": round(float(ms_a.max()), 4), "rank_ms_mean": round(float(ms_a.mean()), 4),
                        "rank_ms_max_over_mean": round(float(ms_a.max() / ms_a.mean()), 4),
                        "rank_ms": [round(x, 3) for x in ms]})
            print(json.dumps(out[-1]), flush=True)
        del q, k, v, o, lse
        torch.cuda.empty_cache()
    return out


def valid_pairs_range(cu, causal, it):
    """Valid (query, key) pairs of one item (closed form per document)."""
    qa, qb, ka, kb = int(it[3]), int(it[4]), int(it[5]), int(it[6])
    total = 0
    for d in range(len(cu) - 1):
        a, b = int(cu[d]), int(cu[d + 1])
        q0, q1 = max(a, qa), min(b, qb)
        k0, k1 = max(a, ka), min(b, kb)
        if q0 >= q1 or k0 >= k1:
            continue
        if not causal:
            total += (q1 - q0) * (k1 - k0)
            continue
        # sum over rows i in [q0, q1) of max(0, min(k1, i + 1) - k0)
        for_rows_lo = max(q0, k0)
        if for_rows_lo >= q1:
            continue
        # rows with i + 1 <= k1: count i + 1 - k0; rows with i + 1 > k1: k1 - k0
        m1 = min(q1, k1)  # rows i < m1 have i + 1 <= k1
        if m1 > for_rows_lo:
            n = m1 - for_rows_lo
            first = for_rows_lo + 1 - k0
            total += n * first + n * (n - 1) // 2
        if q1 > max(m1, for_rows_lo):
            total += (q1 - max(m1, for_rows_lo)) * (k1 - k0)
    return total


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=None,
                    help="seconds of oracle work for the cpu_baseline field (default 12); with "
                         "--impl reference, per timed step (default: 120 s over all steps, 1-20 s each)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the backward measurement reported beside the headline")
    ap.add_argument("--pass", dest="pass_", choices=["forward", "backward"], default="forward",
                    help="with --kernel-only: which pass to run")
    ap.add_argument("--balance", action="store_true",
                    help="per-virtual-rank device time of the chunking policies (one JSON line each)")
    ap.add_argument("--kernel-only", action="store_true",
                    help="only W warm-up + K device-resident steps (driver for ncu captures)")
    ap.add_argument("--split", choices=["ranks", "replicas"], default="ranks",
                    help="with N > 1 GPUs: split the virtual ranks over the GPUs (strong scaling) or run "
                         "one independent copy per GPU (weak scaling)")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the per_workload report (forward/backward of every workload)")
    ap.add_argument("--workload", default=None,
                    help="with --kernel-only: workload name (default: the 32K-token layer)")
    args = ap.parse_args()

    world, rank, local = dist_setup()
    from sequence_blockwise_gb300 import workloads as wl
    w = wl.WORKLOADS[WORKLOAD_INDEX]
    cu = wl.cu_seqlens(w)

    if args.impl == "reference":
        # The fp64 CPU oracle on a bounded sample per step, rank 0 only.
        if rank == 0:
            per_step = (args.cpu_seconds if args.cpu_seconds is not None else
                        max(1.0, min(20.0, 120.0 / max(1, args.steps + args.warmup))))
            for _ in range(args.warmup):
                oracle_sample(w, cu, per_step * 0.25, seed=99)
            flop = elapsed = rows = 0
            threads = 1
            for s in range(args.steps):
                f, e, n, threads = oracle_sample(w, cu, per_step, seed=s)
                flop, elapsed, rows = flop + f, elapsed + e, rows + n
            value = flop / elapsed / 1e12
            sample = (f"{rows} random query rows x {w.Hq} heads over {args.steps} steps "
                      f"(~{per_step:.0f} s each) of {w.name}")
            print(json.dumps({
                "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1000.0 * elapsed / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": w.name, "schedule": sched_name(w.kind), "P_virtual": w.P},
                "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "gpu_launches": 0,
            }), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    if args.kernel_only:
        kernel_only(args, local)
        return
    if args.balance:
        balance_report(args, local)
        return

    result, w, cu = run_ours(args, world, rank, local)
    if rank == 0 and world == 1 and not args.no_per_workload:
        result["per_workload"] = per_workload_report(args, local)
    if rank == 0:
        if args.no_cpu_baseline or world > 1:
            result["cpu_baseline"] = None
        else:
            f, e, n, threads = oracle_sample(w, cu, args.cpu_seconds if args.cpu_seconds is not None else 12.0)
            rate = f / e  # oracle FLOP/s over valid pairs
            result["cpu_baseline"] = {
                "value": round(rate / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
                "kind": "oracle",
                "sample": f"{n} random query rows x {w.Hq} heads of {w.name}, fp64, {e:.1f} s",
                # The whole workload at the sample's rate (rows are independent).
                "full_workload_s": round(result["config"]["flop_per_step"] / rate, 1),
                "gpu_ms_per_step": result["ms_per_step"],
            }
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
