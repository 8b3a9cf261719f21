#!/usr/bin/env python
"""Benchmark of the MoE dispatch / combine hot path on GB300.

One step = routing layout and bf16 dispatch (ep_layout_and_dispatch: the
layout kernel, then the dispatch kernel) -> identity expert (the combine reads
the dispatched rows) -> unweighted combine (ep_combine), on the
DeepSeek-V3-shaped prefill workload: T=4096 tokens,
H=7168 bf16, E=256 experts, top-8 distinct uniform experts per token, R=8
logical ranks in one GPU's memory.  Inputs are seeded synthetic data.

The metric is throughput in GB/s of algorithmic bytes (what the method must
read and write: see ``algorithmic_bytes``) per step, with tokens/s beside it
and the dominant kernel's HBM roofline fraction against the measured copy
bandwidth.  L2 (129 MB) is flushed before the layout and again before the
combine (in a real layer, expert GEMMs run between them), outside the timed
events: a 256 MiB buffer is written and then a second one of 256 MiB is read,
so the flush's own dirty lines are written back before the timed kernel starts
(``--flush write`` keeps only the write, leaving ~129 MB of dirty lines for the
timed kernel to write back).

Multi-GPU: the path does not shard (ranks are partitions of one GPU), so
``--gpus N`` under torchrun runs N independent replicas; the time is the max
over ranks and the value is the sum of all replicas' work ("weak" scaling).

``--impl reference`` times the CPU oracle (the test suite's checker) on the
host cores instead, on a bounded token sample per step.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 256 << 20
HBM_NOMINAL_GBS = 7900.0   # GB300 HBM3e nominal bandwidth (context beside the measured copy peak)


def host_cpu():
    """Host core count and CPU model (as far as /proc/cpuinfo names it)."""
    import platform
    model = platform.machine()
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"host_cores": os.cpu_count(), "cpu_model": model}
# ep_layout_and_dispatch's one-kernel limits (include/ep_get.h)
ONE_KERNEL_MAX_TOKENS, ONE_KERNEL_MAX_RANKS, ONE_KERNEL_MAX_TOPK, ONE_KERNEL_MAX_EXPERTS = 256, 32, 16, 2048


def kernels_per_step(T, R, expanded=False, hierarchical=False, fused=False, K=0, E=0):
    """Launches of this library per step: the layout is one kernel (the
    single-CTA kernel for few tokens, else one cluster), or three tiled kernels
    when T*R passes 2^19 (expanded and node rows ride on the same kernels; the
    tiled fallback for a cluster whose shared memory would not fit does not
    occur on these workloads); dispatch and combine one each, two each on the
    hierarchical path.  ep_layout_and_dispatch (fused) with few tokens runs
    layout and dispatch as one kernel."""
    if (fused and not expanded and not hierarchical and 1 <= T <= ONE_KERNEL_MAX_TOKENS
            and R <= ONE_KERNEL_MAX_RANKS and K <= ONE_KERNEL_MAX_TOPK and E <= ONE_KERNEL_MAX_EXPERTS):
        return 1 + 1
    tiled = T * R > (1 << 19)
    return (3 if tiled else 1) + (4 if hierarchical else 2)


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dsv3")
    ap.add_argument("--path", choices=["rank", "expanded", "hierarchical"], default="rank",
                    help="rank: one receive row per (token, rank); expanded: one per valid (token, k), "
                         "grouped by expert (weighted combine); hierarchical: two-stage dispatch and "
                         "combine through per-node buffers")
    ap.add_argument("--ranks-per-node", type=int, default=0,
                    help="hierarchical path: ranks per node (default: the workload's, else R/2)")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of CUDA graphs")
    ap.add_argument("--fp8", action="store_true",
                    help="FP8 e4m3 dispatch (per-128-channel scales) on any workload; the combine then reads "
                         "bf16 stand-in expert rows")
    ap.add_argument("--num-sms", default="0",
                    help="SM-limited dispatch and combine (persistent grid of this many CTAs); 0 = whole "
                         "GPU; 'rule' = each phase's count from ep_theoretical_num_sms with the measured "
                         "HBM peak and the per-SM rates below")
    ap.add_argument("--sm-read-gbs", type=float, default=200.0, help="per-SM read rate of the SM count rule")
    ap.add_argument("--sm-write-gbs", type=float, default=50.0, help="per-SM write rate of the SM count rule")
    ap.add_argument("--flush", choices=["write+read", "write"], default="write+read",
                    help="L2 flush before layout and combine: write 256 MiB then read another 256 MiB "
                         "(clean L2), or the write alone (dirty L2)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU time budget of the oracle baseline (rank 0, N=1)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------

def algorithmic_bytes_expanded(T, H, K, E, R, M, fp8=False):
    """Bytes per step of the expanded path, M = valid (token, k) slots.

    layout:   as the rank path, plus the [T, K] expanded rows written.
    dispatch: read x, topk_idx, topk_weights and the expanded rows; write M
              rows of payload (+ FP8 scales), a source index and a weight each.
    combine:  read the expanded rows, the weights and M expert-output rows;
              write T rows.
    """
    b_out = 1 if fp8 else 2
    s = 4 * (H // 128) if fp8 else 0
    layout = T * K * 8 + T * R * 5 + T * K * 4 + 4 * (3 * E + 3 * R + 2)
    dispatch = T * H * 2 + T * K * 12 + T * K * 4 + M * (H * b_out + s + 8)
    combine = M * H * 2 + T * K * 8 + T * H * 2
    return dict(layout=layout, dispatch=dispatch, combine=combine, total=layout + dispatch + combine)


def algorithmic_bytes_hierarchical(T, H, K, E, R, nodes, N, M, weighted=False, fp8=False):
    """Bytes per step of the two-stage path, M = node rows (token, node pairs).

    layout:   as the rank path, plus node rows [T, nodes] written.
    dispatch: stage 1 reads x, topk_idx and the node rows and writes M node
              rows (+ FP8 scales) and their source index; stage 2 reads the
              node rows and dst_row, topk_idx and topk_weights, and writes N
              rows with their metadata.
    combine:  stage 1 reads dst_row and N rows (+ topk for weighting) and
              writes M node partials; stage 2 reads the node rows and the M
              partials and writes T rows.
    """
    b_out = 1 if fp8 else 2
    s = 4 * (H // 128) if fp8 else 0
    layout = T * K * 8 + T * R * 5 + T * nodes * 4 + 4 * (3 * E + 3 * R + 2 * nodes + 3)
    stage1 = T * H * 2 + T * K * 8 + T * nodes * 4 + M * (H * b_out + s + 4)
    stage2 = T * nodes * 4 + T * R * 4 + T * K * 12 + M * (H * b_out + s) + N * (H * b_out + s + 8 * K + 4)
    reduce1 = T * nodes * 4 + T * R * 4 + N * H * 2 + M * H * 2 + (T * K * 12 if weighted else 0)
    reduce2 = T * nodes * 4 + M * H * 2 + T * H * 2
    dispatch, combine = stage1 + stage2, reduce1 + reduce2
    return dict(layout=layout, dispatch=dispatch, combine=combine, total=layout + dispatch + combine)


def algorithmic_bytes(T, H, K, E, R, N, weighted=False, fp8=False):
    """Bytes the method must move per step (reads + writes), by kernel.

    layout:   read topk_idx (8 B per entry), write dst_row (4 B) and
              is_token_in_rank (1 B) per (token, rank), plus the O(E + R) counts.
    dispatch: read x, topk_idx, topk_weights and dst_row; write N rows of
              payload (+ FP8 scales), K remapped indices, K weights, 1 source index.
    combine:  read dst_row and N expert-output rows (+ topk for weighting);
              write T rows.
    """
    b_out = 1 if fp8 else 2
    s = 4 * (H // 128) if fp8 else 0
    layout = T * K * 8 + T * R * 5 + 4 * (3 * E + 3 * R + 2)
    dispatch = T * H * 2 + T * K * 12 + T * R * 4 + N * (H * b_out + s + 8 * K + 4)
    combine = N * H * 2 + T * R * 4 + T * H * 2 + (T * K * 12 if weighted else 0)
    return dict(layout=layout, dispatch=dispatch, combine=combine,
                total=layout + dispatch + combine)


# ---------------------------------------------------------------------------
# distributed helpers (replicas)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value, world, device=None):
    """Max of a float over all ranks (identity when world == 1)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def replica_value(units_per_step, steps, max_total_ms, world):
    """Whole-job throughput: all replicas' units / the slowest replica's time."""
    if max_total_ms <= 0:
        return 0.0
    return world * units_per_step * steps / (max_total_ms / 1e3)


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# peaks and recorded DRAM traffic
# ---------------------------------------------------------------------------

def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def _code_only(text):
    """C++ source without comments and with whitespace runs collapsed, so that
    an edit of comments alone keeps the hash (string literals are kept)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':                       # string literal, copied as is
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(kernel):
    """sha256[:16] of the kernel's source file followed by the shared device
    header, comments and whitespace left out."""
    h = hashlib.sha256()
    for name in ("%s.cu" % kernel, "ep_internal.cuh"):
        with open(os.path.join(ROOT, "combine_ep_get_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from an ncu capture, if recorded for this source
    ("layout+dispatch": the sum of the two kernels' records)."""
    if "+" in kernel:
        parts = [recorded_traffic(k, workload) for k in kernel.split("+")]
        return None if any(p is None for p in parts) else sum(parts)
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[workload][kernel]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("source_sha256_16") != kernel_source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import numpy as np
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl")
    from combine_ep_get_gb300 import build as lib_build
    lib_build.build()
    from combine_ep_get_gb300 import binding as B
    from combine_ep_get_gb300.inputs import CONFIGS, make_config, make_rows

    cfg = CONFIGS[args.workload]
    if args.fp8 and not cfg.fp8:
        import dataclasses
        cfg = dataclasses.replace(cfg, fp8=True, description=cfg.description.replace(" bf16", "") + ", FP8 dispatch")
    data = make_config(cfg)
    T, H, E, K, R = cfg.T, cfg.H, cfg.E, cfg.K, cfg.R
    dev = torch.device("cuda", local)

    x_host = torch.from_numpy(data["x_bits"].view(np.int16)).view(torch.bfloat16)
    idx_host = torch.from_numpy(data["topk_idx"])
    w_host = torch.from_numpy(data["topk_weights"])
    x = x_host.to(dev)
    idx = idx_host.to(dev)
    w = w_host.to(dev)

    expanded = args.path == "expanded"
    hierarchical = args.path == "hierarchical"
    rpn = cfg.ranks_per_node
    if hierarchical:
        rpn = args.ranks_per_node or cfg.ranks_per_node or max(1, R // 2)
    lay = B.alloc_layout(T, E, R, rpn, device=dev, K=K if expanded else None, node_rows=hierarchical)
    ws = torch.empty(B.ep_layout_workspace_bytes(T, K, E, R, rpn), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    B.ep_get_layout(idx, E, R, lay, ws, status, rpn)
    # one host read of the row count (rank_offset[R], or expert_offset[E] for the
    # expanded rows), before any timing
    N = int(lay.expert_offset[-1].item()) if expanded else lay.num_recv
    fp8, weighted = cfg.fp8, cfg.weighted
    recv_idx = torch.empty((N, K), dtype=torch.int32, device=dev)
    recv_w = torch.empty((N, K), dtype=torch.float32, device=dev)
    recv_src = torch.empty((N,), dtype=torch.int32, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.zeros(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
    flush_rd2 = torch.zeros(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
    flush_sink = torch.zeros((), dtype=torch.int64, device=dev)

    def flush_l2():
        flush.zero_()
        if args.flush == "write+read":
            torch.sum(flush_rd, dim=0, out=flush_sink)
    if fp8:
        # FP8 dispatch; the combine reads a bf16 stand-in for the expert outputs
        recv_x = torch.empty((N, H), dtype=torch.uint8, device=dev)
        recv_sf = torch.empty((N * (H // 128),), dtype=torch.float32, device=dev)
        y = torch.from_numpy(make_rows(N, H, cfg.seed + 100).view(np.int16)).view(torch.bfloat16).to(dev)
    else:
        # identity expert: the combine reads the dispatched rows
        recv_x = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
        recv_sf = None
        y = recv_x
    dtype_code = B.EP_FP8_E4M3 if fp8 else B.EP_BF16
    w_comb = w if weighted else None
    if expanded:
        weighted = True            # the expanded combine weights every (token, k) output
        recv_weight = torch.empty((N,), dtype=torch.float32, device=dev)
    hier = None
    if hierarchical:
        M = int(lay.node_offset[-1].item())
        hier = dict(rpn=rpn, M=M, node_src=torch.empty((M,), dtype=torch.int32, device=dev),
                    node_y=torch.empty((M, H), dtype=torch.bfloat16, device=dev),
                    node_x=torch.empty((M, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev),
                    node_sf=torch.empty((M * (H // 128),), dtype=torch.float32, device=dev) if fp8 else None)

    if args.num_sms == "rule":
        hbm, _ = hbm_peak()
        rule = dict(H=H, K=K, E=E, R=R, hbm_gbs=hbm, sm_read_gbs=args.sm_read_gbs,
                    sm_write_gbs=args.sm_write_gbs)
        sms_dispatch = B.ep_theoretical_num_sms(H, K, E, R, hbm, out_dtype=dtype_code, is_combine=False,
                                                sm_read_gbs=args.sm_read_gbs, sm_write_gbs=args.sm_write_gbs)
        sms_combine = B.ep_theoretical_num_sms(H, K, E, R, hbm, is_combine=True, sm_read_gbs=args.sm_read_gbs,
                                               sm_write_gbs=args.sm_write_gbs)
        sms_config = {"dispatch": sms_dispatch, "combine": sms_combine, "rule": rule}
    else:
        sms_dispatch = sms_combine = int(args.num_sms)
        sms_config = sms_dispatch or "all"

    def do_layout():
        B.ep_get_layout(idx, E, R, lay, ws, status, rpn)

    # The rank path over the whole GPU runs layout and dispatch as one call
    # (ep_layout_and_dispatch): with few tokens the dispatch then derives its
    # rows itself and runs beside the layout; with many it is the same two
    # launches as the separate calls.
    fused = args.path == "rank" and sms_dispatch == 0
    one_kernel = fused and kernels_per_step(T, R, False, False, True, K, E) == 2

    def do_layout_dispatch():
        if fused:
            B.ep_layout_and_dispatch(x, idx, w, E, R, lay, ws, recv_x, recv_idx, recv_w, recv_src, status,
                                     recv_sf=recv_sf, out_dtype=dtype_code, ranks_per_node=rpn)
        else:
            do_layout()
            do_dispatch()

    def do_dispatch():
        if hierarchical:
            B.ep_dispatch_hierarchical(x, idx, w, E, R, rpn, lay, hier["node_x"], recv_x, status,
                                       node_sf=hier["node_sf"], node_src_idx=hier["node_src"], recv_sf=recv_sf,
                                       recv_topk_idx=recv_idx, recv_topk_weights=recv_w, recv_src_idx=recv_src,
                                       out_dtype=dtype_code)
        elif expanded:
            B.ep_dispatch_expanded(x, idx, w, E, R, lay, recv_x, recv_src, recv_weight, status,
                                   recv_sf=recv_sf, out_dtype=dtype_code, num_sms=sms_dispatch)
        else:
            B.ep_dispatch(x, idx, w, E, R, lay, recv_x, recv_idx, recv_w, recv_src, status,
                          recv_sf=recv_sf, out_dtype=dtype_code, num_sms=sms_dispatch)

    def do_combine():
        if hierarchical:
            B.ep_combine_hierarchical(y, idx, w_comb, E, R, rpn, lay, hier["node_y"], out, status)
        elif expanded:
            B.ep_combine_expanded(y, w, K, E, R, lay, out, status, num_sms=sms_combine)
        else:
            B.ep_combine(y, idx, w_comb, E, R, lay, out, status, num_sms=sms_combine)

    # eager warm-up (sets kernel attributes outside any capture)
    for _ in range(2):
        do_layout()
        do_dispatch()
        do_combine()
        do_layout_dispatch()
        do_combine()
    torch.cuda.synchronize()
    st = int(status.item())
    if st != 0:
        raise RuntimeError("device status after warm-up: %s" % B.ep_status_string(st))

    use_graph = not args.no_graph

    def step_body(ev, split):
        # split (per-kernel breakdown): separate calls with an event between
        # layout and dispatch, and after the combine two read passes over
        # different 256 MiB buffers: the first also writes back what the
        # combine left dirty in L2, the second finds only clean lines.
        # Without split the dispatch launch overlaps the layout (programmatic
        # dependent launch), as in a real layer.
        flush_l2()
        ev[0].record()
        if split:
            do_layout()
            ev[4].record()
            do_dispatch()
        else:
            do_layout_dispatch()
        ev[1].record()
        flush_l2()
        ev[2].record()
        do_combine()
        ev[3].record()
        if split:
            torch.sum(flush_rd, dim=0, out=flush_sink)
            ev[5].record()
            torch.sum(flush_rd2, dim=0, out=flush_sink)
            ev[6].record()

    def new_events():
        if use_graph:
            return [torch.cuda.Event(enable_timing=True, external=True) for _ in range(7)]
        return [torch.cuda.Event(enable_timing=True) for _ in range(7)]

    # One CUDA graph per step holds the flushes, the three calls and the timing
    # events; n_graphs instances rotate so the GPU never waits for the host
    # while the times of a finished instance are read.
    n_graphs = 4

    def make_slots(split):
        slots = []
        for _ in range(n_graphs):
            ev = new_events()
            g = None
            if use_graph:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    step_body(ev, split)
            slots.append((g, ev))
        return slots

    def run(slots, split, steps, warm):
        times = []

        def launch(k):
            g, ev = slots[k]
            if g is not None:
                g.replay()
            else:
                step_body(ev, split)

        def harvest(k):
            ev = slots[k][1]
            ev[6 if split else 3].synchronize()
            t = [ev[0].elapsed_time(ev[1]), ev[2].elapsed_time(ev[3])]
            if split:
                t += [ev[0].elapsed_time(ev[4]), ev[4].elapsed_time(ev[1]),
                      ev[3].elapsed_time(ev[5]) - ev[5].elapsed_time(ev[6])]
            times.append(t)

        for i in range(warm):
            launch(i % n_graphs)
        torch.cuda.synchronize()
        pending = []
        for i in range(steps):
            k = i % n_graphs
            if len(pending) == n_graphs:
                harvest(pending.pop(0))
            launch(k)
            pending.append(k)
        for k in pending:
            harvest(k)
        torch.cuda.synchronize()
        return times

    main_slots = make_slots(False)
    split_slots = make_slots(True)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.25)
    run(main_slots, False, 0, args.warmup)
    barrier(world)
    torch.cuda.synchronize()
    times = run(main_slots, False, args.steps, 0)          # the timed region
    torch.cuda.synchronize()
    barrier(world)
    time.sleep(0.15)
    clocks = sampler.stop()
    st = int(status.item())
    if st != 0:
        raise RuntimeError("device status after timing: %s" % B.ep_status_string(st))
    # per-kernel breakdown (layout and dispatch apart), after the timed region
    n_split = max(50, args.steps // 10)
    split_times = run(split_slots, True, n_split, args.warmup)

    t_ld = [t[0] for t in times]
    t_combine = [t[1] for t in times]
    local_total = sum(t_ld) + sum(t_combine)
    max_total = reduce_max(local_total, world, dev)

    if expanded:
        nbytes = algorithmic_bytes_expanded(T, H, K, E, R, int((idx >= 0).sum().item()), fp8=fp8)
    elif hierarchical:
        nbytes = algorithmic_bytes_hierarchical(T, H, K, E, R, R // rpn, N, hier["M"], weighted=weighted, fp8=fp8)
    else:
        nbytes = algorithmic_bytes(T, H, K, E, R, N, weighted=weighted, fp8=fp8)
    value_bps = replica_value(nbytes["total"], args.steps, max_total, world)
    tokens_ps = replica_value(T, args.steps, max_total, world)
    ms_per_step = max_total / args.steps

    # Timed region: the layout+dispatch call(s) and the combine, each between
    # its own events.  Breakdown pass: layout and dispatch apart, and the
    # combine plus the write-back of its dirty L2 lines (the extra time a
    # 256 MiB read pass right after it takes over one over clean L2).
    avg = {"layout+dispatch": statistics.mean(t_ld),
           "combine": statistics.mean(t_combine),
           "layout": statistics.mean(t[2] for t in split_times),
           "dispatch": statistics.mean(t[3] for t in split_times),
           "combine_with_writeback": statistics.mean(t[1] + max(t[4], 0.0) for t in split_times)}
    source = {"layout+dispatch": "timed region", "combine": "timed region", "layout": "breakdown pass",
              "dispatch": "breakdown pass",
              "combine_with_writeback": "breakdown pass: combine + write-back of its dirty L2 lines"}
    nbytes["layout+dispatch"] = nbytes["layout"] + nbytes["dispatch"]
    nbytes["combine_with_writeback"] = nbytes["combine"]
    # the roofline's kernel: the longer of the two timed-region intervals
    dominant = "layout+dispatch" if avg["layout+dispatch"] >= avg["combine"] else "combine"
    peak, peak_kind = hbm_peak()
    achieved = nbytes[dominant] / (avg[dominant] * 1e-3) / 1e9
    per_kernel = {k: {"ms": avg[k], "gbs": nbytes[k] / (avg[k] * 1e-3) / 1e9,
                      "frac_of_" + peak_kind: nbytes[k] / (avg[k] * 1e-3) / 1e9 / peak,
                      "timed_in": source[k]}
                  for k in avg}

    # end to end through the public API with host buffers
    e2e = run_e2e(args, B, torch, dev, x_host, idx_host, w_host, lay, ws, status, recv_x, recv_sf, y,
                  recv_idx, recv_w, recv_src, out, cfg, nbytes, world, rpn, hier)

    result = {
        "metric": "dispatch+combine GB/s and tokens/s on 1 GB300; % of HBM roofline",
        "value": value_bps / 1e9,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8_e4m3" if fp8 else "bf16",
        "data": "synthetic",
        "tokens_per_s": tokens_ps,
        "config": {
            "workload": cfg.description,
            "T": T, "H": H, "E": E, "K": K, "R": R, "N": N, "path": args.path,
            **({"ranks_per_node": rpn, "node_rows": hier["M"]} if hierarchical else {}),
            "num_sms": sms_config,
            "bytes_per_step": nbytes,
            "parallelism": "replicas" if world > 1 else "single",
            "l2": ("flushed before layout and before combine, outside the timed events: 256 MiB written, "
                   "then another 256 MiB read (the flush's dirty lines drained)" if args.flush == "write+read"
                   else "flushed (256 MiB write) before layout and before combine, outside the timed events"),
            "launch": ("one CUDA graph per step (flushes, calls and timing events inside)"
                       if use_graph else "eager"),
            "arithmetic": ("fp8 e4m3 dispatch with fp32 per-128-channel scales; combine of bf16 "
                           "stand-in expert rows, weighted, fp32 accumulate, bf16 out" if fp8 else
                           "bf16 row copies; combine of the dispatched rows (identity expert), "
                           "%s, fp32 accumulate, bf16 out" % ("weighted" if weighted else "unweighted")) +
                          ("; expanded rows: one per valid (token, k), grouped by expert" if expanded else "") +
                          ("; two stages: each token once per node into per-node buffers, then fanned out to "
                           "the node's ranks; combine partials per (token, node) stored as bf16"
                           if hierarchical else ""),
        },
        "per_kernel": per_kernel,
        "roofline": {"bound": "hbm",
                     "kernel": (("layout+dispatch (ep_layout_and_dispatch: one kernel, the layout inside the "
                                 "dispatch)" if one_kernel else
                                 "layout+dispatch (%s: the layout kernel, then the dispatch kernel launched "
                                 "during it)" % ("ep_layout_and_dispatch" if fused else "ep_get_layout, ep_dispatch"))
                                if dominant == "layout+dispatch" else "combine"),
                     "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "frac_of_nominal": achieved / HBM_NOMINAL_GBS,
                     # recorded DRAM traffic is of the rank path's bf16 kernels only
                     "traffic": (recorded_traffic(dominant, args.workload)
                                 if args.path == "rank" and not args.fp8 else None),
                     "algorithmic_bytes_per_launch": nbytes[dominant], "timed_in": source[dominant]},
        "e2e": e2e,
        "gpu_launches": kernels_per_step(T, R, expanded, hierarchical, fused, K, E) * args.steps,
        "clocks": clocks,
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(cfg, data, nbytes, N, args.cpu_seconds)
        result["cpu_baseline_all_cores"] = cpu_baseline_all_cores(cfg, data, N, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, B, torch, dev, x_host, idx_host, w_host, lay, ws, status, recv_x, recv_sf, y, recv_idx,
            recv_w, recv_src, out, cfg, nbytes, world, rpn, hier):
    """End to end through the public calls with host buffers.

    Every step copies its inputs (x, topk_idx, topk_weights) from pinned host
    memory to the device, runs ep_layout_and_dispatch (the rank path; the
    other paths ep_get_layout and their dispatch) and the combine, and
    copies the combined rows back to pinned host memory.  Steps are pipelined
    on three streams with double-buffered device inputs and outputs: the
    copy-in of step i+1 and the copy-out of step i-1 overlap the kernels of
    step i, as a serving loop would run them.
    """
    E, R = cfg.E, cfg.R
    xp = x_host.pin_memory()
    ip = idx_host.pin_memory()
    wp = w_host.pin_memory()
    outp = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(xp, device=dev) for _ in range(2)]
    idd = [torch.empty_like(ip, device=dev) for _ in range(2)]
    wd = [torch.empty_like(wp, device=dev) for _ in range(2)]
    outd = [torch.empty_like(out) for _ in range(2)]
    s_in, s_comp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_comp[b])          # step i-2 no longer reads these inputs
            xd[b].copy_(xp, non_blocking=True)
            idd[b].copy_(ip, non_blocking=True)
            wd[b].copy_(wp, non_blocking=True)
            ev_in[b].record(s_in)
        s_comp.wait_event(ev_in[b])
        s_comp.wait_event(ev_out[b])             # step i-2's output has been copied out
        dtype_code = B.EP_FP8_E4M3 if cfg.fp8 else B.EP_BF16
        if args.path != "rank":
            B.ep_get_layout(idd[b], E, R, lay, ws, status, rpn, stream=s_comp)
        if args.path == "hierarchical":
            B.ep_dispatch_hierarchical(xd[b], idd[b], wd[b], E, R, rpn, lay, hier["node_x"], recv_x, status,
                                       node_sf=hier["node_sf"], node_src_idx=hier["node_src"], recv_sf=recv_sf,
                                       recv_topk_idx=recv_idx, recv_topk_weights=recv_w, recv_src_idx=recv_src,
                                       out_dtype=dtype_code, stream=s_comp)
            B.ep_combine_hierarchical(y, idd[b], wd[b] if cfg.weighted else None, E, R, rpn, lay, hier["node_y"],
                                      outd[b], status, stream=s_comp)
        elif args.path == "expanded":
            B.ep_dispatch_expanded(xd[b], idd[b], wd[b], E, R, lay, recv_x, recv_src, None, status,
                                   recv_sf=recv_sf, out_dtype=dtype_code, stream=s_comp)
            B.ep_combine_expanded(y, wd[b], idd[b].shape[1], E, R, lay, outd[b], status, stream=s_comp)
        else:
            B.ep_layout_and_dispatch(xd[b], idd[b], wd[b], E, R, lay, ws, recv_x, recv_idx, recv_w, recv_src,
                                     status, recv_sf=recv_sf, out_dtype=dtype_code, ranks_per_node=rpn,
                                     stream=s_comp)
            B.ep_combine(y, idd[b], wd[b] if cfg.weighted else None, E, R, lay, outd[b], status,
                         stream=s_comp)
        ev_comp[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            outp[b].copy_(outd[b], non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record(s_in)
    for i in range(args.e2e_steps):
        step(i)
    s_out.wait_stream(s_comp)
    end.record(s_out)
    torch.cuda.synchronize()
    barrier(world)
    ms = reduce_max(start.elapsed_time(end), world, dev)
    torch.cuda.synchronize()
    if not torch.equal(outp[(args.e2e_steps - 1) % 2].view(torch.int16), out.cpu().view(torch.int16)):
        raise RuntimeError("end-to-end output differs from the device-resident run")
    h2d = xp.numel() * xp.element_size() + ip.numel() * ip.element_size() + wp.numel() * wp.element_size()
    d2h = outp[0].numel() * outp[0].element_size()
    return {"value": replica_value(nbytes["total"], args.e2e_steps, ms, world) / 1e9, "unit": "GB/s",
            "ms_per_step": ms / args.e2e_steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "launch": "eager calls through the binding; copies and kernels pipelined on 3 streams"}


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------

def _oracle_step(oracle, np, data, cfg, tokens):
    """The oracle's layout on all tokens, then dispatch and combine of `tokens`."""
    idx, w, xb = data["topk_idx"], data["topk_weights"], data["x_bits"]
    L = oracle.layout(idx, cfg.E, cfg.R, cfg.ranks_per_node)
    d = oracle.dispatch(xb, idx, w, cfg.E, cfg.R, L.dst_row, tokens=tokens)
    mask = L.dst_row[tokens] >= 0
    local = np.full(mask.shape, -1, np.int32)
    local[mask] = np.arange(int(mask.sum()), dtype=np.int32)
    oracle.combine(d["recv_x"].view(np.uint16), idx[tokens], None, cfg.E, cfg.R, local)
    return int(mask.sum())


def _sample_bytes(cfg, n_tok, n_rows):
    T, H, K, E, R = cfg.T, cfg.H, cfg.K, cfg.E, cfg.R
    full = algorithmic_bytes(T, H, K, E, R, 0)
    disp = n_tok * H * 2 + n_tok * K * 12 + n_tok * R * 4 + n_rows * (H * 2 + 8 * K + 4)
    comb = n_rows * H * 2 + n_tok * R * 4 + n_tok * H * 2
    return full["layout"] + disp + comb


def cpu_baseline(cfg, data, nbytes, N, seconds):
    import numpy as np
    import oracle
    tokens = np.arange(cfg.T, dtype=np.int32)
    done, moved = 0, 0
    t0 = time.perf_counter()
    while True:
        rows = _oracle_step(oracle, np, data, cfg, tokens)
        done += 1
        moved += _sample_bytes(cfg, cfg.T, rows)
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    return {"value": moved / el / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "%d full step(s) of the workload (all %d tokens), single-threaded C oracle"
                      % (done, cfg.T),
            "tokens_per_s": done * cfg.T / el, **host_cpu()}


def cpu_baseline_all_cores(cfg, data, N, seconds):
    """The oracle's OpenMP build (same C source, token loops of dispatch and
    combine split over the host's cores; the layout stays sequential) on
    whole steps of the workload: layout, dispatch of every token into its
    rows, combine of the dispatched rows."""
    import numpy as np
    import oracle
    idx, w, xb = data["topk_idx"], data["topk_weights"], data["x_bits"]
    with oracle.threads() as n:
        if n is None:
            return {"unavailable": "no OpenMP build of the oracle on this host"}
        done, moved = 0, 0
        t0 = time.perf_counter()
        while True:
            L = oracle.layout(idx, cfg.E, cfg.R, cfg.ranks_per_node)
            d = oracle.dispatch(xb, idx, w, cfg.E, cfg.R, L.dst_row, capacity=L.num_recv)
            oracle.combine(d["recv_x"].view(np.uint16), idx, None, cfg.E, cfg.R, L.dst_row)
            done += 1
            moved += _sample_bytes(cfg, cfg.T, L.num_recv)
            if time.perf_counter() - t0 >= seconds:
                break
        el = time.perf_counter() - t0
    return {"value": moved / el / 1e9, "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": "%d full step(s) of the workload (all %d tokens), OpenMP build of the C oracle on %d "
                      "threads" % (done, cfg.T, n),
            "tokens_per_s": done * cfg.T / el, **host_cpu()}


def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from combine_ep_get_gb300.inputs import CONFIGS, make_config
    cfg = CONFIGS[args.workload]
    data = make_config(cfg)
    # size each step's token sample so that warm-up + timed steps take ~2 minutes
    probe = np.arange(64, dtype=np.int32)
    t0 = time.perf_counter()
    _oracle_step(oracle, np, data, cfg, probe)
    per_tok = max((time.perf_counter() - t0) / 64, 1e-7)
    budget = 120.0 / max(args.steps + args.warmup, 1)
    n_tok = int(min(cfg.T, max(8, budget / per_tok)))
    starts = [(i * n_tok) % cfg.T for i in range(args.steps + args.warmup)]

    def toks(s):
        return (np.arange(s, s + n_tok) % cfg.T).astype(np.int32)

    for s in starts[:args.warmup]:
        _oracle_step(oracle, np, data, cfg, toks(s))
    moved = 0
    t0 = time.perf_counter()
    for s in starts[args.warmup:]:
        rows = _oracle_step(oracle, np, data, cfg, toks(s))
        moved += _sample_bytes(cfg, n_tok, rows)
    el = time.perf_counter() - t0
    value = moved / el / 1e9
    sample = ("%d tokens per step (layout on all %d tokens, dispatch and combine of the sample), "
              "single-threaded C oracle" % (n_tok, cfg.T))
    print(json.dumps({
        "impl": "reference",
        "metric": "dispatch+combine GB/s and tokens/s on 1 GB300; % of HBM roofline",
        "value": value, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el * 1e3 / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "tokens_per_s": args.steps * n_tok / el,
        "config": {"workload": cfg.description, "T": cfg.T, "H": cfg.H, "E": cfg.E, "K": cfg.K,
                   "R": cfg.R, "l2": "n/a (host)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
                         **host_cpu()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
