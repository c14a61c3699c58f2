#!/usr/bin/env python3
"""Benchmark: block-sparse FP8 attention prefill over a paged KV cache on GB300.

One step = one bsa_fp8_prefill call over the whole workload (active-tile compaction, paged
TMA loads, tcgen05 QK^T and PV, online softmax with e4m3 P, epilogue), inputs resident in HBM.
The default workload is the largest block-sparse one: a varlen batch of four prefills of
16384, 12000, 9000 and 4097 tokens, 64 query / 8 KV heads, page 32, per-token K and per-head V
descales, sparse index lists holding 25% of each Q tile's causal KV tiles (tile 0 and the
diagonal always in), two empty tasks.  The same JSON line reports the other full-size
workloads (2 x 8K block mask, 4K over a 64K cache, dense 32K), timed the same way, under
"other_workloads".

Metric: effective TFLOP/s over active tiles, FLOPs = sum over (task, active tile) of
4 * 128 * rows_valid * cols_valid.  Prints one JSON line (rank 0).

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]
Under torchrun every rank runs an independent replica of the workload (weak scaling; the
path has no data exchange), timed between barriers, max over ranks.
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = ("block-sparse FP8 prefill effective TFLOPS (active tiles) and ms/call, "
          "% FP8 roofline")
DEFAULT_WORKLOAD = "varlen_4x16k_h64kv8_idx25"
OTHER_WORKLOADS = ("prefill_2x8k_h32kv8_bsm50_outliers", "chunked_4k_over_64k_h32kv4_local_sink",
                   "dense_32k_h32kv8")
# workloads also timed with 256-wide macro blocks (two list tiles per online-softmax step)
MACRO_WORKLOADS = ("varlen_4x16k_h64kv8_idx25", "prefill_2x8k_h32kv8_bsm50_outliers",
                   "dense_32k_h32kv8")
FP8_PER_BF16 = 2.0        # nominal dense fp8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s)
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 512 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=W.WORKLOAD_ORDER)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the other full-size workloads (profiling runs)")
    ap.add_argument("--no-macro", action="store_true",
                    help="skip the 256-wide macro-block timings")
    ap.add_argument("--tiles-per-step", type=int, default=1, choices=[1, 2],
                    help="online-softmax step of the timed prefill: one 128-token tile, or a "
                         "256-wide macro block of two")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--op", choices=["prefill", "quantize"], default="prefill",
                    help="prefill (the hot path, default) or the quantise step that feeds it: "
                         "bf16 Q rows + K/V append of the workload's shapes")
    ap.add_argument("--batch", type=int, default=0,
                    help="keep only the first N sequences of the workload (profiling runs)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "hbm_gbs": 6800.0}, "fallback"


def max_over_ranks(values, device):
    """Element-wise maximum of a list of floats over the ranks of the default process group
    (the slowest replica sets the time); the values themselves with one rank."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def weak_scaling_value(world, work_per_replica, ms):
    """Whole-job throughput of `world` replicas each doing `work_per_replica` units in `ms`
    (the maximum over ranks): total units per second."""
    return world * work_per_replica / (ms * 1e-3)


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "bsa_attention_kernel__dram_traffic.json")
# the attention kernel's device code (its launch shape is fixed: one 640-thread CTA per SM)
KERNEL_SOURCES = ("bsa_attention.cuh", "bsa_common.cuh", "ptx_sm103.cuh")


def kernel_sources_digest():
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "block_sparse_fp8_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload):
    """DRAM bytes (read + write) per launch of the attention kernel on `workload`, from the
    committed ncu record; None when the record was taken on other kernel sources."""
    try:
        with open(TRAFFIC_RECORD) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_sources_sha256") != kernel_sources_digest():
        return None
    return rec.get("dram_bytes_per_launch", {}).get(workload)


def config_of(case, name, tiles, flops):
    Q = sum(-(-ql // 128) for ql in case.q_lens) * case.N1
    mask = ("block_mask" if case.block_mask is not None else
            "sparse_indices" if case.sparse_indices is not None else "dense")
    extra = {}
    if mask == "dense":
        # the FlashAttention convention: 4 * q * kv * D * N1 per sequence, halved when causal
        # (counts the masked half of the diagonal tiles out; the effective figure keeps them)
        fa = sum(4.0 * ql * kl * 128 * case.N1 * (0.5 if case.causal else 1.0)
                 for ql, kl in zip(case.q_lens, case.kv_lens))
        extra["fa_convention_gflop"] = round(fa / 1e9, 3)
    return {"workload": name, "B": case.B, "q_lens": case.q_lens, "kv_lens": case.kv_lens,
            "N1": case.N1, "N2": case.N2, "D": 128, "page_size": case.page_size,
            "k_scale": ["per_tensor", "per_token_head"][case.k_scale_kind],
            "v_scale": ["per_tensor", "", "per_head"][case.v_scale_kind],
            "mask": mask, "causal": bool(case.causal), "tasks": Q,
            "active_tiles": int(tiles), "effective_gflop": round(flops / 1e9, 3),
            "l2": "flushed (512 MiB write) before every step, outside the per-step events",
            **extra}


def cpu_info():
    import oracle

    return oracle.cpu_model(), os.cpu_count()


def _task_rows(case, lists, counts, chunk):
    """The (token, head) rows of the (b, h, q-tile) tasks in `chunk` and their effective FLOPs
    (4 * 128 * valid rows * valid keys of every active tile)."""
    rows, fl = [], 0
    for b, h, qt in chunk:
        q0, ql, kl = int(case.cu_seqlens_q[b]), case.q_lens[b], case.kv_lens[b]
        nr = min(128, ql - qt * 128)
        rows += [(q0 + qt * 128 + r, h) for r in range(nr)]
        ts = lists[b, h, qt, :counts[b, h, qt]].astype(np.int64)
        fl += 4 * 128 * nr * int(np.minimum(128, kl - ts * 128).sum())
    return np.array(rows, dtype=np.int32).reshape(-1, 2), fl


def _oracle_sample(orc, case, lists, counts, tasks, order, mode, seconds):
    """Times `mode` of the oracle on whole tasks taken in `order` until `seconds` have run."""
    done_flops, done_tasks, done_rows, t_total = 0, 0, 0, 0.0
    i = 0
    while t_total < seconds and i < len(order):
        chunk = [tasks[j] for j in order[i:i + 8]]
        i += 8
        rows, fl = _task_rows(case, lists, counts, chunk)
        t0 = time.perf_counter()
        orc.rows(rows, mode)
        t_total += time.perf_counter() - t0
        done_flops += fl
        done_tasks += len(chunk)
        done_rows += len(rows)
    return done_flops, done_tasks, done_rows, t_total


def cpu_baseline(case, lists, counts, seconds, seed=11):
    """The oracle (exact fp64 mode, all host threads) on a bounded sample of whole tasks; its
    P-emulating mode is timed beside it on a quarter of the time budget."""
    import oracle

    orc = oracle.Oracle(case)
    threads = orc.lib.oracle_max_threads()
    tasks = [(b, h, qt) for b in range(case.B) for h in range(case.N1)
             for qt in range(-(-case.q_lens[b] // 128))]
    order = np.random.default_rng(seed).permutation(len(tasks))
    fl, nt, nr, t = _oracle_sample(orc, case, lists, counts, tasks, order, oracle.EXACT, seconds)
    pfl, pnt, pnr, pt = _oracle_sample(orc, case, lists, counts, tasks, order, oracle.PEMU,
                                       seconds / 4)
    model, _ = cpu_info()
    return {"value": fl / t / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{nt} of {len(tasks)} (b, h, q-tile) tasks ({nr} rows), "
                      f"seeded random, exact fp64 mode, {t:.1f} s on {threads} threads "
                      f"({model})",
            "pemu": {"value": pfl / pt / 1e12, "unit": "TFLOP/s",
                     "sample": f"the first {pnt} of those tasks ({pnr} rows), P-emulating mode, "
                               f"{pt:.1f} s"}}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.bus_id = bus_id
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.bus_id:
            cmd += ["-i", self.bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

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
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def make_workload(args):
    kw = dict(W.WORKLOADS[args.workload])
    if args.batch:
        kw["q_lens"] = kw["q_lens"][:args.batch]
        kw["kv_lens"] = kw["kv_lens"][:args.batch]
    return W.make_case(args.workload, **kw)


def time_steps(step, steps, warmup, flush, stream, dev):
    """Per-step CUDA-event times (ms) of `steps` calls of step(), L2 flushed before each."""
    import torch

    for _ in range(warmup):
        flush.zero_()
        step()
    per = []
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        per.append(e0.elapsed_time(e1))
    return per


def macro_line(per, flops, fp8_peak):
    """The 256-wide macro-block run of a workload, timed like the 128-wide one."""
    ms = statistics.mean(per)
    return {"ms_per_call": {"mean": ms, "median": statistics.median(per), "min": min(per)},
            "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "roofline_frac": flops / (ms * 1e-3) / 1e12 / fp8_peak,
            "kernel": "bsa_attention_wide_kernel"}


def upload(case, dev):
    import torch

    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return dict(q=t(case.q), k_pages=t(case.k_pages), v_pages=t(case.v_pages),
                q_descale=t(case.q_descale), k_descale=t(case.k_descale),
                v_descale=t(case.v_descale), cu_seqlens_q=t(case.cu_seqlens_q),
                seqused_kv=t(case.seqused_kv), block_table=t(case.block_table),
                block_mask=t(case.block_mask), sparse_indices=t(case.sparse_indices),
                sparse_seq_len=t(case.sparse_seq_len))


def time_other_workload(name, steps, warmup, dev, flush, fp8_peak, traffic_of, macro=False):
    """One more full-size workload timed like the main one (L2 flushed before every step,
    CUDA events around each call); its buffers are freed before returning."""
    import torch

    import block_sparse_fp8_gb300 as bsa

    case = W.make_workload(name)
    d = upload(case, dev)
    dims = bsa.Dims(**case.dims())
    lists, counts = bsa.compact_tiles(d["cu_seqlens_q"], d["seqused_kv"], dims,
                                      block_mask=d["block_mask"],
                                      sparse_indices=d["sparse_indices"],
                                      sparse_seq_len=d["sparse_seq_len"])
    tiles, flops = W.active_work(case, (lists.cpu().numpy(), counts.cpu().numpy()))
    out = torch.empty((case.T, case.N1, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((case.N1, case.T), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    workspace = torch.empty(max(bsa.workspace_size(dims), 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(tiles_per_step=1):
        bsa.prefill(d["q"], d["k_pages"], d["v_pages"], d["q_descale"], d["k_descale"],
                    d["v_descale"], d["cu_seqlens_q"], d["seqused_kv"], d["block_table"],
                    case.max_q_len, case.max_kv_len, block_mask=d["block_mask"],
                    sparse_indices=d["sparse_indices"], sparse_seq_len=d["sparse_seq_len"],
                    softmax_scale=case.softmax_scale, p_scale=case.p_scale,
                    causal=bool(case.causal), out=out, lse=lse, dev_status=status,
                    workspace=workspace, stream=stream, k_scale_kind=case.k_scale_kind,
                    v_scale_kind=case.v_scale_kind, tiles_per_step=tiles_per_step)

    per = time_steps(step, steps, warmup, flush, stream, dev)
    per2 = time_steps(lambda: step(2), steps, warmup, flush, stream, dev) if macro else None
    if int(status.item()) != 0:
        raise RuntimeError(f"{name}: device status {int(status.item())}")
    ms = statistics.mean(per)
    achieved = flops / (ms * 1e-3) / 1e12
    res = {"ms_per_call": {"mean": ms, "median": statistics.median(per), "min": min(per)},
           "value": achieved, "unit": "TFLOP/s",
           "roofline": {"bound": "tensor", "achieved": achieved, "peak": fp8_peak,
                        "unit": "TFLOP/s", "frac": achieved / fp8_peak,
                        "traffic": traffic_of(name)},
           "config": config_of(case, name, tiles, flops)}
    if "fa_convention_gflop" in res["config"]:
        res["fa_convention_tflops"] = res["config"]["fa_convention_gflop"] * 1e9 / (ms * 1e-3) / 1e12
    if per2 is not None:
        res["macro_block_256"] = macro_line(per2, flops, fp8_peak)
    del d, out, lse, workspace
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world):
    import torch

    import block_sparse_fp8_gb300 as bsa
    from block_sparse_fp8_gb300 import _build

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    if _build.needs_build():
        if rank == 0:
            _build.build()
        if world > 1:
            torch.distributed.barrier()
    bsa.lib()

    case = make_workload(args)
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    d = dict(q=t(case.q), k_pages=t(case.k_pages), v_pages=t(case.v_pages),
             q_descale=t(case.q_descale), k_descale=t(case.k_descale),
             v_descale=t(case.v_descale), cu_seqlens_q=t(case.cu_seqlens_q),
             seqused_kv=t(case.seqused_kv), block_table=t(case.block_table),
             block_mask=t(case.block_mask), sparse_indices=t(case.sparse_indices),
             sparse_seq_len=t(case.sparse_seq_len))
    dims = bsa.Dims(**case.dims())
    lists, counts = bsa.compact_tiles(d["cu_seqlens_q"], d["seqused_kv"], dims,
                                      block_mask=d["block_mask"],
                                      sparse_indices=d["sparse_indices"],
                                      sparse_seq_len=d["sparse_seq_len"])
    lists, counts = lists.cpu().numpy(), counts.cpu().numpy()
    tiles, flops = W.active_work(case, (lists, counts))

    out = torch.empty((case.T, case.N1, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((case.N1, case.T), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    workspace = torch.empty(max(bsa.workspace_size(dims), 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(tiles_per_step=args.tiles_per_step):
        bsa.prefill(d["q"], d["k_pages"], d["v_pages"], d["q_descale"], d["k_descale"],
                    d["v_descale"], d["cu_seqlens_q"], d["seqused_kv"], d["block_table"],
                    case.max_q_len, case.max_kv_len, block_mask=d["block_mask"],
                    sparse_indices=d["sparse_indices"], sparse_seq_len=d["sparse_seq_len"],
                    softmax_scale=case.softmax_scale, p_scale=case.p_scale,
                    causal=bool(case.causal), out=out, lse=lse, dev_status=status,
                    workspace=workspace, stream=stream, k_scale_kind=case.k_scale_kind,
                    v_scale_kind=case.v_scale_kind, tiles_per_step=tiles_per_step)

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during warm-up")

    sampler = None
    if rank == 0 and not args.no_clocks:
        bus = None
        try:
            p = torch.cuda.get_device_properties(dev)
            bus = f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
        except AttributeError:
            bus = None
        sampler = ClockSampler(bus)
        sampler.start()
        time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop() if sampler else None
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(per) / len(per)
    ms, wall = max_over_ranks([ms, wall], dev)
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the timed region")

    # secondary figure: the same launch back to back with no flush, so that the inputs (the
    # ones that fit) stay in L2 between calls
    warm = []
    for _ in range(min(args.steps, 20)):
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        step()
        w1.record(stream)
        torch.cuda.synchronize(dev)
        warm.append(w0.elapsed_time(w1))

    # the same workload with 256-wide macro blocks (two list tiles per online-softmax step),
    # timed the same way after the timed region
    macro = None
    if (not args.no_macro and args.tiles_per_step == 1 and args.batch == 0 and
            args.workload in MACRO_WORKLOADS):
        per2 = time_steps(lambda: step(2), max(5, min(args.steps, 20)), max(args.warmup, 3),
                          flush, stream, dev)
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())} (macro blocks)")
        macro = per2

    # end to end through the C ABI's host-buffer call (bsa_fp8_prefill_host): every step copies
    # all of its inputs from pinned host memory to the device, runs the prefill and copies O
    # and the LSE back, all queued by the one call on one stream.  Consecutive steps alternate
    # between two streams with their own device buffers and workspaces, as a serving loop
    # would issue them, so that one step's copies overlap the other's prefill.
    e2e = None
    if not args.no_e2e:
        step()  # out / lse again hold this configuration's result (the macro timing reused them)
        host_in = {k: v.cpu().pin_memory() for k, v in d.items() if v is not None}
        sets = []
        for _ in range(2):
            dv = {k: torch.empty_like(v) for k, v in d.items() if v is not None}
            dv["out"], dv["lse"] = torch.empty_like(out), torch.empty_like(lse)
            hv = dict(host_in)
            hv["out"] = torch.empty(out.shape, dtype=out.dtype).pin_memory()
            hv["lse"] = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
            sets.append((hv, dv, torch.empty_like(workspace), torch.cuda.Stream(dev)))
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = out.numel() * 2 + lse.numel() * 4
        n_e2e = max(3, min(args.steps, 20))

        def e2e_step(i):
            hv, dv, ws, s = sets[i % 2]
            bsa.prefill_host(hv, dv, case.max_q_len, case.max_kv_len,
                             softmax_scale=case.softmax_scale, p_scale=case.p_scale,
                             causal=bool(case.causal), workspace=ws, dev_status=status,
                             stream=s, k_scale_kind=case.k_scale_kind,
                             v_scale_kind=case.v_scale_kind, tiles_per_step=args.tiles_per_step)

        e2e_step(0)
        e2e_step(1)
        torch.cuda.synchronize(dev)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _, _, _, s in sets:
            s.wait_event(ev0)                             # the first copies in are inside
        for i in range(n_e2e):
            e2e_step(i)
        for _, _, _, s in sets:
            done = torch.cuda.Event()
            done.record(s)
            stream.wait_event(done)                       # the last copies out are inside
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = ev0.elapsed_time(ev1) / n_e2e
        e2e_ms = max_over_ranks([e2e_ms], dev)[0]
        if int(status.item()) != 0:
            raise RuntimeError(f"device status {int(status.item())} in the end-to-end steps")
        # the host output of the last step is the device output of the timed region's launches
        hv_last = sets[(n_e2e - 1) % 2][0]
        if not (torch.equal(hv_last["out"], out.cpu()) and torch.equal(hv_last["lse"], lse.cpu())):
            raise RuntimeError("the host-buffer call's output differs from the device call's")
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        dev_in = [sets[0][1], sets[1][1]]
        dev_out = [(sets[0][1]["out"], sets[0][1]["lse"]), (sets[1][1]["out"], sets[1][1]["lse"])]
        host_out = [(sets[0][0]["out"], sets[0][0]["lse"]), (sets[1][0]["out"], sets[1][0]["lse"])]

        # the host link alone: the same copies with no prefill, each direction by itself and
        # both at once (the floor of a step under this overlap scheme)
        def copies_ms(do_in, do_out):
            torch.cuda.synchronize(dev)
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            s_in.wait_event(c0)
            s_out.wait_event(c0)
            for i in range(n_e2e):
                di, (o_b, l_b), (ho, hl) = dev_in[i % 2], dev_out[i % 2], host_out[i % 2]
                if do_in:
                    with torch.cuda.stream(s_in):
                        for k, v in host_in.items():
                            if v is not None:
                                di[k].copy_(v, non_blocking=True)
                if do_out:
                    with torch.cuda.stream(s_out):
                        ho.copy_(o_b, non_blocking=True)
                        hl.copy_(l_b, non_blocking=True)
            e_in, e_out = torch.cuda.Event(), torch.cuda.Event()
            e_in.record(s_in)
            e_out.record(s_out)
            stream.wait_event(e_in)
            stream.wait_event(e_out)
            c1.record(stream)
            torch.cuda.synchronize(dev)
            return c0.elapsed_time(c1) / n_e2e

        in_ms, out_ms, both_ms = copies_ms(True, False), copies_ms(False, True), copies_ms(True, True)
        e2e = {"value": weak_scaling_value(world, flops, e2e_ms) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms,
               "call": "bsa_fp8_prefill_host (host buffers in and out), two streams",
               "host_link": {"h2d_gbs": h2d / in_ms / 1e6, "d2h_gbs": d2h / out_ms / 1e6,
                             "copies_only_ms_per_step": both_ms,
                             "note": "the same per-step copies timed without the prefill"}}

    if rank != 0:
        return None
    pk, src = peaks()
    fp8_peak = pk.get("bf16_tflops", FALLBACK_BF16_TFLOPS) * FP8_PER_BF16
    achieved = flops / (ms * 1e-3) / 1e12
    traffic = measured_traffic(args.workload) if args.batch == 0 else None
    hbm_peak = pk.get("hbm_gbs", 6800.0)
    hbm = None if traffic is None else {
        "achieved": traffic / (ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
        "frac": traffic / (ms * 1e-3) / 1e9 / hbm_peak,
        "note": "recorded DRAM bytes per launch over the measured launch time"}
    line = {
        "metric": METRIC, "value": weak_scaling_value(world, flops, ms) / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3 (fp32 accumulate)", "data": "synthetic (seeded)",
        "config": config_of(case, args.workload, tiles, flops),
        "ms_per_call": {"mean": ms, "median": statistics.median(per), "min": min(per)},
        "warm_l2_ms_per_call": {"median": statistics.median(warm), "min": min(warm),
                                "tflops_at_median": flops / (statistics.median(warm) * 1e-3) / 1e12,
                                "note": "no flush between calls; secondary to the flushed value"},
        "wall_ms_per_step_incl_flush": wall * 1e3 / args.steps,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": achieved / fp8_peak, "traffic": traffic,
                     "hbm": hbm,
                     "peak_source": f"{src}: bf16 {'burst' if src == 'measured' else ''} "
                                    f"{pk.get('bf16_tflops')} TFLOP/s x {FP8_PER_BF16} "
                                    f"(nominal fp8/bf16 ratio)",
                     "kernel": "bsa_attention_kernel"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "e2e": e2e,
    }
    if "fa_convention_gflop" in line["config"]:
        line["fa_convention_tflops"] = (weak_scaling_value(world, line["config"]["fa_convention_gflop"] * 1e9, ms)
                                        / 1e12)
    if args.tiles_per_step == 2:
        line["config"]["tiles_per_step"] = 2
        line["roofline"]["kernel"] = "bsa_attention_wide_kernel"
    if macro is not None:
        line["macro_block_256"] = macro_line(macro, flops, fp8_peak)
    # the CPU baseline and the other workloads belong to the one-GPU line: under torchrun the
    # other ranks have finished and would wait on rank 0 for them
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(case, lists, counts, args.cpu_seconds)
    if not args.no_others and args.batch == 0 and world == 1:
        # the other full-size workloads, one after the other on this GPU (not part of the
        # timed region above)
        del d, out, lse
        torch.cuda.empty_cache()
        steps = max(5, min(args.steps, 20))
        line["other_workloads"] = {
            name: time_other_workload(name, steps, max(args.warmup, 3), dev, flush, fp8_peak,
                                      measured_traffic,
                                      macro=not args.no_macro and name in MACRO_WORKLOADS)
            for name in OTHER_WORKLOADS if name != args.workload}
    return line


def run_reference(args, rank):
    """The CPU oracle, as it stands, on the host cores: each step a bounded sample of tasks."""
    if rank != 0:
        return None
    import oracle

    case = make_workload(args)
    orc = oracle.Oracle(case)
    lists, counts, _err = orc.lists()
    tiles, flops = W.active_work(case, (lists, counts))
    tasks = [(b, h, qt) for b in range(case.B) for h in range(case.N1)
             for qt in range(-(-case.q_lens[b] // 128))]
    rng = np.random.default_rng(5)
    per_step_tasks = 4
    threads = orc.lib.oracle_max_threads()

    def step(i):
        sel = rng.choice(len(tasks), per_step_tasks, replace=False)
        rows, fl = _task_rows(case, lists, counts, [tasks[j] for j in sel])
        t0 = time.perf_counter()
        orc.rows(rows, oracle.EXACT)
        return fl, time.perf_counter() - t0

    for i in range(max(args.warmup, 3)):
        step(i)
    tot_f, tot_t = 0, 0.0
    for i in range(args.steps):
        f, dt = step(i)
        tot_f += f
        tot_t += dt
    value = tot_f / tot_t / 1e12
    model, _ = cpu_info()
    sample = (f"{per_step_tasks} seeded random (b, h, q-tile) tasks per step of {len(tasks)}, "
              f"exact fp64 mode, {threads} threads ({model})")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": tot_t * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": config_of(case, args.workload, tiles, flops),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def run_quantize(args, rank, world):
    """The quantise step at the workload's shapes: bsa_fp8_quantize_rows over Q [T, N1, 128]
    bf16 and bsa_fp8_append_kv of all K/V tokens [T_kv, N2, 128] bf16 (per-token K, per-head
    V) into fresh pages.  HBM-bound: value = algorithmic bytes / time."""
    import torch

    import block_sparse_fp8_gb300 as bsa
    from block_sparse_fp8_gb300 import _build

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    if _build.needs_build():
        if rank == 0:
            _build.build()
        if world > 1:
            torch.distributed.barrier()
    bsa.lib()
    w = dict(W.WORKLOADS[args.workload])
    q_lens, kv_lens, N1, N2, ps = w["q_lens"], w["kv_lens"], w["N1"], w["N2"], w["page_size"]
    T, Tkv, B = sum(q_lens), sum(kv_lens), len(kv_lens)
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + rank)
    q = torch.randn((T, N1, 128), generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn((Tkv, N2, 128), generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn((Tkv, N2, 128), generator=g, device=dev).to(torch.bfloat16)
    pages = [-(-kv // ps) for kv in kv_lens]
    P, L = sum(pages), max(pages)
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(5)).to(torch.int32)
    bt = torch.full((B, L), -1, dtype=torch.int32)
    o = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[o:o + n]
        o += n
    bt = bt.to(dev)
    cu_new = torch.tensor([0] + list(np.cumsum(kv_lens)), dtype=torch.int32, device=dev)
    cache_len = torch.zeros(B, dtype=torch.int32, device=dev)
    k_pages = torch.zeros((P, N2, ps, 128), dtype=torch.uint8, device=dev)
    v_pages = torch.zeros_like(k_pages)
    k_desc = torch.zeros((P, N2, ps), dtype=torch.float32, device=dev)
    v_scale = torch.full((N2,), 4.0 / 448.0, dtype=torch.float32, device=dev)
    q8 = torch.empty((T, N1, 128), dtype=torch.uint8, device=dev)
    qd = torch.empty((T, N1), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        bsa.quantize_rows(q, q8, qd)
        bsa.append_kv(k, v, cu_new, cache_len, bt, k_pages, v_pages, k_descale=k_desc,
                      v_scale=v_scale, dev_status=status)

    # algorithmic bytes: bf16 in, e4m3 out, one fp32 descale per row (Q and K); block table
    # and lengths are negligible
    nbytes = T * N1 * (256 + 128 + 4) + Tkv * N2 * (2 * (256 + 128) + 4)
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    per = []
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0.record()
        step()
        e1.record()
        torch.cuda.synchronize()
        per.append(e0.elapsed_time(e1))
    ms = max_over_ranks([statistics.mean(per)], dev)[0]
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    # each kernel alone, timed the same way (after the timed region)
    def alone(fn):
        ts = []
        for _ in range(max(5, min(args.steps, 20))):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    q_bytes = T * N1 * (256 + 128 + 4)
    kv_bytes = nbytes - q_bytes
    q_ms = alone(lambda: bsa.quantize_rows(q, q8, qd))
    kv_ms = alone(lambda: bsa.append_kv(k, v, cu_new, cache_len, bt, k_pages, v_pages,
                                        k_descale=k_desc, v_scale=v_scale, dev_status=status))
    if rank != 0:
        return None
    pk, src = peaks()
    hbm = pk.get("hbm_gbs", 6800.0)
    achieved = nbytes / (ms * 1e-3) / 1e9
    per_kernel = {
        name: {"ms_median": t, "bytes": b, "gbs": b / (t * 1e-3) / 1e9,
               "frac": b / (t * 1e-3) / 1e9 / hbm}
        for name, t, b in (("quantize_rows_kernel", q_ms, q_bytes),
                           ("append_kv_kernel", kv_ms, kv_bytes))}
    return {
        "metric": "quantise step (bf16 Q rows -> e4m3 + descale, K/V append into pages) "
                  "HBM throughput",
        "value": weak_scaling_value(world, nbytes, ms) / 1e9, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 -> fp8_e4m3",
        "data": "synthetic (seeded normal)",
        "config": {"workload": args.workload, "op": "quantize", "q_rows": T * N1,
                   "kv_rows": Tkv * N2, "page_size": ps, "k_scale": "per_token_head",
                   "v_scale": "per_head", "bytes_per_step": nbytes,
                   "l2": "flushed (512 MiB write) before every step, outside the events"},
        "ms_per_call": {"mean": ms, "median": statistics.median(per), "min": min(per)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": None,
                     "peak_source": f"{src}: copy bandwidth", "kernel": "quantize_rows + append_kv"},
        "per_kernel": per_kernel,
        "gpu_launches": 2 * args.steps,
    }


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference" and args.op == "quantize":
        line = {"impl": "reference", "unavailable": "the reference arm times the attention oracle only"}
        if rank != 0:
            line = None
    elif args.impl == "reference":
        line = run_reference(args, rank)
    elif args.op == "quantize":
        line = run_quantize(args, rank, world)
    else:
        line = run_ours(args, rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)
    if args.impl == "ours" and world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
