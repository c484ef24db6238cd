#!/usr/bin/env python3
"""Benchmark of the GB300 speculative-sampling verifier.

One step = one spec_verify call over one batch of the largest-vocabulary
workload (B=256 requests, K=3 drafts, V=151936, bf16 logits, ragged
num_draft ~ U{0..3}, 25% greedy), inputs resident in HBM.  Prints one JSON
line (rank 0).

  value     verified draft positions / s (sum_b num_draft[b] per call),
            device-timed with CUDA events around each call; L2 is flushed
            before every timed call (256 MiB written, then another 256 MiB
            read, so that it holds clean unrelated lines).
  e2e       same metric through spec_verify_host: from pinned host inputs
            only the rows the verifier reads are copied in, then verified,
            outputs copied back, all inside the timed region.
  roofline  the dominant kernel of the verifier spec_verify runs for the
            workload: k_verify when it verifies request by request (bytes:
            rows 0..a_b of every request + the q row of each residual draw +
            the small terms), k_row_stats when it runs the all-rows pass
            (bytes: every valid logits row once); bytes per launch / its
            CUDA-event duration, against the measured HBM copy bandwidth.
  cpu_baseline  the float64 oracle on the host cores, on a bounded sample.

--impl reference times the oracle (the only reference this method has) on
the same workload and prints the same line with "impl": "reference".
Multi-GPU (torchrun): every rank verifies its own batch of the workload
(request indices offset by rank * B): weak scaling, no collective on the
data path.
"""
from __future__ import annotations

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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "verified draft positions/sec and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "positions/s"
PEAK_FALLBACK_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
TILE = 2048  # tokens per row-statistics chunk (one 16-byte partial each)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=4, help="workload 1..5 (default 4)")
    ap.add_argument("--batch", type=int, default=None, help="leading-B subset (sweep)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--oracle-seconds", type=float, default=1.0,
                    help="budget of each per-config oracle timing (1 thread, all cores)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config table (every workload and config 5's B sweep)")
    ap.add_argument("--mode", choices=["chain", "typical", "tree", "early_exit", "lmhead"], default="chain",
                    help="chain: the lossless / greedy verifier (the headline line); "
                         "typical: typical acceptance on the same workload; tree: "
                         "token-tree verification of tries with --tree-nodes nodes; "
                         "early_exit: the verifier that stops reading a request's rows at "
                         "its first rejection, timed beside the all-rows verifier; lmhead: "
                         "the verifier fed with hidden states (the fused tcgen05 LM-head "
                         "projection), timed beside separate projections")
    ap.add_argument("--hidden", type=int, default=4096, help="hidden size H of --mode lmhead")
    ap.add_argument("--threshold", type=float, default=0.01, help="typical acceptance threshold")
    ap.add_argument("--tree-nodes", type=int, default=16)
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured", d
    except Exception:
        return PEAK_FALLBACK_GBS, "fallback", {}


# the sources each dominant kernel is compiled from, and the committed file
# with its ncu DRAM bytes per launch
KERNEL_SOURCES = {
    "k_verify": (("verify.cu", "stats.cuh", "draw.cuh", "accept.cuh", "common.cuh"),
                 "verify_traffic.json"),
    "k_row_stats": (("row_stats.cu", "stats.cuh", "accept.cuh", "common.cuh"),
                    "row_stats_traffic.json"),
}


def kernel_sha(kernel="k_verify"):
    """Digest of the sources `kernel` is compiled from."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel][0]:
        h.update(open(os.path.join(ROOT, "speculative_decoding_verification_51_gb300", "csrc", f),
                      "rb").read())
    return h.hexdigest()[:16]


def verify_sha():
    return kernel_sha("k_verify")


def profiled_traffic(workload_name: str, kernel="k_verify"):
    """ncu DRAM bytes per launch of `kernel` for this workload, if the
    committed summary was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", KERNEL_SOURCES[kernel][1])
    try:
        d = json.load(open(p))
    except Exception:
        return None
    if d.get("source_sha") != kernel_sha(kernel):
        return None
    e = d.get("workloads", {}).get(workload_name)
    return None if e is None else float(e["dram_bytes_per_launch"])


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled through NVML every
    millisecond during the timed region (falls back to nvidia-smi at 100 ms)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device: torch.device):
        self.device = device
        self.samples = []  # (sm_mhz, max_mhz, reason_bits)
        self.stop = threading.Event()
        self.nvml = None
        self.handle = None
        self.source = None
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            props = torch.cuda.get_device_properties(device)
            uuid = str(getattr(props, "uuid", ""))
            h = ctypes.c_void_p()
            ok = False
            if uuid:
                ok = nv.nvmlDeviceGetHandleByUUID(f"GPU-{uuid}".encode(), ctypes.byref(h)) == 0
            if not ok:
                vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
                idx = int(vis.split(",")[device.index or 0]) if vis and vis.split(",")[0].isdigit() \
                    else (device.index or 0)
                ok = nv.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(h)) == 0
            if not ok:
                raise OSError("no NVML handle")
            self.nvml, self.handle, self.ct = nv, h, ctypes
            self.getreasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.source = "nvml"
        except Exception:
            self.nvml = None

    def _poll(self):
        ct, nv, h = self.ct, self.nvml, self.handle
        mhz, mx, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        while not self.stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz)) == 0 and \
                    nv.nvmlDeviceGetMaxClockInfo(h, 1, ct.byref(mx)) == 0 and \
                    self.getreasons(h, ct.byref(rs)) == 0:
                self.samples.append((mhz.value, mx.value, rs.value))
            time.sleep(0.001)

    def _smi(self):
        try:
            proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device.index or 0),
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        self.source = "nvidia-smi"
        while not self.stop.is_set():
            ln = proc.stdout.readline()
            if not ln:
                break
            parts = [x.strip() for x in ln.split(",")]
            try:
                self.samples.append((float(parts[0]), float(parts[1]), int(parts[2], 16)))
            except (ValueError, IndexError):
                pass
        proc.terminate()

    def __enter__(self):
        self.t = threading.Thread(target=self._poll if self.nvml else self._smi, daemon=True)
        self.t.start()
        return self

    def __exit__(self, *a):
        self.stop.set()
        self.t.join(timeout=5)

    def summary(self):
        if not self.samples:
            return None
        reasons = set()
        for _, _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(x[0] for x in self.samples),
                "sm_max_mhz": max(x[1] for x in self.samples), "reasons": sorted(reasons),
                "samples": len(self.samples), "source": self.source}


def workload_name(cid, B):
    return f"config{cid}" + (f"_B{B}" if B else "")


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    from speculative_decoding_verification_51_gb300 import workloads as W
    w = W.make_workload(args.config, device="cpu")
    if args.batch:
        w = w.leading(args.batch)
    inputs = W.to_numpy(w)
    pos = W.positions(w.num_draft)
    threads = oracle.omp_threads()
    oracle.spec_verify(**inputs, n_threads=threads)  # warm (build, page in)
    for _ in range(max(0, args.warmup - 1)):
        oracle.spec_verify(**inputs, n_threads=threads)
    t = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.spec_verify(**inputs, n_threads=threads)
        t.append(time.perf_counter() - t0)
    sec = sum(t) / len(t)
    value = pos / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"{workload_name(args.config, args.batch)}: {w.spec.description}",
                       "B": w.B, "K": w.K, "V": w.V, "positions_per_step": pos},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"the whole batch ({w.B} requests) per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(w, budget_s):
    import oracle
    from speculative_decoding_verification_51_gb300 import workloads as W
    inputs = W.to_numpy(w)
    threads = oracle.omp_threads()
    pos = W.positions(w.num_draft)
    oracle.spec_verify(**inputs, n_threads=threads)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.spec_verify(**inputs, n_threads=threads)
        reps += 1
        if time.perf_counter() - t0 >= budget_s or reps >= 50:
            break
    sec = (time.perf_counter() - t0) / reps
    return {"value": pos / sec, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"the whole batch ({w.B} requests, {pos} positions) x {reps} "
                      f"repetitions, {sec * 1e3:.1f} ms each"}


def run_variant(args, rank, world, local):
    """Device time per call of the typical-acceptance or token-tree verifier
    (L2 flushed before every call, CUDA events on the call's stream)."""
    from speculative_decoding_verification_51_gb300 import binding
    from speculative_decoding_verification_51_gb300 import build as _build
    from speculative_decoding_verification_51_gb300 import workloads as W
    from speculative_decoding_verification_51_gb300 import sharding

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.build()
    binding.lib()
    spec = W.SPECS[args.config]
    esz = 2 if spec.dtype == "bf16" else 4
    if args.mode == "typical":
        w = W.make_workload(args.config, device=dev)
        B, K, V = w.B, w.K, w.V
        offset = sharding.weak_offset(rank, B)
        pos = W.positions(w.num_draft)
        ws = binding.new_workspace(B, K, V, dev)
        out_ids = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
        out_nacc = torch.empty((B,), dtype=torch.int32, device=dev)
        rows = W.valid_rows(w.num_draft)
        algo = rows * V * esz + B * (K * 4 + 8) + B * ((K + 1) * 4 + 4)

        def step(seed):
            binding.spec_verify_typical(w.target_logits, w.draft_ids, w.num_draft, w.temperature,
                                        args.threshold, seed, out_ids=out_ids,
                                        out_num_accepted=out_nacc, workspace=ws,
                                        request_offset=offset)
        wname = (f"config{args.config} ({spec.description}), typical acceptance, "
                 f"threshold {args.threshold}")
    else:
        N = args.tree_nodes
        tw = W.make_tree_workload(spec.B, N, spec.V, bf16=spec.dtype == "bf16",
                                  seed=args.config, device=dev)
        B, V = spec.B, spec.V
        offset = sharding.weak_offset(rank, B)
        pos = int((tw.nodes.long() - 1).sum())
        ws = torch.empty(binding.lib().spec_verify_tree_workspace_size(B, N, V),
                         dtype=torch.uint8, device=dev)
        rows = int(tw.nodes.long().sum())
        algo = rows * V * esz + B * N * 8 + B * (N * 4 + 8)  # every node row once; lower bound

        def step(seed):
            binding.spec_verify_tree(tw.logits, tw.probs, tw.tokens, tw.parents, tw.nodes,
                                     tw.temp, seed, workspace=ws, request_offset=offset)
        wname = (f"token trees: B={B} tries of up to {N} nodes (num_nodes ~ U{{1..{N}}}), "
                 f"V={V} {spec.dtype} logits, 30% greedy")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2(i):
        flush.fill_(i & 0xFF)
        flush_rd.sum()

    for i in range(args.warmup):
        flush_l2(i)
        step(1000 + i)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        for i in range(args.steps):
            flush_l2(i + 7)
            evs[i][0].record(stream)
            step(2000 + i)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    ms = sharding.max_over_ranks(ms, device=dev)
    peak, peak_kind, _ = measured_peak()
    gbs = algo / (ms * 1e-3) / 1e9
    # tree: plan, row stats, walk; typical: plan, row stats, accept, emit (no
    # residual draws, so no k_sample)
    n_kernels = 3 if args.mode == "tree" else 4
    line = {
        "metric": METRIC, "value": world * pos / (ms * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "mode": args.mode,
        "config": {"workload": wname, "positions_per_step": pos,
                   "l2": "flushed before every timed call: 256 MiB write, then 256 MiB read"},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "traffic": None, "kernel": "whole call",
                     "algorithmic_bytes_per_launch": algo, "peak_kind": peak_kind},
        "gpu_launches": n_kernels * args.steps, "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_early_exit(args, rank, world, local):
    """The early-exit verifier (one pass per draft position, requests dropped
    at their first rejection) against the all-rows verifier on the same
    workload: both captured in CUDA graphs with the seed in device memory,
    replayed alternately, L2 flushed before every replay."""
    from speculative_decoding_verification_51_gb300 import binding
    from speculative_decoding_verification_51_gb300 import build as _build
    from speculative_decoding_verification_51_gb300 import workloads as W
    from speculative_decoding_verification_51_gb300 import sharding

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.build()
    binding.lib()
    w = W.make_workload(args.config, device=dev)
    if args.batch:
        w = w.leading(args.batch)
    B, K, V = w.B, w.K, w.V
    esz = 2 if w.target_logits.dtype == torch.bfloat16 else 4
    offset = sharding.weak_offset(rank, B)
    pos = W.positions(w.num_draft)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2(i):
        flush.fill_(i & 0xFF)
        flush_rd.sum()

    seed_buf = torch.zeros(1, dtype=torch.int64, device=dev)
    graphs, outs, keep = {}, {}, {}
    for name, ee in (("all_rows", False), ("early_exit", True)):
        ws = binding.new_workspace(B, K, V, dev)
        oi = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
        on = torch.empty((B,), dtype=torch.int32, device=dev)

        def call(st, ws=ws, oi=oi, on=on, ee=ee):
            binding.spec_verify(w.target_logits, w.draft_probs, w.draft_ids, w.num_draft,
                                w.temperature, 0, out_ids=oi, out_num_accepted=on,
                                workspace=ws, request_offset=offset, seed_dev=seed_buf,
                                stream=st, early_exit=ee)
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            call(cap)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            call(cap)
        torch.cuda.synchronize()
        # the graph keeps the raw pointers: hold its buffers for its lifetime
        graphs[name], outs[name], keep[name] = g, (oi, on), ws
    for i in range(args.warmup):
        for g in graphs.values():
            flush_l2(i)
            seed_buf.fill_(1500 + i)
            g.replay()
    torch.cuda.synchronize()

    evs = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)] for n in graphs}
    nacc_log = torch.empty((args.steps, B), dtype=torch.int32, device=dev)
    same = torch.ones(args.steps, dtype=torch.bool, device=dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        for i in range(args.steps):
            seed_buf.fill_(2000 + i)
            for n, g in graphs.items():
                flush_l2(i + 7)
                evs[n][i][0].record(stream)
                g.replay()
                evs[n][i][1].record(stream)
            nacc_log[i].copy_(outs["early_exit"][1])
            same[i] = (outs["early_exit"][0] == outs["all_rows"][0]).all() & \
                (outs["early_exit"][1] == outs["all_rows"][1]).all()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = {n: sharding.max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in e), device=dev)
          for n, e in evs.items()}
    nl = nacc_log.cpu().long()
    n = w.num_draft.cpu().long()
    valid = nl >= 0
    rows_read = float(((nl + 1) * valid).sum(1).float().mean())
    rows_all = float(((n + 1) * valid[0]).sum())
    sampling = (w.temperature.cpu() > 0)
    resid = float(((nl < n) & valid & sampling).sum(1).float().mean())
    small = B * (K * 4 + 8) + B * ((K + 1) * 4 + 4)
    algo_ee = rows_read * V * esz + resid * V * 4 + small
    algo_all = rows_all * V * esz + resid * V * 4 + small
    peak, peak_kind, _ = measured_peak()
    gbs = algo_ee / (ms["early_exit"] * 1e-3) / 1e9
    wname = workload_name(args.config, args.batch)
    line = {
        "metric": METRIC, "value": world * pos / (ms["early_exit"] * 1e-3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms["early_exit"], 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "mode": "early_exit",
        "config": {"workload": f"{wname}: {w.spec.description}", "B": B, "K": K, "V": V,
                   "positions_per_step": pos,
                   "l2": "flushed before every timed replay: 256 MiB write, then 256 MiB read",
                   "launch": "each verifier captured in its own CUDA graph (seed in device "
                             "memory), the two replayed alternately"},
        "all_rows_ms_per_step": round(ms["all_rows"], 5),
        "speedup_vs_all_rows": round(ms["all_rows"] / ms["early_exit"], 4),
        "outputs_identical_all_steps": bool(same.all().item()),
        "rows_read_per_step": rows_read, "rows_all_rows_pass": rows_all,
        "bytes_early_exit": algo_ee, "bytes_all_rows": algo_all,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "traffic": None, "kernel": "whole call",
                     "algorithmic_bytes_per_launch": algo_ee, "peak_kind": peak_kind},
        # early exit: plan, K + 1 passes, sample, emit; all rows: plan, row
        # stats, accept, sample, emit
        "gpu_launches": (K + 4 + 5) * args.steps, "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_lmhead(args, rank, world, local):
    """The fused logits producer: the verifier fed with the target's hidden
    states and LM head (spec_verify_lmhead), against the same verification
    fed with logits from a separate projection (this library's tcgen05 GEMM,
    or cuBLAS through torch.matmul), L2 flushed before every timed call."""
    from speculative_decoding_verification_51_gb300 import binding
    from speculative_decoding_verification_51_gb300 import build as _build
    from speculative_decoding_verification_51_gb300 import workloads as W
    from speculative_decoding_verification_51_gb300 import sharding

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.build()
    binding.lib()
    spec = W.SPECS[args.config]
    B, K, V, H = spec.B, spec.K, spec.V, args.hidden
    w = W.make_lmhead_workload(B, K, V, H, seed=args.config, ragged=args.config != 3,
                               device=dev)
    offset = sharding.weak_offset(rank, B)
    n = w.num_draft.long()
    pos = int(n.sum())
    rows = int((n + 1).sum())
    K1 = K + 1
    ws = torch.empty(binding.lib().spec_verify_lmhead_workspace_size(B, K, V, H),
                     dtype=torch.uint8, device=dev)
    logits = torch.empty((B, K1, V), dtype=torch.bfloat16, device=dev)
    out_ids = torch.empty((B, K1), dtype=torch.int32, device=dev)
    out_nacc = torch.empty((B,), dtype=torch.int32, device=dev)
    ws2 = binding.new_workspace(B, K, V, dev)
    # the listed rows' hidden states, for the projection-only timings
    valid = (torch.arange(K1, device=dev)[None, :] <= n.to(dev)[:, None]).reshape(-1)
    hid_rows = w.hidden.reshape(B * K1, H)[valid].contiguous()
    lg_rows = torch.empty((rows, V), dtype=torch.bfloat16, device=dev)
    hid_all = w.hidden.reshape(B * K1, H)
    lg_all = logits.reshape(B * K1, V)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2(i):
        flush.fill_(i & 0xFF)
        flush_rd.sum()

    def fused(seed):
        binding.spec_verify_lmhead(w.hidden, w.lm_head, w.draft_probs, w.draft_ids, w.num_draft,
                                   w.temperature, seed, logits_out=logits, out_ids=out_ids,
                                   out_num_accepted=out_nacc, workspace=ws,
                                   request_offset=offset)

    def gemm_ours(seed):
        binding.lmhead_logits(hid_rows, w.lm_head, out=lg_rows)

    def gemm_cublas(seed):
        torch.matmul(hid_rows, w.lm_head.T, out=lg_rows)

    def two_step_cublas(seed):  # an engine's unfused step: project every row, then verify
        torch.matmul(hid_all, w.lm_head.T, out=lg_all)
        binding.spec_verify(logits, w.draft_probs, w.draft_ids, w.num_draft, w.temperature, seed,
                            out_ids=out_ids, out_num_accepted=out_nacc, workspace=ws2,
                            request_offset=offset)

    variants = {"fused": fused, "gemm_ours": gemm_ours, "gemm_cublas": gemm_cublas,
                "two_step_cublas": two_step_cublas}
    for i in range(args.warmup):
        for f in variants.values():
            flush_l2(i)
            f(1000 + i)
    torch.cuda.synchronize()
    evs = {k: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)] for k in variants}
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        for i in range(args.steps):
            for k, f in variants.items():
                flush_l2(i + 7)
                evs[k][i][0].record(stream)
                f(2000 + i)
                evs[k][i][1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = {k: sharding.max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in e), device=dev)
          for k, e in evs.items()}
    flops = 2.0 * rows * V * H
    d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = float(d.get("bf16_tflops", 1900.0))
    tf_fused = flops / (ms["fused"] * 1e-3) / 1e12
    tf_ours = flops / (ms["gemm_ours"] * 1e-3) / 1e12
    tf_cublas = flops / (ms["gemm_cublas"] * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": world * pos / (ms["fused"] * 1e-3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms["fused"], 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 x bf16 -> f32 (projection); f32 (verification)",
        "data": "synthetic", "mode": "lmhead",
        "config": {"workload": f"{workload_name(args.config, None)} shapes (B={B}, K={K}, "
                               f"V={V}) fed as hidden states, H={H}, integer operands",
                   "rows_projected": rows, "positions_per_step": pos,
                   "l2": "flushed before every timed call: 256 MiB write, then 256 MiB read"},
        "ms": {k: round(v, 5) for k, v in ms.items()},
        "tflops": {"fused_whole_call": round(tf_fused, 1), "gemm_ours": round(tf_ours, 1),
                   "gemm_cublas": round(tf_cublas, 1)},
        "speedup_fused_vs_two_step_cublas": round(ms["two_step_cublas"] / ms["fused"], 4),
        "roofline": {"bound": "tensor", "achieved": round(tf_fused, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tf_fused / peak, 4), "traffic": None,
                     "kernel": "whole fused call (projection of the listed rows)",
                     "algorithmic_flops_per_launch": flops,
                     "peak_kind": "measured (cuBLAS bf16 burst)"},
        # fused: plan, gather, projection, accept, sample, emit; projection
        # alone: 1; cuBLAS + spec_verify: the five verification kernels
        "gpu_launches": (6 + 1 + 5) * args.steps, "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.mode == "early_exit":
        run_early_exit(args, rank, world, local)
        return
    if args.mode == "lmhead":
        run_lmhead(args, rank, world, local)
        return
    if args.mode != "chain":
        run_variant(args, rank, world, local)
        return

    run_chain(args, rank, world, local)



# ---------------------------------------------------------------- chain mode

SWEEP = ((5, 32), (5, 128))  # config 5's B sweep (B = 512 is config 5 itself)


def call_bytes(w, nacc_log):
    """Bytes per call, averaged over the calls whose a_b are in nacc_log
    [calls, B]: 'algorithmic' = every valid logits row 0..n_b once + the q row
    of each residual draw + the q(x_j) gathers + ids, counts, temperatures and
    outputs; 'literal' = logits + draft probabilities once (rows 0..n_b and
    q rows 0..n_b-1); 'read' = what a verifier that stops at the first
    rejection must read: rows 0..a_b, the residual q rows, the same small
    terms."""
    n = w.num_draft.long().cpu()
    T = w.temperature.cpu()
    V, esz = w.V, (2 if w.target_logits.dtype == torch.bfloat16 else 4)
    ok = (n >= 0) & (n <= w.K)
    samp = (T > 0) & ok
    nl = nacc_log.long()
    valid = nl >= 0
    resid = ((nl < n[None]) & valid & samp[None]).sum(1).double().mean().item()
    rows_read = ((nl + 1) * valid).sum(1).double().mean().item()
    small = w.B * (w.K * 4 + 8) + w.B * ((w.K + 1) * 4 + 4) + int(n[samp].sum()) * 4
    rows_all = int(((n + 1) * ok).sum())
    return {"algorithmic": rows_all * V * esz + resid * V * 4 + small,
            "literal": rows_all * V * esz + int((n * ok).sum()) * V * 4,
            "read": rows_read * V * esz + resid * V * 4 + small,
            "rows_all": rows_all, "rows_read": rows_read, "residual_rows": resid}


class Caller:
    """One verification call on a workload, captured in a CUDA graph with the
    seed read from device memory (a step writes its seed, then replays)."""

    def __init__(self, w, dev, offset, all_rows=False, by_request=False):
        from speculative_decoding_verification_51_gb300 import binding
        self.w, self.dev, self.binding = w, dev, binding
        B, K, V = w.B, w.K, w.V
        self.ws = binding.new_workspace(B, K, V, dev)
        self.out_ids = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
        self.out_nacc = torch.empty((B,), dtype=torch.int32, device=dev)
        self.seed_buf = torch.zeros(1, dtype=torch.int64, device=dev)
        self.offset, self.all_rows, self.by_request = offset, all_rows, by_request
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cap):
            self._call(cap)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=cap):
            self._call(cap)
        torch.cuda.synchronize()

    def _call(self, st):
        w = self.w
        self.binding.spec_verify(w.target_logits, w.draft_probs, w.draft_ids, w.num_draft,
                                 w.temperature, 0, out_ids=self.out_ids,
                                 out_num_accepted=self.out_nacc, workspace=self.ws,
                                 request_offset=self.offset, seed_dev=self.seed_buf, stream=st,
                                 all_rows=self.all_rows, by_request=self.by_request)

    def direct(self, seed):
        w = self.w
        self.binding.spec_verify(w.target_logits, w.draft_probs, w.draft_ids, w.num_draft,
                                 w.temperature, seed, out_ids=self.out_ids,
                                 out_num_accepted=self.out_nacc, workspace=self.ws,
                                 request_offset=self.offset, all_rows=self.all_rows,
                                 by_request=self.by_request)


class L2Flush:
    """Write 256 MiB, then read another 256 MiB: the L2 ends up full of clean
    lines of unrelated data, so the timed call neither hits its own inputs in
    L2 nor pays for write-backs it did not cause."""

    def __init__(self, dev):
        self.a = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.b = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def __call__(self, i):
        self.a.fill_(i & 0xFF)
        self.b.sum()


def time_replays(c, steps, stream, flush=None, seed0=2000):
    """Device time (ms) of each of `steps` graph replays, L2 flushed before
    each when `flush` is given; the a_b of every replay are kept."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    nacc_log = torch.empty((steps, c.w.B), dtype=torch.int32, device=c.dev)
    for i in range(steps):
        if flush is not None:
            flush(i + 7)
        c.seed_buf.fill_(seed0 + i)
        evs[i][0].record(stream)
        c.graph.replay()
        evs[i][1].record(stream)
        nacc_log[i].copy_(c.out_nacc)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs], nacc_log.cpu()


def oracle_rate(w, threads, budget_s):
    """The float64 oracle (as it stands) on a bounded leading sample of the
    workload's requests: (positions/s, the sample, threads used)."""
    import oracle
    from speculative_decoding_verification_51_gb300 import workloads as W
    inputs = W.to_numpy(w)
    B = w.B
    nb, t = 1, 0.0
    while True:  # grow the sample until one pass takes about a quarter of the budget
        sub = {k: (v[:nb] if isinstance(v, np.ndarray) else v) for k, v in inputs.items()}
        t0 = time.perf_counter()
        oracle.spec_verify(**sub, n_threads=threads)
        t = time.perf_counter() - t0
        if nb == B or t >= budget_s / 4:
            break
        nb = min(B, nb * 4)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.spec_verify(**sub, n_threads=threads)
        reps += 1
        if time.perf_counter() - t0 >= budget_s or reps >= 200:
            break
    sec = (time.perf_counter() - t0) / reps
    pos = int(np.clip(sub["num_draft"], 0, None).sum())
    return pos / sec, f"{nb} of {B} requests ({pos} positions) x {reps}, {sec * 1e3:.2f} ms each"


def measure_config(w, dev, offset, steps, stream, flush, peak):
    """Cold- and hot-L2 time per call of one workload, with its byte figures."""
    from speculative_decoding_verification_51_gb300 import workloads as W
    c = Caller(w, dev, offset)
    for i in range(3):
        flush(i)
        c.seed_buf.fill_(1500 + i)
        c.graph.replay()
    torch.cuda.synchronize()
    cold, nacc_log = time_replays(c, steps, stream, flush)
    hot, _ = time_replays(c, steps, stream, None, seed0=2000)
    ms_cold, ms_hot = statistics.mean(cold), statistics.mean(hot)
    by = call_bytes(w, nacc_log)
    pos = W.positions(w.num_draft)
    valid = nacc_log >= 0
    acc = float((nacc_log.clamp(min=0)).sum()) / max(1, pos * nacc_log.shape[0])
    path = c.binding.verify_path(w.B, w.K, w.V, w.target_logits.dtype, dev)
    out = {"B": w.B, "K": w.K, "V": w.V, "positions_per_call": pos,
           "verifier": "request by request" if path else "all rows",
           "ms_per_call_cold_l2": round(ms_cold, 5), "ms_per_call_hot_l2": round(ms_hot, 5),
           "positions_per_s": round(pos / (ms_cold * 1e-3), 1),
           "accept_rate": round(acc, 4), "rows_all": by["rows_all"],
           "rows_read": round(by["rows_read"], 1), "residual_rows": round(by["residual_rows"], 1)}
    for k in ("algorithmic", "literal", "read"):
        gbs = by[k] / (ms_cold * 1e-3) / 1e9
        out[f"{k}_bytes"] = int(by[k])
        out[f"{k}_gbs"] = round(gbs, 1)
        out[f"{k}_frac"] = round(gbs / peak, 4)
    out["requests_all_valid"] = bool(valid.all())
    del c
    return out


def run_chain(args, rank, world, local):
    from speculative_decoding_verification_51_gb300 import binding
    from speculative_decoding_verification_51_gb300 import build as _build
    from speculative_decoding_verification_51_gb300 import sharding
    from speculative_decoding_verification_51_gb300 import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.build()
    binding.lib()
    peak, peak_kind, _ = measured_peak()
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)

    w = W.make_workload(args.config, device=dev)
    if args.batch:
        w = w.leading(args.batch)
    B, K, V = w.B, w.K, w.V
    offset = sharding.weak_offset(rank, B)  # each rank holds its own requests
    pos = W.positions(w.num_draft)
    c = Caller(w, dev, offset)
    for i in range(args.warmup):
        flush(i)
        c.direct(1000 + i)
    for i in range(args.warmup):
        flush(i)
        c.seed_buf.fill_(1500 + i)
        c.graph.replay()
    torch.cuda.synchronize()

    # ---- timed region: K steps, device time per step, L2 flushed before each
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        step_ms, nacc_log = time_replays(c, args.steps, stream, flush)
    if world > 1:
        torch.distributed.barrier()
    ms = sharding.max_over_ranks(sum(step_ms) / len(step_ms), device=dev)
    clocks = clk.summary()

    # the same call launched directly (no graph), and the all-rows verifier
    n_aux = min(args.steps, 50)
    devs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n_aux)]
    for i in range(n_aux):
        flush(i + 5)
        devs[i][0].record(stream)
        c.direct(2500 + i)
        devs[i][1].record(stream)
    torch.cuda.synchronize()
    ms_direct = statistics.mean(a.elapsed_time(b) for a, b in devs)
    forced = {}
    for name in ("all_rows", "by_request"):  # each verifier forced, at this workload
        ca = Caller(w, dev, offset, **{name: True})
        for i in range(3):
            flush(i)
            ca.graph.replay()
        torch.cuda.synchronize()
        forced[name] = statistics.mean(time_replays(ca, n_aux, stream, flush)[0])
        del ca
    path = binding.verify_path(B, K, V, w.target_logits.dtype, dev)
    kernels = binding.KERNELS if path else binding.KERNELS_ALL_ROWS

    # ---- per-kernel durations (marks between the kernels of the call)
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(binding.N_MARKS)]
             for _ in range(n_aux)]
    for m in marks:
        for e in m:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(n_aux):
        flush(i + 3)
        binding.spec_verify_profiled(w.target_logits, w.draft_probs, w.draft_ids, w.num_draft,
                                     w.temperature, 3000 + i, c.out_ids, c.out_nacc, c.ws,
                                     marks[i], by_request=bool(path), all_rows=not path)
    torch.cuda.synchronize()
    kern_ms = [statistics.mean(m[k].elapsed_time(m[k + 1]) for m in marks)
               for k in range(len(kernels))]

    # ---- bytes and the roofline of the dominant kernel: k_verify (the whole
    # verification) when the call runs request by request, else k_row_stats
    by = call_bytes(w, nacc_log)
    t_kern = kern_ms[1]
    wname = workload_name(args.config, args.batch)
    if path:
        kb = by["read"]
        kdef = ("rows 0..a_b of every request + the q row of each residual draw + gathers, "
                "ids, counts and outputs")
    else:
        kb = by["rows_all"] * V * w.target_logits.element_size()
        kdef = "every valid logits row 0..n_b once"
    ach = kb / (t_kern * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4),
                "traffic": profiled_traffic(wname, kernels[1]),
                "kernel": kernels[1], "kernel_ms": round(t_kern, 5),
                "algorithmic_bytes_per_launch": int(kb), "bytes_definition": kdef,
                "peak_kind": peak_kind}
    gate_gbs = by["algorithmic"] / (ms * 1e-3) / 1e9
    literal_gbs = by["literal"] / (ms * 1e-3) / 1e9

    # ---- end to end through host buffers (spec_verify_host)
    e2e = None
    if not args.no_e2e:
        e2e = e2e_host(w, dev, stream, args, world, pos)

    # ---- every workload: per_config (rank 0 only)
    per_config = None
    if rank == 0 and not args.no_per_config:
        per_config = {}
        n_pc = max(3, min(args.steps, 30))
        for cid in (1, 2, 3, 4, 5):
            wc = w if (cid == args.config and not args.batch) else W.make_workload(cid, device=dev)
            ent = measure_config(wc, dev, 0, n_pc, stream, flush, peak)
            if not args.no_cpu:
                for thr, key in ((1, "oracle_1t"), (0, "oracle_all_cores")):
                    import oracle
                    t_used = 1 if thr == 1 else oracle.omp_threads()
                    rate, sample = oracle_rate(wc, thr, args.oracle_seconds)
                    ent[key] = {"positions_per_s": round(rate, 1), "threads": t_used,
                                "sample": sample}
            per_config[f"config{cid}"] = ent
            if cid == 5:
                for (_, bb) in SWEEP:
                    ws_ = wc.leading(bb)
                    per_config[f"config5_B{bb}"] = measure_config(ws_, dev, 0, n_pc, stream,
                                                                  flush, peak)
                    del ws_
            if wc is not w:
                del wc
            torch.cuda.empty_cache()

    cpu = None
    parity_line = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(w, args.cpu_seconds)
        parity_line = bench_parity(w, c)

    value = world * pos / (ms * 1e-3)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{wname}: {w.spec.description}", "B": B, "K": K, "V": V,
                   "logits_dtype": str(w.target_logits.dtype).replace("torch.", ""),
                   "positions_per_step": pos, "rows_per_step": W.valid_rows(w.num_draft),
                   "l2": "flushed before every timed call: 256 MiB write, then 256 MiB read "
                         "(L2 left full of clean unrelated lines)",
                   "launch": "one spec_verify call captured in a CUDA graph (seed read from "
                             "device memory, written before each replay); ms_per_step_direct: "
                             "the same call launched directly",
                   "verifier": ("request by request (k_prep + k_verify)" if path else
                                "all rows (k_plan, k_row_stats, k_accept_all, k_sample, "
                                "k_emit)")},
        "ms_per_step_direct": round(ms_direct, 5),
        "ms_per_step_all_rows": round(forced["all_rows"], 5),
        "ms_per_step_by_request": round(forced["by_request"], 5),
        "hbm_gbs_step": round(gate_gbs, 1), "hbm_frac_step": round(gate_gbs / peak, 4),
        "hbm_step_bytes": int(by["algorithmic"]),
        "literal_bytes": {"bytes": int(by["literal"]), "gbs": round(literal_gbs, 1),
                          "frac": round(literal_gbs / peak, 4),
                          "definition": "logits rows 0..n_b + draft probability rows "
                                        "0..n_b-1, each read once"},
        "bytes_read_per_step": int(by["read"]),
        "kernels_ms": {n: round(t, 5) for n, t in zip(kernels, kern_ms)},
        "accept_rate": float(nacc_log.clamp(min=0).sum()) / max(1, pos * nacc_log.shape[0]),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "parity": parity_line,
        "per_config": per_config,
        "gpu_launches": len(kernels) * args.steps, "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def bench_parity(w, c):
    """Outputs of one GPU call against the oracle on the same inputs and seed:
    requests whose outputs are identical, and the differing ones classified
    by the parity tests' rule (tests/parity.py): excused near-ties (against
    the bound of 1e-4 of the rows) or failures."""
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import parity
    from speculative_decoding_verification_51_gb300 import binding
    from speculative_decoding_verification_51_gb300 import workloads as W
    seed = 4242
    ids, nacc, rows, _ = binding.spec_verify(w.target_logits, w.draft_probs, w.draft_ids,
                                             w.num_draft, w.temperature, seed, workspace=c.ws,
                                             debug=True)
    torch.cuda.synchronize()
    inputs = W.to_numpy(w)
    inputs["seed"] = seed
    ref = oracle.spec_verify(**inputs)
    ids, nacc, rows = ids.cpu().numpy(), nacc.cpu().numpy(), rows.cpu().numpy()
    same = (ids == ref["out_ids"]).all(1) & (nacc == ref["out_num_accepted"])
    rep = parity.compare(inputs, ids, nacc, rows, ref)
    return {"seed": seed, "requests": int(w.B), "identical": int(same.sum()),
            "differing": int((~same).sum()), "rows": int(rep.rows),
            "excused_accept": int(rep.excused_accept), "excused_cdf": int(rep.excused_cdf),
            "failures": len(rep.failures), "max_p_rel": float(rep.max_p_rel),
            "excused_within_1e-4_of_rows": bool(rep.excused < 1e-4 * rep.rows)}


def e2e_host(w, dev, stream, args, world, pos):
    """The same metric through spec_verify_host: inputs in pinned host memory,
    outputs copied back, all inside the timed region."""
    from speculative_decoding_verification_51_gb300 import binding
    B, K, V = w.B, w.K, w.V
    h = {k: getattr(w, k).cpu().pin_memory() for k in
         ("target_logits", "draft_probs", "draft_ids", "num_draft", "temperature")}
    h_out = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
    h_nacc = torch.empty((B,), dtype=torch.int32).pin_memory()
    d_l = torch.empty_like(w.target_logits)
    d_p = torch.empty_like(w.draft_probs)
    small = torch.empty(binding.host_small_bytes(B, K), dtype=torch.uint8, device=dev)
    ws = binding.new_workspace(B, K, V, dev)
    e2e_steps = max(3, min(args.steps, 10))

    def host_step(seed):
        binding.spec_verify_host(h["target_logits"], h["draft_probs"], h["draft_ids"],
                                 h["num_draft"], h["temperature"], seed, h_out, h_nacc, d_l,
                                 d_p, small, ws)

    for i in range(2):
        host_step(4000 + i)
    torch.cuda.synchronize()
    a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_ev.record(stream)
    for i in range(e2e_steps):
        host_step(5000 + i)
    b_ev.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a_ev.elapsed_time(b_ev) / e2e_steps
    # Pinned (mapped) host buffers take the rows-only path of
    # spec_verify_host: the logits rows 0..n_b, q_j(x_j) of every draft, and
    # the q row of each residual draw cross the link (the residual count of
    # each timed seed is taken from an untimed device call).
    n_cpu = h["num_draft"].long()
    valid = (n_cpu >= 0) & (n_cpu <= K)
    rows = torch.where(valid, n_cpu + 1, torch.ones_like(n_cpu))
    esz = h["target_logits"].element_size()
    h2d = int(rows.sum()) * V * esz
    h2d += sum(t.numel() * t.element_size()
               for t in (h["draft_ids"], h["num_draft"], h["temperature"]))
    h2d += int(torch.where(valid, n_cpu, torch.zeros_like(n_cpu)).sum()) * 4
    samp = (h["temperature"] > 0) & valid
    n_res = 0
    for i in range(e2e_steps):
        _, nacc_i = binding.spec_verify(w.target_logits, w.draft_probs, w.draft_ids,
                                        w.num_draft, w.temperature, 5000 + i)
        n_res += int(((nacc_i.cpu().long() < n_cpu) & samp & (nacc_i.cpu() >= 0)).sum())
    h2d += int(round(n_res / e2e_steps)) * V * 4
    d2h = h_out.numel() * 4 + h_nacc.numel() * 4
    return {"value": world * pos / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
            "path": "spec_verify_host (all-rows verifier over the copied rows)"}


if __name__ == "__main__":
    main()
