#!/usr/bin/env python3
"""Benchmark of MLA tree-verify attention on GB300 (one JSON line on stdout).

A step is one verify-attention call (partial kernel + split-K combine) over the
capture-safe stress workload (16 requests x 131,072-token prefix x 64-node
tree on a 2.2M-slot pool), captured once into a CUDA graph and replayed every
step, unless --workload says otherwise (the other workloads are timed as
direct calls).  Timing: CUDA events on the launching stream around each step,
L2 flushed (256 MiB write) between steps outside the events, W untimed
warm-up steps, K timed steps bracketed by barrier + synchronize.  ``value`` is
microseconds per call of the whole batch.  The roofline block times the
dominant kernel (the split-K partial kernel) alone, launched through
mla_tree_verify_run_steps with CUDA events on its stream.  With N GPUs (torchrun)
the batch's requests are partitioned over the ranks (balanced on
(p_r + n_r) * n_r; requests are independent, so no collective touches the data
path) and ``value`` is the slowest rank's time per call of the whole batch.

--impl reference times the CPU oracle (the only other implementation of this
path) on the host cores on a bounded row sample of the same workload and
extrapolates to microseconds per call.

--op mask / --op accept / --op defrag time the steps around verify attention
instead (the custom_mask build from parent arrays, the greedy acceptance walk,
the copy of each prefix into one contiguous run of slots) on the named
workload; --op shared times requests sharing one prefix, per request and
grouped into one; the default, --op verify, is the attention.
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_mla_speculative_tree_gb300 import binding  # noqa: E402
from paged_mla_speculative_tree_gb300 import partition as PT  # noqa: E402
from paged_mla_speculative_tree_gb300 import workloads as W  # noqa: E402

METRIC = "verify-attn µs/call, effective HBM GB/s, % of roofline (1×GB300)"
UNIT = "us/call"
DEFAULT_WORKLOAD = "stress"
GRAPH_WORKLOADS = {"stress"}  # timed as replays of the captured call


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def max_over_ranks(ms, ws, dev=None):
    """The slowest rank's time: the ranks run their shares of the batch concurrently."""
    if ws <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """SM clock and clock-event reasons sampled during the timed region through
    NVML (ctypes; read-only queries): a background thread every ~0.5 ms, plus
    synchronous samples the timed loop takes between launches (``sample()``),
    so that even a region of a few milliseconds is sampled under load."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index):
        self.cuda_index = cuda_index
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self.err = None
        self._stop = None
        self._thread = None
        self.nvml = None
        self.handle = None
        try:
            import ctypes
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            h = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(cuda_index)
            bus = getattr(props, "pci_bus_id", None)
            ok = False
            if bus is not None:
                busid = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), bus,
                                              getattr(props, "pci_device_id", 0))
                ok = lib.nvmlDeviceGetHandleByPciBusId_v2(busid.encode(), ctypes.byref(h)) == 0
            if not ok and lib.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(h)) != 0:
                raise RuntimeError("no NVML handle")
            self.nvml, self.handle = lib, h
            m = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(m)) == 0:
                self.max_mhz = float(m.value)
            self._reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception as e:  # pragma: no cover - depends on the box
            self.err = str(e)

    def sample(self):
        """One synchronous clock + reasons sample (no-op without NVML)."""
        if self.nvml is None:
            return
        import ctypes
        mhz = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz)) == 0:
            self.samples.append(float(mhz.value))
        if self._reason_fn(self.handle, ctypes.byref(rs)) == 0:
            self.reasons |= int(rs.value)

    def _poll(self):
        while not self._stop.is_set():
            self.sample()
            time.sleep(0.0005)

    def __enter__(self):
        if self.nvml is not None:
            import threading
            self._stop = threading.Event()
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=2)

    def summary(self):
        if self.nvml is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [f"nvml unavailable: {self.err}"]}
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"]}
        names = sorted(n for bit, n in self.REASONS.items() if self.reasons & bit)
        return {"sm_mhz": float(np.median(self.samples)), "sm_max_mhz": self.max_mhz,
                "samples": len(self.samples), "reasons": names, "source": "nvml"}


def make_workload(name):
    if name not in W.WORKLOADS:
        raise SystemExit(f"unknown workload {name}; choose from {sorted(W.WORKLOADS)}")
    return W.WORKLOADS[name]()


def device_inputs(wl, dev):
    return dict(q=wl.q.to(dev), kv_pool=wl.kv_pool.to(dev), kv_indices=wl.kv_indices.to(dev),
                kv_indptr=wl.kv_indptr.to(dev), out_cache_loc=wl.out_cache_loc.to(dev),
                qo_indptr=wl.qo_indptr.to(dev), custom_mask=wl.custom_mask.to(dev),
                mask_indptr=wl.mask_indptr.to(dev))


STEP_INPUTS = ("q", "kv_indices", "kv_indptr", "out_cache_loc", "qo_indptr", "custom_mask", "mask_indptr")


def cpu_oracle_timing(wl, target_s=15.0, seed=0):
    """Times the oracle on a bounded row sample; returns (us per full call, cores, sample text)."""
    import oracle
    cores = oracle.default_threads()
    H = wl.num_heads
    total_rows = wl.total_q * H
    rng = np.random.default_rng(seed)
    # calibrate on a handful of rows, then size the sample for ~target_s
    n = min(total_rows, max(cores, 16))
    rows = np.sort(rng.choice(total_rows, size=n, replace=False))
    t0 = time.perf_counter()
    oracle.mla_tree_verify(wl, rows=rows, num_threads=cores)
    dt = time.perf_counter() - t0
    per_row = dt / n
    n2 = int(min(total_rows, max(n, target_s / max(per_row, 1e-9))))
    if n2 > n:
        rows = np.sort(rng.choice(total_rows, size=n2, replace=False))
        t0 = time.perf_counter()
        oracle.mla_tree_verify(wl, rows=rows, num_threads=cores)
        dt = time.perf_counter() - t0
        n = n2
    us_per_call = dt / n * total_rows * 1e6
    return us_per_call, cores, f"{n} of {total_rows} (token, head) rows, seeded uniform; {dt:.1f} s"


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    wl = make_workload(args.workload)
    import oracle
    cores = oracle.default_threads()
    H = wl.num_heads
    total_rows = wl.total_q * H
    rng = np.random.default_rng(123)
    # size each step's sample so the whole run stays within a few minutes
    probe = np.sort(rng.choice(total_rows, size=min(total_rows, max(cores, 16)), replace=False))
    t0 = time.perf_counter()
    oracle.mla_tree_verify(wl, rows=probe, num_threads=cores)
    per_row = (time.perf_counter() - t0) / probe.size
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(min(total_rows, max(probe.size, budget / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        oracle.mla_tree_verify(wl, rows=np.sort(rng.choice(total_rows, size=n, replace=False)), num_threads=cores)
    times = []
    for _ in range(args.steps):
        rows = np.sort(rng.choice(total_rows, size=n, replace=False))
        t0 = time.perf_counter()
        oracle.mla_tree_verify(wl, rows=rows, num_threads=cores)
        times.append((time.perf_counter() - t0) / n * total_rows * 1e6)
    value = float(np.mean(times))
    sample = f"{n} of {total_rows} (token, head) rows per step, seeded uniform, extrapolated to the full call"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": value / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "bs": wl.bs, "prefix": wl.prefix_lens[0] if wl.bs else 0,
                       "tree": wl.tree_sizes[0] if wl.bs else 0},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    full = make_workload(args.workload)
    if ws > 1:
        # requests are independent: each rank runs its share of the batch
        # (balanced on (p_r + n_r) * n_r), no exchange on the data path
        parts = PT.partition_requests(full.prefix_lens, full.tree_sizes, ws)
        wl = W.sub_workload(full, parts[rank])
    else:
        parts = [list(range(full.bs))]
        wl = full
    d = device_inputs(wl, dev)
    T = max(wl.total_q, 1)
    out = torch.empty((T, 64, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, 64), dtype=torch.float32, device=dev)
    # For the end-to-end steps, the per-step inputs (q and the metadata) live in
    # one packed device buffer and the outputs in another, so that a step from
    # host memory is one copy in and one copy out (the pool stays in HBM).
    in_dev, in_views, in_host, in_host_views, h2d = packed_buffers({k: wl_tensor(wl, k) for k in STEP_INPUTS}, dev)
    for k in STEP_INPUTS:
        in_host_views[k].copy_(wl_tensor(wl, k))
    d_e2e = dict(d, **in_views)
    out_dev, out_views, out_host, _, d2h = packed_buffers(
        {"out": torch.empty((T, 64, 512), dtype=torch.bfloat16),
         "lse": torch.empty((T, 64), dtype=torch.float32)}, dev)
    flags = binding.FLAG_SIMT_FLOOR if args.simt else 0
    # the batch's request lengths are known on the host when it is planned:
    # the split count comes from them (an explicit --nsplit overrides)
    m = binding.MlaTreeVerify(wl.bs, wl.max_q_per_req, T, wl.max_prefix, device=local,
                              mask_layout=wl.mask_layout, flags=flags, nsplit=args.nsplit,
                              lengths=(wl.prefix_lens, wl.tree_sizes))
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def call(steps=None):
        binding.run(m.plan, d["q"], d["kv_pool"], d["kv_indices"], d["kv_indptr"], d["out_cache_loc"],
                    d["qo_indptr"], d["custom_mask"], d["mask_indptr"], wl.scale, out, lse, m.workspace,
                    steps=steps)

    def call_e2e():
        m(d_e2e["q"], d_e2e["kv_pool"], d_e2e["kv_indices"], d_e2e["kv_indptr"], d_e2e["out_cache_loc"],
          d_e2e["qo_indptr"], d_e2e["custom_mask"], d_e2e["mask_indptr"], wl.scale, out_views["out"],
          out_views["lse"])

    use_graph = args.graph if args.graph is not None else (args.workload in GRAPH_WORKLOADS)
    step = call
    if use_graph:
        # captured once with static buffers, replayed every step (the capture-safe use of the call)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            call()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()
        torch.cuda.synchronize()
        step = graph.replay

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    assert m.device_error() == 0, "device error word set during warm-up"

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for k in range(args.steps):
            flush.fill_(k & 0xff)
            starts[k].record(stream)
            step()
            ends[k].record(stream)
            if k % 2 == 1:
                clk.sample()  # host-side, between launches: the GPU is still busy with the queued steps
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        wall = time.perf_counter() - t_wall
    per_call_ms = [s_.elapsed_time(e) for s_, e in zip(starts, ends)]
    ms = max_over_ranks(float(np.mean(per_call_ms)), ws, dev)
    clocks = clk.summary()
    launches_per_call = (1 + (1 if m.plan.nsplit > 1 else 0)) if wl.bs else 0

    # the dominant kernel alone: the partial (split-K) launch, CUDA events on its stream
    for _ in range(max(1, args.warmup // 2)):
        flush.fill_(1)
        call(binding.STEP_PARTIAL)
    p_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    p_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for k in range(args.steps):
        flush.fill_(k & 0xff)
        p_s[k].record(stream)
        call(binding.STEP_PARTIAL)
        p_e[k].record(stream)
    torch.cuda.synchronize()
    partial_ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in zip(p_s, p_e)])), ws, dev)

    # end to end through the public API with host buffers (pinned), copies inside the timed region
    for _ in range(max(1, args.warmup)):
        e2e_step(in_host, in_dev, call_e2e, out_dev, out_host)
    torch.cuda.synchronize()
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for k in range(args.steps):
        flush.fill_(k & 0xff)
        e_s[k].record(stream)
        e2e_step(in_host, in_dev, call_e2e, out_dev, out_host)
        e_e[k].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(float(np.mean([s_.elapsed_time(e) for s_, e in zip(e_s, e_e)])), ws, dev)
    assert m.device_error() == 0, "device error word set during the timed runs"

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return 0
    peaks = load_peaks()
    # whole-job figures: the full batch (all ranks' requests) per step
    flops = full.algorithmic_flops()
    nbytes = full.algorithmic_bytes()
    achieved_tf = flops / (ms * 1e-3) / 1e12
    achieved_gbs = nbytes / (ms * 1e-3) / 1e9
    peak_tf = peaks["bf16_tflops"]
    roof_ms = max(nbytes / (peaks["hbm_gbs"] * 1e9), flops / (peak_tf * 1e12)) * 1e3
    bound = "tensor" if flops / (peak_tf * 1e12) >= nbytes / (peaks["hbm_gbs"] * 1e9) else "hbm"
    # the dominant kernel on this rank's share (rank 0's launch)
    k_flops, k_bytes = wl.algorithmic_flops(), wl.algorithmic_bytes()
    k_tf = k_flops / (partial_ms * 1e-3) / 1e12 if partial_ms > 0 else 0.0
    k_gbs = k_bytes / (partial_ms * 1e-3) / 1e9 if partial_ms > 0 else 0.0
    traffic = load_traffic(wl.name, m.plan)
    kernel_name = "partial_simt_kernel" if args.simt else "partial_tc_kernel"
    if bound == "tensor":
        roof = {"bound": "tensor", "achieved": k_tf, "peak": peak_tf, "unit": "TFLOP/s", "frac": k_tf / peak_tf,
                "traffic": traffic}
    else:
        roof = {"bound": "hbm", "achieved": k_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": k_gbs / peaks["hbm_gbs"], "traffic": traffic}
    roof.update({
        "kernel": kernel_name, "kernel_us": partial_ms * 1e3,
        "peak_source": peaks["source"] + (" burst" if bound == "tensor" else ""),
        "frac_of_sustained": k_tf / peaks["bf16_tflops_sustained"] if bound == "tensor" else None,
        "timed": "the partial kernel alone (run_steps PARTIAL), CUDA events on its launch stream, "
                 f"{args.steps} launches, L2 flushed between",
        "algorithmic_flops_per_launch": k_flops, "algorithmic_bytes_per_launch": k_bytes,
        "whole_call": {"achieved_tflops": achieved_tf, "frac": achieved_tf / peak_tf if bound == "tensor" else
                       achieved_gbs / peaks["hbm_gbs"], "roofline_us": roof_ms * 1e3,
                       "frac_of_roofline": roof_ms / ms, "effective_hbm_gbs": achieved_gbs}})
    line = {
        "metric": METRIC, "value": ms * 1e3, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
        "scaling": "strong" if ws > 1 else "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": full.name, "bs": full.bs, "prefix": full.prefix_lens, "tree": full.tree_sizes,
                   "num_slots": full.num_slots, "heads": 64, "d_qk": 576, "d_v": 512,
                   "kernel": "simt-floor" if args.simt else "tcgen05", "nsplit": int(m.plan.nsplit),
                   "nsplit_from": "--nsplit" if args.nsplit else "the batch's request lengths",
                   "split_keys": int(m.plan.split_keys),
                   "parallelism": f"requests partitioned over {ws} GPUs" if ws > 1 else "1 GPU",
                   "requests_per_rank": [len(p_) for p_ in parts],
                   "timing": "CUDA-graph replay of the captured call" if use_graph else "direct calls",
                   "l2": "flushed between calls (256 MiB write outside the timed events); the inputs "
                         + ("also exceed L2" if full.algorithmic_bytes() > 129e6 else "fit in L2")},
        "effective_hbm_gbs": achieved_gbs, "achieved_tflops": achieved_tf,
        "roofline": roof, "clocks": clocks, "gpu_launches": launches_per_call * args.steps,
        "e2e": {"value": e2e_ms * 1e3, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "wall_s_timed_region": wall,
    }
    if not args.no_cpu_baseline and ws == 1:
        us, cores, sample = cpu_oracle_timing(full, target_s=args.cpu_seconds)
        line["cpu_baseline"] = {"value": us, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def tree_shapes(name):
    """(prefix lengths, parent arrays) of a named workload; the Stress trees are
    drawn directly (seed 5005) so that its 2.5 GB pool is not generated."""
    if name == "stress":
        g = torch.Generator().manual_seed(5005)
        return [131072] * 16, [W.random_parents(64, g) for _ in range(16)], "stress_bs16_p131072_n64"
    wl = make_workload(name)
    return wl.prefix_lens, wl.parents, wl.name


def run_tree_op(args):
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.op == "defrag":
        return run_defrag(args, dev, local)
    if args.op == "shared":
        return run_shared(args, dev, local)
    prefix, trees, wname = tree_shapes(args.workload)
    bs, sizes = len(trees), [len(t) for t in trees]
    max_q = max(sizes + [0])
    total = sum(sizes)
    g = torch.Generator().manual_seed(77)
    host = {
        "parents": torch.tensor([p for t in trees for p in t], dtype=torch.int32),
        "qo_indptr": torch.tensor([0] + list(np.cumsum(sizes)), dtype=torch.int64),
        "kv_indptr": torch.tensor([0] + list(np.cumsum(prefix)), dtype=torch.int32),
        "draft": torch.randint(0, 4, (total,), generator=g, dtype=torch.int32),
        "target": torch.randint(0, 4, (total,), generator=g, dtype=torch.int32),
        "root": torch.randint(0, 4, (bs,), generator=g, dtype=torch.int32),
        "slots": torch.randperm(4 * total + 1, generator=g)[:total].to(torch.int64),
    }
    d = {k: v.to(dev) for k, v in host.items()}
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    if args.op == "mask":
        mask_bytes = sum(n * (p + n) for p, n in zip(prefix, sizes))
        outs = {"mask": torch.empty(mask_bytes, dtype=torch.uint8, device=dev),
                "indptr": torch.empty(bs + 1, dtype=torch.int64, device=dev)}
        in_keys = ("parents", "qo_indptr", "kv_indptr")

        def call():
            binding.tree_mask_build(d["parents"], d["qo_indptr"], d["kv_indptr"], bs, max_q, binding.MASK_FULL_ROW,
                                    outs["mask"], outs["indptr"], err)
    else:
        outs = {"len": torch.empty(bs, dtype=torch.int32, device=dev),
                "nodes": torch.empty((bs, max_q), dtype=torch.int32, device=dev),
                "aslots": torch.empty((bs, max_q), dtype=torch.int64, device=dev),
                "bonus": torch.empty(bs, dtype=torch.int32, device=dev)}
        in_keys = ("parents", "qo_indptr", "draft", "target", "root", "slots")

        def call():
            binding.tree_accept(d["parents"], d["draft"], d["target"], d["root"], d["slots"], d["qo_indptr"], bs,
                                max_q, outs["len"], outs["nodes"], outs["aslots"], outs["bonus"], err)
    in_bytes = sum(d[k].numel() * d[k].element_size() for k in in_keys)
    out_bytes = sum(t.numel() * t.element_size() for t in outs.values())
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        flush.fill_(1)
        call()
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "device error word set during warm-up"
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for k in range(args.steps):
            flush.fill_(k & 0xff)
            starts[k].record(stream)
            call()
            ends[k].record(stream)
            if k % 2 == 1:
                clk.sample()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t_wall
    ms = float(np.mean([s_.elapsed_time(e) for s_, e in zip(starts, ends)]))
    # end to end: inputs from pinned host memory, outputs back, copies timed
    hpin = {k: host[k].pin_memory() for k in in_keys}
    hout = {k: torch.empty_like(v, device="cpu").pin_memory() for k, v in outs.items()}
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for k in range(args.steps + 1):
        if k:
            e_s[k - 1].record(stream)
        for kk in in_keys:
            d[kk].copy_(hpin[kk], non_blocking=True)
        call()
        for kk, t in outs.items():
            hout[kk].copy_(t, non_blocking=True)
        if k:
            e_e[k - 1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = float(np.mean([s_.elapsed_time(e) for s_, e in zip(e_s, e_e)]))
    # the oracle on the host, one whole call
    from oracle import tree_ops as TO
    t0 = time.perf_counter()
    if args.op == "mask":
        TO.tree_mask(trees, prefix, TO.MASK_FULL_ROW)
    else:
        hq = host["qo_indptr"].tolist()
        for r in range(bs):
            sl = slice(hq[r], hq[r + 1])
            TO.tree_accept(trees[r], host["draft"][sl].tolist(), host["target"][sl].tolist(), int(host["root"][r]),
                           host["slots"][sl].tolist())
    cpu_us = (time.perf_counter() - t0) * 1e6
    peaks = load_peaks()
    nbytes = in_bytes + out_bytes
    gbs = nbytes / (ms * 1e-3) / 1e9
    line = {
        "metric": f"tree-{args.op} µs/call (1×GB300)", "value": ms * 1e3, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "int32/u8", "data": "synthetic",
        "config": {"workload": wname, "op": args.op, "bs": bs, "prefix": prefix, "tree": sizes,
                   "l2": "flushed between calls (256 MiB write outside the timed events)"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                     "peak_source": peaks["source"], "algorithmic_bytes": nbytes},
        "clocks": clk.summary(), "gpu_launches": args.steps,
        "e2e": {"value": e2e_ms * 1e3, "unit": UNIT, "h2d_bytes_per_step": in_bytes,
                "d2h_bytes_per_step": out_bytes},
        "cpu_baseline": {"value": cpu_us, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "one whole call, single-threaded Python"},
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_shared(args, dev, local):
    """Requests that share one prefix: verify per request, against the grouped
    path (merge into one request per group + mask build + verify), both timed
    as whole calls."""
    wl = make_workload(args.workload if args.workload.startswith("shared") else "shared_tree3")
    d = device_inputs(wl, dev)
    G = 1
    n_m = wl.total_q
    par = torch.tensor([p for t in wl.parents for p in t], dtype=torch.int32, device=dev)
    gi = torch.tensor([0, wl.bs], dtype=torch.int32, device=dev)
    kvp = torch.empty(G + 1, dtype=torch.int32, device=dev)
    idx = torch.empty(wl.prefix_lens[0], dtype=torch.int64, device=dev)
    qop = torch.empty(G + 1, dtype=torch.int64, device=dev)
    parout = torch.empty_like(par)
    mask = torch.empty(n_m * (wl.prefix_lens[0] + n_m), dtype=torch.uint8, device=dev)
    mip = torch.empty(G + 1, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty((wl.total_q, 64, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((wl.total_q, 64), dtype=torch.float32, device=dev)
    per_req = binding.MlaTreeVerify(wl.bs, wl.max_q_per_req, wl.total_q, wl.max_prefix, device=local)
    grouped = binding.MlaTreeVerify(G, n_m, wl.total_q, wl.max_prefix, device=local)

    def call_per_request():
        per_req(d["q"], d["kv_pool"], d["kv_indices"], d["kv_indptr"], d["out_cache_loc"], d["qo_indptr"],
                d["custom_mask"], d["mask_indptr"], wl.scale, out, lse)

    def call_grouped():
        binding.tree_group_prefix(gi, G, wl.max_prefix, d["kv_indices"], d["kv_indptr"], d["qo_indptr"], par,
                                  kvp, idx, qop, parout, err)
        binding.tree_mask_build(parout, qop, kvp, G, n_m, binding.MASK_FULL_ROW, mask, mip, err)
        grouped(d["q"], d["kv_pool"], idx, kvp, d["out_cache_loc"], qop, mask, mip, wl.scale, out, lse)

    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def time_it(fn, clk=None):
        for _ in range(args.warmup):
            flush.fill_(1)
            fn()
        torch.cuda.synchronize()
        st = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        en = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for k in range(args.steps):
            flush.fill_(k & 0xff)
            st[k].record(stream)
            fn()
            en[k].record(stream)
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in zip(st, en)]))

    ms_per = time_it(call_per_request)
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        ms = time_it(call_grouped)
        wall = time.perf_counter() - t_wall
    assert int(err.item()) == 0 and per_req.device_error() == 0 and grouped.device_error() == 0
    peaks = load_peaks()
    flops = wl.algorithmic_flops()
    tf = flops / (ms * 1e-3) / 1e12
    line = {
        "metric": "shared-prefix verify µs/call (1×GB300)", "value": ms * 1e3, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "op": "shared", "bs": wl.bs, "prefix": wl.prefix_lens[0],
                   "tree": wl.tree_sizes[0], "per_request_us": ms_per * 1e3,
                   "grouped_includes": "group + mask build + verify",
                   "l2": "flushed between calls (256 MiB write outside the timed events)"},
        "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": tf / peaks["bf16_tflops"], "traffic": None, "peak_source": peaks["source"] + " burst"},
        "clocks": clk.summary(), "gpu_launches": 4 * args.steps,
        "e2e": {"value": ms * 1e3, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0,
                "note": "inputs device-resident; see --op verify for the host-buffer path"},
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_defrag(args, dev, local):
    """Each request's prefix rows copied into one contiguous run of a second
    pool (run r starts where run r-1 ends) and its indices rewritten."""
    wl = make_workload(args.workload)
    src = wl.kv_pool.to(dev)
    dst = torch.zeros_like(src)
    idx = wl.kv_indices.to(dev)
    indptr = wl.kv_indptr.to(dev)
    base = torch.tensor([0] + list(np.cumsum(wl.prefix_lens))[:-1], dtype=torch.int64, device=dev)
    out_idx = torch.empty_like(idx)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def call():
        binding.kv_defrag(src, dst, idx, indptr, wl.bs, wl.max_prefix, base, out_idx, err)

    rows = int(wl.kv_indptr[-1])
    nbytes = rows * 1152 * 2 + rows * 8 * 2 + (wl.bs + 1) * 4 + wl.bs * 8
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        flush.fill_(1)
        call()
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "device error word set during warm-up"
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for k in range(args.steps):
            flush.fill_(k & 0xff)
            starts[k].record(stream)
            call()
            ends[k].record(stream)
            if k % 2 == 1:
                clk.sample()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t_wall
    ms = float(np.mean([s_.elapsed_time(e) for s_, e in zip(starts, ends)]))
    from oracle import tree_ops as TO
    sample = min(wl.bs, 2)
    t0 = time.perf_counter()
    src16 = wl.kv_pool.view(torch.int16).numpy()
    TO.kv_defrag(src16, src16, wl.kv_indices.numpy(), wl.kv_indptr.numpy()[:sample + 1], base.cpu().numpy()[:sample])
    cpu_s = time.perf_counter() - t0
    cpu_us = cpu_s * 1e6 * rows / max(1, int(wl.kv_indptr[sample]))
    peaks = load_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    line = {
        "metric": "kv-defrag µs/call (1×GB300)", "value": ms * 1e3, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (copy)", "data": "synthetic",
        "config": {"workload": wl.name, "op": "defrag", "bs": wl.bs, "rows": rows,
                   "l2": "flushed between calls (256 MiB write outside the timed events)"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None, "peak_source": peaks["source"],
                     "algorithmic_bytes": nbytes},
        "clocks": clk.summary(), "gpu_launches": args.steps,
        "e2e": {"value": ms * 1e3, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0,
                "note": "device-resident pools: the call moves KV inside HBM"},
        "cpu_baseline": {"value": cpu_us, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{sample} request(s) timed, scaled by rows ({cpu_s:.2f} s)"},
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)
    return 0


def wl_tensor(wl, k):
    return getattr(wl, k).contiguous()


def packed_buffers(tensors, dev):
    """One device byte buffer and one pinned host byte buffer holding every
    tensor of ``tensors`` at a 256-byte aligned offset; returns (device buffer,
    device views, host buffer, host views, total bytes)."""
    offs, total = {}, 0
    for k, t in tensors.items():
        offs[k] = total
        total = (total + t.numel() * t.element_size() + 255) // 256 * 256
    dbuf = torch.empty(max(total, 256), dtype=torch.uint8, device=dev)
    hbuf = torch.empty(max(total, 256), dtype=torch.uint8).pin_memory()
    dv, hv = {}, {}
    for k, t in tensors.items():
        nb = t.numel() * t.element_size()
        dv[k] = dbuf[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
        hv[k] = hbuf[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
    return dbuf, dv, hbuf, hv, total


def e2e_step(in_host, in_dev, call, out_dev, out_host):
    in_dev.copy_(in_host, non_blocking=True)
    call()
    out_host.copy_(out_dev, non_blocking=True)


def load_traffic(workload_name, plan):
    """DRAM bytes per launch of the partial kernel from the committed ncu
    summary (profiles/traffic.md), if it was measured on these kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    rev = kernel_revision()
    for line in open(path):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) == 3 and cells[0] == workload_name and cells[1] == rev:
            try:
                return int(cells[2])
            except ValueError:
                return None
    return None


def _code_only(text: str) -> str:
    """C/C++ source without comments and blank lines (string literals in
    these files hold no comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_revision():
    """Hash of the code the partial kernel is built from: its .cu and the
    headers it includes, comments and blank lines removed, plus the ABI
    header's #define lines (its constants); edits to comments or to host
    declarations leave it unchanged."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_mla_speculative_tree_gb300", "csrc")
    for f in ("partial_tc.cu", "tc_ptx.cuh", "mtv_internal.cuh"):
        h.update(_code_only(open(os.path.join(csrc, f)).read()).encode())
    hdr = _code_only(open(os.path.join(ROOT, "include", "mla_tree_verify.h")).read())
    h.update("\n".join(line for line in hdr.splitlines() if line.lstrip().startswith("#define")).encode())
    return h.hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--nsplit", type=int, default=0)
    ap.add_argument("--simt", action="store_true", help="time the SIMT correctness-floor kernel")
    ap.add_argument("--graph", dest="graph", action="store_true", default=None,
                    help="time replays of a captured CUDA graph (default for stress)")
    ap.add_argument("--no-graph", dest="graph", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--op", choices=["verify", "mask", "accept", "defrag", "shared"], default="verify",
                    help="verify attention (default) or one of the tree steps around it")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.op != "verify":
        return run_tree_op(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
