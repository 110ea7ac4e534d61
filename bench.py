"""Benchmark of the paged decode hot path on one GB300 (or N replicas).

One step = one pass of the whole hot path over one decode batch: slot mapping
of each sequence's new token, the slot-mapped KV write, and decode attention
through the block tables (split-K partitions plus the reduce). Inputs are
resident in HBM when the timed region starts; the pool (about 1.4 GB for the
default workload) is far larger than L2, so no flush is needed between steps.

value  = algorithmic bytes of a step x steps x ranks / max-over-ranks time, GB/s
e2e    = the same metric through the same calls with pinned host buffers:
         every step copies its inputs host -> device and reads the output back.
roofline = decode call only (partition kernel + reduce): algorithmic bytes per
         call / mean call time from CUDA events on the launching stream.

With --kv-dtype e4m3 the same workload shape runs on an FP8 (E4M3) pool: one
byte per cached element, q and the new K/V rows fp16/bf16, codes quantised by
the write and widened by decode.

--prefill NAME times pa_prefill alone (multi-token causal attention) on a named
workload instead: verify4_70b_bf16_b16 or verify4_long_bf16_b16 (speculative
verification, HBM-bound), chunk512_gqa_bf16_b16 or prompt2k_mha_fp16_b16
(tensor-bound). The call gets a workspace when the shape can use one
(--no-workspace withholds it).

--swap times pa_swap_blocks: a preempted batch's blocks (every layer, K and V)
out to a pinned host pool and back in, against a contiguous copy of the same
bytes by the copy engine as the link's reference rate.

--hash times pa_prefix_hash: SHA-256 chain keys of every full block of 4,096
prompts of 2,048 token ids (b = 16).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--kv-dtype e4m3]
                       [--impl reference] [--prefill NAME [--no-workspace]] [--swap] [--hash]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention achieved HBM GB/s (% of peak) and decode tokens/s"
SPEC_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.json")
KERNEL_SOURCES = ["pa_decode.cuh", "pa_decode_grouped.cuh", "pa_ptx.cuh", "pa_decode_reduce.cu",
                  "pa_decode_inst.cu"]


# ----------------------------------------------------------------------------- accounting


def step_tokens(w):
    """Indices of the rows a timed step writes: each sequence's newest token
    (config 1 writes its whole scenario, all 60 tokens)."""
    from workloads import decode_step_tokens
    if w.name.startswith("tiny"):
        return np.arange(len(w.positions))
    return decode_step_tokens(w)


def kv_elem(w):
    """Bytes per cached element: 1 for an E4M3 pool, else 2."""
    return 1 if w.kv_dtype == "e4m3" else 2


def load_workload(config, block_size=None, kv_dtype="native"):
    from workloads import make_config
    return make_config(config, block_size=block_size if config == 4 else None,
                       kv_dtype="e4m3" if kv_dtype == "e4m3" else None)


def decode_bytes(w, out_elem=4):
    """Algorithmic bytes of one decode call: every valid K and V row once, q,
    the output, the table entries the lengths cover, and the lengths."""
    L = w.seq_lens.astype(np.int64)
    kv = int(L.sum()) * w.num_kv_heads * w.head_dim * kv_elem(w) * 2
    q = w.num_seqs * w.num_q_heads * w.head_dim * 2
    out = w.num_seqs * w.num_q_heads * w.head_dim * out_elem
    tables = int((-(-L // w.block_size)).sum()) * 4
    return kv + q + out + tables + 4 * w.num_seqs


def unique_decode_bytes(w):
    """Like decode_bytes but counting shared prefix blocks once (config 5)."""
    if not w.shared_blocks:
        return decode_bytes(w)
    shared_tokens = len(w.shared_blocks) * w.block_size
    row = w.num_kv_heads * w.head_dim * kv_elem(w) * 2
    return decode_bytes(w) - (w.num_seqs - 1) * shared_tokens * row


def write_bytes(w, n_tokens):
    """Slot mapping (ids, positions, table entries in; slots out) and the KV write
    (key/value rows read once at 2 bytes an element, written once at the
    cache's element size)."""
    elems = w.num_kv_heads * w.head_dim
    return n_tokens * (4 + 4 + 4 + 8) + n_tokens * (8 + 2 * elems * 2 + 2 * elems * kv_elem(w))


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_hash():
    """Hash of what the decode kernels are built from: their sources and the
    DecodeArgs struct they take (other declarations in the shared internal
    header do not change them)."""
    csrc = os.path.join(ROOT, "paged_kv_cache_114_gb300", "csrc")
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    with open(os.path.join(csrc, "pa_internal.h")) as f:
        text = f.read()
    start = text.index("struct DecodeArgs")
    h.update(text[start:text.index("};", start)].encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload, partition):
    """DRAM bytes per decode call from the committed ncu summary, or None when
    the kernel sources changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_hash") != kernel_hash():
        return None
    entry = rec.get("workloads", {}).get(f"{workload}/p{partition}")
    return None if entry is None else int(entry["dram_bytes_per_call"])


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm


class Run:
    """One workload resident on the device, driven through pa.DecodeStep."""

    def __init__(self, w, dev, partition):
        import torch

        import paged_kv_cache_114_gb300 as pa
        self.w, self.dev, self.pa, self.torch = w, dev, pa, torch
        fp8 = w.kv_dtype == "e4m3"
        self.k = to_dev(w.k_cache, dev, None if fp8 else w.dtype)
        self.v = to_dev(w.v_cache, dev, None if fp8 else w.dtype)
        scales = {"k_scale": w.k_scale, "v_scale": w.v_scale} if fp8 else {}
        idx = step_tokens(w)
        # scenario rows written before timing (config 5's suffixes, after its copies)
        setup = np.setdiff1d(np.arange(len(w.positions)), idx)
        tables = to_dev(w.block_tables, dev)
        if len(w.copy_pairs):
            pa.copy_blocks([self.k], [self.v], to_dev(w.copy_pairs, dev))
        if len(setup):
            sl = pa.slot_mapping(tables, to_dev(w.seq_idx[setup], dev),
                                 to_dev(w.positions[setup], dev), w.block_size, w.num_blocks)
            pa.write_kv(to_dev(w.key[setup], dev, w.dtype), to_dev(w.value[setup], dev, w.dtype),
                        sl, self.k, self.v, **scales)
        self.n_tokens = len(idx)
        self.partition = partition
        self.step_obj = pa.DecodeStep(
            self.k, self.v, num_seqs=w.num_seqs, num_q_heads=w.num_q_heads,
            num_tokens=self.n_tokens, max_blocks_per_seq=w.max_blocks_per_seq,
            max_seq_len=w.max_seq_len, scale=w.scale, out_dtype=torch.float32,
            partition_tokens=partition,
            act_dtype=torch.float16 if w.dtype == "f16" else torch.bfloat16, **scales)
        host, _ = self.step_obj.host_buffers()
        fill = {"q": w.q, "key": w.key[idx], "value": w.value[idx], "seq_idx": w.seq_idx[idx],
                "positions": w.positions[idx], "block_tables": w.block_tables,
                "seq_lens": w.seq_lens}
        for name, arr in fill.items():
            t = host[name]
            src = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16 if arr.dtype == np.uint16
                                                                  else arr.dtype))
            t.view(src.dtype).copy_(src.view(t.shape))
        with torch.cuda.stream(self.step_obj.stream):
            self.step_obj.staging.copy_(self.step_obj._host_staging)
        # slot mapping + KV write + the decode's kernels (the reduce of fixed
        # split-K partitions, the merge of the grouped kernel's cut pieces)
        kname = pa.decode_kernel_name(w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                      w.max_seq_len, partition)
        self.launches_per_step = 2 + len(kname.split("+"))

    def step(self, ev=None):
        self.step_obj.run(decode_events=ev)


def to_dev(a, dev, dtype=None):
    """Host numpy array -> device tensor (fp16/bf16 bit patterns viewed as that dtype)."""
    import torch
    a = np.ascontiguousarray(a)
    if dtype is not None:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(
            torch.float16 if dtype == "f16" else torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return world, rank, local


def reduce_max(value, world, device=None):
    """Max of a float over ranks (identity on one rank)."""
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


def run_gpu(args):
    import torch

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import paged_kv_cache_114_gb300 as pa
    pa.lib()

    w = load_workload(args.config, args.block_size, args.kv_dtype)
    partition = args.partition if args.partition is not None else pa.default_partition(
        w.num_seqs, w.num_kv_heads, w.max_seq_len, w.block_size)
    run = Run(w, dev, partition)
    if pa.get_device_error(dev):
        raise RuntimeError("device error during setup")

    step_bytes = write_bytes(w, run.n_tokens) + decode_bytes(w)
    dec_bytes = decode_bytes(w)
    K, W = args.steps, args.warmup

    for _ in range(W):
        run.step()
    torch.cuda.synchronize()
    if pa.get_device_error(dev):
        raise RuntimeError("device error during warm-up")

    stream = run.step_obj.stream  # every timed launch goes to the step's stream
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        e0.record(stream)
        for i in range(K):
            run.step(evs[i])
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms_total = reduce_max(e0.elapsed_time(e1), world, dev)
    dec_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    err = pa.get_device_error(dev)
    if err:
        raise RuntimeError(f"device error word {err} after the timed region")

    ms_step = ms_total / K
    value = step_bytes * K * world / (ms_total / 1e3) / 1e9
    tok_s = w.num_seqs * K * world / (ms_total / 1e3)

    # ---- end to end: pinned host inputs in, output back to the host, every step
    e2e = run_e2e(run, K, W, world, dev, step_bytes)

    peak, peak_kind = measured_peaks()
    achieved = dec_bytes / (dec_ms / 1e3) / 1e9
    workload = f"{w.name}"
    traffic = recorded_traffic(workload, partition)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs copy rate)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "frac_of_8tbs_spec": round(achieved / SPEC_HBM_GBS, 4),
                "kernel": pa.decode_kernel_name(w.num_q_heads, w.num_kv_heads, w.head_dim,
                                                w.block_size, w.max_seq_len, partition),
                "algorithmic_bytes_per_call": dec_bytes, "mean_call_us": round(dec_ms * 1e3, 2)}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.kv_dtype or w.dtype, "data": "synthetic",
        "config": {
            "workload": workload,
            "shape": f"{w.num_seqs} seqs, {w.num_q_heads} q heads / {w.num_kv_heads} kv heads, "
                     f"head_dim {w.head_dim}, block {w.block_size}, seq_len {int(w.seq_lens.min())}.."
                     f"{int(w.seq_lens.max())} (mean {float(w.seq_lens.mean()):.0f})",
            "step": "pa_slot_mapping + pa_write_kv (one new token per sequence) + pa_decode",
            "kv_dtype": w.cache_dtype,
            "act_dtype": w.dtype,
            "partition_tokens": partition,
            "pool_bytes": int(w.k_cache.nbytes + w.v_cache.nbytes),
            "l2": "inputs larger than L2: the K/V pool far exceeds the 129 MB L2; no flush",
            "algorithmic_bytes_per_step": step_bytes,
            "parallelism": f"{world} independent replica(s), no collective",
        },
        "decode_tok_s": round(tok_s, 1),
        "decode_tok_s_note": "attention-only, one layer: sequences decoded per second",
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": run.launches_per_step * K,
        "clocks": clocks.summary(),
    }
    if w.shared_blocks:
        line["config"]["unique_decode_bytes"] = unique_decode_bytes(w)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_child(args.config, args.block_size, "cpu_baseline",
                                                  kv_dtype=args.kv_dtype)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(run, K, W, world, dev, step_bytes):
    """The same step end to end through the library's public calls, every step:
    pa.DecodeStep.run_from_host copies the pinned host staging buffer (all of
    the step's inputs) to the device, calls pa_slot_mapping, pa_write_kv and
    pa_decode through the C ABI (each call validates its arguments, encodes its
    TMA descriptors and launches), copies the output back and waits for it.
    That eager leg is the e2e value. The same sequence replayed from a CUDA
    graph captured once (as a serving loop with fixed shapes would run it) is
    reported beside it under "graph"."""
    import torch
    st = run.step_obj
    host, out_host = st.host_buffers()
    h2d = st.nbytes
    d2h = out_host.numel() * out_host.element_size()

    def timed():
        for _ in range(W):
            st.run_from_host()
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(K):
            st.run_from_host()
        t1 = time.perf_counter()
        barrier(world)
        return reduce_max(t1 - t0, world, dev)

    secs = timed()  # no graph captured yet: every call goes through the C ABI
    st.capture_graph()
    secs_graph = timed()
    return {"value": round(step_bytes * K * world / secs / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(secs / K * 1e3, 5),
            "path": "eager: pa.DecodeStep.run_from_host without a graph: one pinned H2D copy, "
                    "pa_slot_mapping + pa_write_kv + pa_decode through the C ABI (argument "
                    "checks, TMA descriptors, launches), one D2H copy, stream synchronize; "
                    "every step",
            "graph": {"value": round(step_bytes * K * world / secs_graph / 1e9, 2), "unit": "GB/s",
                      "ms_per_step": round(secs_graph / K * 1e3, 5),
                      "path": "the same copies and calls captured once as a CUDA graph and "
                              "replayed each step, stream synchronize per step"}}


# ----------------------------------------------------------------------------- prefill


def prefill_keys(w):
    """(query, key) pairs the causal mask admits, per query head: query i of
    sequence s (n new of L) sees L - n + i + 1 keys."""
    qn = np.diff(w.q_start).astype(np.int64)
    L = w.seq_lens.astype(np.int64)
    return int((qn * (L - qn) + qn * (qn + 1) // 2).sum())


def prefill_flops(w):
    """QK^T and PV: 2 * D multiply-adds each per admitted (query head, key)."""
    return 4 * w.head_dim * w.num_q_heads * prefill_keys(w)


def prefill_bytes(w, out_elem=4):
    """Every cached K and V row of a sequence once per KV head, q, the output,
    the table entries and q_start / lengths."""
    L = w.seq_lens.astype(np.int64)
    t = int(w.q_start[-1])
    kv = int(L.sum()) * w.num_kv_heads * w.head_dim * 2 * kv_elem(w)
    q = t * w.num_q_heads * w.head_dim * 2
    out = t * w.num_q_heads * w.head_dim * out_elem
    return kv + q + out + int((-(-L // w.block_size)).sum()) * 4 + 8 * w.num_seqs


def run_prefill(args):
    import torch

    import paged_kv_cache_114_gb300 as pa
    from workloads import make_prefill_config
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pa.lib()
    w = make_prefill_config(args.prefill, kv_dtype="e4m3" if args.kv_dtype == "e4m3" else None)
    fp8 = w.kv_dtype == "e4m3"
    k = to_dev(w.k_cache, dev, None if fp8 else w.dtype)
    v = to_dev(w.v_cache, dev, None if fp8 else w.dtype)
    sc = {"k_scale": w.k_scale, "v_scale": w.v_scale} if fp8 else {}
    tables, lens = to_dev(w.block_tables, dev), to_dev(w.seq_lens, dev)
    slots = pa.slot_mapping(tables, to_dev(w.seq_idx, dev), to_dev(w.positions, dev),
                            w.block_size, w.num_blocks)
    pa.write_kv(to_dev(w.key, dev, w.dtype), to_dev(w.value, dev, w.dtype), slots, k, v, **sc)
    q = to_dev(w.q, dev, w.dtype)
    q_start = to_dev(w.q_start, dev)
    out = torch.empty(tuple(q.shape), dtype=torch.float32, device=dev)
    max_q = int(np.diff(w.q_start).max())
    ws = None if args.no_workspace else pa.new_prefill_workspace(
        w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, max_q, dev)

    def call():
        pa.prefill(q, k, v, tables, lens, q_start, w.scale, max_q_len=max_q, out=out, workspace=ws,
                   **sc)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    if pa.get_device_error(dev):
        raise RuntimeError("device error during warm-up")
    stream = torch.cuda.current_stream(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    with ClockSampler(0) as clocks:
        for a, b in evs:
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize()
    if pa.get_device_error(dev):
        raise RuntimeError("device error in the timed region")
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    flops, nbytes = prefill_flops(w), prefill_bytes(w)
    tflops = flops / (ms / 1e3) / 1e12
    gbs = nbytes / (ms / 1e3) / 1e9
    hbm, _ = measured_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tc_peak, tc_kind = float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        tc_peak, tc_kind = 1900.0, "fallback"
    hbm_bound = args.prefill.startswith("verify")
    kernel = pa.prefill_kernel_name(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                    w.block_size, max_q, ws is not None)
    if w.kv_dtype == "e4m3" and kernel == "prefill_tc_kernel":
        kernel = "prefill_tc_e4m3_kernel"  # the same routing, the E4M3 instantiation
    roofline = ({"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                 "frac": round(gbs / hbm, 4)} if hbm_bound else
                {"bound": "tensor", "achieved": round(tflops, 2), "peak": tc_peak, "unit": "TFLOP/s",
                 "frac": round(tflops / tc_peak, 4)})
    roofline.update({"traffic": None, "kernel": kernel, "mean_call_us": round(ms * 1e3, 2),
                     "peak_source": f"{tc_kind if not hbm_bound else 'measured'} "
                                    f"(MEASURED_PEAKS.json {'hbm_gbs' if hbm_bound else 'bf16_tflops'})"})
    qn = np.diff(w.q_start)
    line = {
        "metric": "paged prefill attention throughput (multi-token causal, one layer)",
        "value": round(gbs if hbm_bound else tflops, 2), "unit": "GB/s" if hbm_bound else "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.kv_dtype or w.dtype, "data": "synthetic",
        "config": {"workload": w.name + ("_e4m3" if fp8 else ""), "kv_dtype": w.cache_dtype,
                   "shape": f"{w.num_seqs} seqs, {w.num_q_heads} q heads / {w.num_kv_heads} kv heads, "
                            f"head_dim {w.head_dim}, block {w.block_size}, seq_len "
                            f"{int(w.seq_lens.min())}..{int(w.seq_lens.max())}, new tokens "
                            f"{int(qn.min())}..{int(qn.max())}",
                   "step": "pa_prefill (new K/V written before the timed region)",
                   "flops_per_call": flops, "algorithmic_bytes_per_call": nbytes,
                   "l2": "K/V pool larger than L2 for verify and prompt; chunk's 189 MB pool "
                         "exceeds the 129 MB L2"},
        "tflops": round(tflops, 2), "kv_gbs": round(gbs, 1), "roofline": roofline,
        "gpu_launches": args.steps, "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- swap


SWAP_WORKLOAD = {"name": "swap16x4096_70b_bf16_b16_8layers", "layers": 8, "seqs": 16,
                 "tokens": 4096, "block_size": 16, "kv_heads": 8, "head_dim": 128}


def run_swap(args):
    """Swap out 16 sequences of 4,096 tokens on the 70B head shape (8 layers of
    the pool, K and V: 2.15 GB) to a pinned host pool and back in, each step one
    pa_swap_blocks call per direction; blocks are scattered in both pools."""
    import torch

    import paged_kv_cache_114_gb300 as pa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pa.lib()
    cfg = SWAP_WORKLOAD
    rng = np.random.default_rng(3000)
    b, h, d, L = cfg["block_size"], cfg["kv_heads"], cfg["head_dim"], cfg["layers"]
    nblk = cfg["seqs"] * cfg["tokens"] // b
    dev_blocks = int(nblk * 1.25)
    pools = [(torch.randn(dev_blocks, b, h, d, dtype=torch.bfloat16, device=dev),
              torch.randn(dev_blocks, b, h, d, dtype=torch.bfloat16, device=dev)) for _ in range(L)]
    host = [(torch.empty(nblk, b, h, d, dtype=torch.bfloat16).pin_memory(),
             torch.empty(nblk, b, h, d, dtype=torch.bfloat16).pin_memory()) for _ in range(L)]
    src_ids = rng.choice(dev_blocks, nblk, replace=False).astype(np.int64)
    host_ids = rng.permutation(nblk).astype(np.int64)
    out_pairs = torch.from_numpy(np.stack([src_ids, host_ids], 1)).to(dev)
    in_pairs = torch.from_numpy(np.stack([host_ids, src_ids], 1)).to(dev)
    dk, dv = [p[0] for p in pools], [p[1] for p in pools]
    hk, hv = [p[0] for p in host], [p[1] for p in host]
    nbytes = 2 * L * nblk * b * h * d * 2

    def timed(fn, steps):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        stream = torch.cuda.current_stream(dev)
        for a, e in evs:
            a.record(stream)
            fn()
            e.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(e) for a, e in evs)

    swap_out = lambda: pa.swap_blocks(dk, dv, hk, hv, out_pairs)
    swap_in = lambda: pa.swap_blocks(hk, hv, dk, dv, in_pairs)
    for _ in range(args.warmup):
        swap_out()
        swap_in()
    torch.cuda.synchronize()
    if pa.get_device_error(dev):
        raise RuntimeError("device error during warm-up")
    with ClockSampler(0) as clocks:
        ms_out = timed(swap_out, args.steps)
        ms_in = timed(swap_in, args.steps)
    if pa.get_device_error(dev):
        raise RuntimeError("device error in the timed region")
    # the link's reference: one contiguous copy-engine transfer of the same bytes
    flat_d = torch.empty(nbytes // 2, dtype=torch.bfloat16, device=dev)
    flat_h = torch.empty(nbytes // 2, dtype=torch.bfloat16).pin_memory()
    ms_ce_out = timed(lambda: flat_h.copy_(flat_d, non_blocking=True), max(3, args.steps // 2))
    ms_ce_in = timed(lambda: flat_d.copy_(flat_h, non_blocking=True), max(3, args.steps // 2))
    # the same pa_swap_blocks between two device pools (HBM read + write)
    pools2 = [(torch.empty_like(p[0]), torch.empty_like(p[1])) for p in pools]
    dd_pairs = torch.from_numpy(np.stack([src_ids, rng.permutation(dev_blocks)[:nblk]], 1)).to(dev)
    ms_dd = timed(lambda: pa.swap_blocks(dk, dv, [p[0] for p in pools2], [p[1] for p in pools2],
                                         dd_pairs), args.steps)
    gbs = lambda ms: nbytes / (ms / 1e3) / 1e9
    hbm, _ = measured_peaks()
    line = {
        "metric": "swap (preemption) block copy GB/s between the GPU pool and a pinned host pool",
        "value": round(gbs(ms_out), 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_out, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg["name"],
                   "shape": f"{cfg['seqs']} seqs x {cfg['tokens']} tokens, {L} layers, K and V, "
                            f"{h} kv heads, head_dim {d}, block {b}: {nblk} blocks per layer, "
                            f"scattered in a {dev_blocks}-block device pool",
                   "bytes_per_call": nbytes},
        "swap_out_gbs": round(gbs(ms_out), 1), "swap_in_gbs": round(gbs(ms_in), 1),
        "swap_out_ms": round(ms_out, 4), "swap_in_ms": round(ms_in, 4),
        "copy_engine_contiguous_gbs": {"out": round(gbs(ms_ce_out), 1), "in": round(gbs(ms_ce_in), 1)},
        "device_to_device_gbs": round(gbs(ms_dd), 1),
        "roofline": {"bound": "c2c", "achieved": round(gbs(ms_out), 1),
                     "peak": round(gbs(ms_ce_out), 1), "unit": "GB/s",
                     "frac": round(ms_ce_out / ms_out, 4), "traffic": None,
                     "peak_source": "measured in this run: one contiguous pinned copy of the same "
                                    "bytes by the copy engine (device to host)",
                     "in": {"achieved": round(gbs(ms_in), 1), "peak": round(gbs(ms_ce_in), 1),
                            "frac": round(ms_ce_in / ms_in, 4)},
                     "device_to_device_frac_of_hbm": round(2 * gbs(ms_dd) / hbm, 4)},
        "gpu_launches": 2 * args.steps, "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- prefix keys

# 32-bit integer operations of one SHA-256 compression as FIPS 180-4 writes it:
# 64 rounds of 26 (Sigma0 5, Sigma1 5, Ch 4, Maj 5, T1 4 adds, T2 1, e 1, a 1),
# 48 schedule words of 13 (sigma0 5, sigma1 5, 3 adds), 8 final adds.
SHA256_OPS_PER_COMPRESSION = 64 * 26 + 48 * 13 + 8
# Integer peak: 152 SMs x 128 INT32 lanes x 2.07 GHz (Blackwell's unified
# FP32/INT32 cores, every lane able to issue an integer op each clock).
ALU_PEAK_TOPS = 152 * 128 * 2.07e9 / 1e12


def run_hash(args):
    import torch

    import paged_kv_cache_114_gb300 as pa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pa.lib()
    n_seq, n_tok, b = 4096, 2048, 16
    rng = np.random.default_rng(4000)
    toks = torch.from_numpy(rng.integers(0, 128000, size=n_seq * n_tok).astype(np.int32)).to(dev)
    off = torch.arange(0, (n_seq + 1) * n_tok, n_tok, dtype=torch.int64, device=dev)
    key_off = torch.arange(0, (n_seq + 1) * (n_tok // b), n_tok // b, dtype=torch.int64, device=dev)
    keys = torch.empty((n_seq * n_tok // b, 32), dtype=torch.uint8, device=dev)
    call = lambda: pa.prefix_hash(toks, off, b, key_offsets=key_off, out=keys)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    with ClockSampler(0) as clocks:
        for a, e in evs:
            a.record(stream)
            call()
            e.record(stream)
        torch.cuda.synchronize()
    if pa.get_device_error(dev):
        raise RuntimeError("device error in the timed region")
    ms = statistics.mean(a.elapsed_time(e) for a, e in evs)
    n_keys = n_seq * n_tok // b
    words = 8 + b
    chunks = n_keys * (((words + 3 + 15) // 16))
    tops = chunks * SHA256_OPS_PER_COMPRESSION / (ms / 1e3) / 1e12
    line = {
        "metric": "prefix-cache keys per second (SHA-256 chain over full blocks)",
        "value": round(n_keys / (ms / 1e3) / 1e6, 2), "unit": "Mkeys/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
        "data": "synthetic",
        "config": {"workload": "hash4096x2048_b16", "shape": f"{n_seq} prompts x {n_tok} token ids, "
                   f"block {b}: {n_keys} keys, {chunks} SHA-256 compressions",
                   "token_bytes": n_seq * n_tok * 4},
        "token_gbs": round(n_seq * n_tok * 4 / (ms / 1e3) / 1e9, 1),
        "roofline": {"bound": "alu", "achieved": round(tops, 2), "peak": round(ALU_PEAK_TOPS, 2),
                     "unit": "Tops/s (32-bit integer)", "frac": round(tops / ALU_PEAK_TOPS, 4),
                     "traffic": None, "kernel": "prefix_hash_kernel",
                     "peak_source": "derived: 152 SMs x 128 INT32 lanes x 2.07 GHz",
                     "ops_per_compression": SHA256_OPS_PER_COMPRESSION},
        "gpu_launches": args.steps, "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- CPU oracle


class OracleSample:
    """Per-sequence inputs for bounded oracle steps.

    A step covers one sequence: the slot mapping and write of its newest token
    and decode of all its query heads. The oracle's write returns a new copy of
    the pool it is given, so each sequence gets a sub-pool holding just its own
    blocks (table remapped to 0..n-1); building it is input preparation and is
    not timed. The oracle functions run unchanged.
    """

    def __init__(self, w):
        self.w = w
        self.state = prepared_oracle_state(w)
        self.newest = {int(w.seq_idx[i]): int(i) for i in step_tokens(w)}
        self.cache = {}
        self.cache_all = False  # keep every sequence's sub-pool (else only the last one)

    def inputs(self, s):
        if s not in self.cache:
            w = self.w
            nblk = -(-int(w.seq_lens[s]) // w.block_size)
            blocks = w.block_tables[s, :nblk]
            entry = (self.state["k"][blocks], self.state["v"][blocks],
                     np.arange(max(nblk, 1), dtype=np.int32)[None])
            if self.cache_all:
                self.cache[s] = entry
            else:
                self.cache = {s: entry}
        return self.cache[s]

    def step(self, s):
        import oracle
        w = self.w
        k, v, table = self.inputs(s)
        i = self.newest.get(s)
        n_tok = 0
        fp8 = {"kv_dtype": "e4m3", "k_scale": w.k_scale, "v_scale": w.v_scale} \
            if w.kv_dtype == "e4m3" else {}
        if i is not None:
            slots = oracle.slot_mapping(table, [0], [int(w.positions[i])], w.block_size)
            if fp8:
                k, v = oracle.write_kv_e4m3(k, v, w.key[i:i + 1], w.value[i:i + 1], slots, w.dtype,
                                            w.k_scale, w.v_scale)
            else:
                k, v = oracle.write_kv(k, v, w.key[i:i + 1], w.value[i:i + 1], slots)
            n_tok = 1
        oracle.decode(w.q[s:s + 1], k, v, table, w.seq_lens[s:s + 1], w.scale, w.dtype, **fp8)
        return n_tok


def sample_bytes(w, seqs, n_tok):
    L = w.seq_lens[list(seqs)].astype(np.int64)
    kv = int(L.sum()) * w.num_kv_heads * w.head_dim * 2 * kv_elem(w)
    q = len(seqs) * w.num_q_heads * w.head_dim * (2 + 4)
    tables = int((-(-L // w.block_size)).sum()) * 4 + 4 * len(seqs)
    return kv + q + tables + write_bytes(w, n_tok)


def prepared_oracle_state(w):
    """The pool as the timed steps see it (config 5: copies and suffix writes applied)."""
    import oracle
    k, v = w.k_cache, w.v_cache
    idx = step_tokens(w)
    setup = np.setdiff1d(np.arange(len(w.positions)), idx)
    if len(w.copy_pairs):
        ks, vs = oracle.copy_blocks([k], [v], [tuple(p) for p in w.copy_pairs.tolist()])
        k, v = ks[0], vs[0]
    if len(setup):
        sl = oracle.slot_mapping(w.block_tables, w.seq_idx[setup], w.positions[setup], w.block_size)
        if w.kv_dtype == "e4m3":
            k, v = oracle.write_kv_e4m3(k, v, w.key[setup], w.value[setup], sl, w.dtype,
                                        w.k_scale, w.v_scale)
        else:
            k, v = oracle.write_kv(k, v, w.key[setup], w.value[setup], sl)
    return {"k": k, "v": v}


def cpu_baseline_child(config, block_size, mode, steps=0, warmup=0, kv_dtype="native"):
    """Runs the oracle timing in a fresh single-threaded process."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-child", mode, "--config", str(config),
           "--steps", str(steps), "--warmup", str(warmup), "--kv-dtype", kv_dtype]
    if block_size is not None:
        cmd += ["--block-size", str(block_size)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=1200)
    if r.returncode != 0:
        return {"value": None, "error": r.stderr.strip().splitlines()[-1:] or ["failed"]}
    return json.loads(r.stdout.strip().splitlines()[-1])


_POOL_SAMPLER = None  # the forked workers' view of the parent's OracleSample


def _pool_step(s):
    """One oracle step in a pool worker: (bytes, seconds)."""
    t0 = time.perf_counter()
    n_tok = _POOL_SAMPLER.step(int(s))
    dt = time.perf_counter() - t0
    return sample_bytes(_POOL_SAMPLER.w, [int(s)], n_tok), dt


def oracle_all_cores(sampler, seqs, cores):
    """Wall-clock rate of the oracle over `seqs` spread across `cores` worker
    processes (one sequence per task, BLAS threads pinned to 1 in each). The
    workers are forked from this process, which has never touched a GPU, after
    every sequence's sub-pool is built, so they share those inputs."""
    import multiprocessing as mp
    global _POOL_SAMPLER
    for s in seqs:
        sampler.inputs(int(s))
    _POOL_SAMPLER = sampler
    ctx = mp.get_context("fork")
    with ctx.Pool(cores) as pool:
        pool.map(_pool_step, seqs[:cores], chunksize=1)  # workers warmed up
        t0 = time.perf_counter()
        res = pool.map(_pool_step, seqs, chunksize=1)
        wall = time.perf_counter() - t0
    return sum(r[0] for r in res), wall


def cpu_child(args):
    """Oracle timing: 'cpu_baseline' = a bounded single-thread sample (about
    12 s of CPU) and the same steps across all host cores; 'reference' = the
    reference arm's W + K steps, each one random sequence."""
    w = load_workload(args.config, args.block_size, args.kv_dtype)
    sampler = OracleSample(w)
    rng = np.random.default_rng(0)
    if args.cpu_child == "cpu_baseline":
        budget, done_b, t_used, order = 12.0, 0, 0.0, rng.permutation(w.num_seqs)
        seqs_done = 0
        for s in order:
            sampler.inputs(int(s))
            t0 = time.perf_counter()
            n_tok = sampler.step(int(s))
            t_used += time.perf_counter() - t0
            done_b += sample_bytes(w, [int(s)], n_tok)
            seqs_done += 1
            if t_used >= budget:
                break
        one = {"value": round(done_b / t_used / 1e9, 4), "unit": "GB/s", "cores": 1,
               "sample": f"{seqs_done} of {w.num_seqs} sequences in random order, each: its new "
                         f"token's slot mapping and write, decode of all {w.num_q_heads} heads; "
                         f"{t_used:.1f} s of single-thread CPU time"}
        cores = os.cpu_count() or 1
        # about 10 s of wall time on every core (at the single-thread rate),
        # passes over the batch in the same random order
        n_all = int(min(max(cores, round(10.0 * cores * seqs_done / t_used)), 32 * w.num_seqs))
        seqs = [int(order[i % w.num_seqs]) for i in range(n_all)]
        sampler.cache_all = True
        all_b, wall = oracle_all_cores(sampler, seqs, cores)
        res = {"value": round(all_b / wall / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{n_all} sequence steps (the batch of {w.num_seqs} in random order, "
                         f"repeated as needed), each: its new token's slot mapping and write, decode "
                         f"of all {w.num_q_heads} heads; {cores} worker processes, one BLAS thread "
                         f"each, {wall:.1f} s wall",
               "single_core": one}
        print(json.dumps(res))
        return
    total_b, total_t = 0, 0.0
    for i in range(args.warmup + args.steps):
        s = int(rng.integers(0, w.num_seqs))
        sampler.inputs(s)
        t0 = time.perf_counter()
        n_tok = sampler.step(s)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            total_b += sample_bytes(w, [s], n_tok)
            total_t += dt
    print(json.dumps({"value": round(total_b / total_t / 1e9, 4),
                      "ms_per_step": round(total_t / max(args.steps, 1) * 1e3, 4),
                      "sample": f"each step: one random sequence of {w.num_seqs} (its new token's "
                                f"slot mapping and write, decode of all {w.num_q_heads} heads), "
                                f"single thread"}))


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    res = cpu_baseline_child(args.config, args.block_size, "reference", args.steps, args.warmup,
                             kv_dtype=args.kv_dtype)
    w = load_workload(args.config, args.block_size, args.kv_dtype)
    line = {
        "impl": "reference", "metric": METRIC, "value": res.get("value"), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": res.get("ms_per_step"), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name,
                   "note": "the pages publish no runnable reference; this arm times the fp64 CPU oracle"},
        "cpu_baseline": {"value": res.get("value"), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": res.get("sample")},
        "e2e": {"value": res.get("value"), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--block-size", type=int, default=None, help="config 4 block size (8/16/32)")
    ap.add_argument("--partition", type=int, default=None, help="split-K partition tokens (default: library's)")
    ap.add_argument("--prefill", default=None,
                    choices=["verify4_70b_bf16_b16", "chunk512_gqa_bf16_b16", "prompt2k_mha_fp16_b16",
                             "verify4_long_bf16_b16"],
                    help="time pa_prefill on a named multi-token workload instead")
    ap.add_argument("--no-workspace", action="store_true",
                    help="with --prefill: no workspace, so few-token batches run one CTA per "
                         "(sequence, KV head, 64 rows) instead of the balanced kernel")
    ap.add_argument("--hash", action="store_true",
                    help="time pa_prefix_hash on 4,096 prompts of 2,048 token ids instead")
    ap.add_argument("--swap", action="store_true",
                    help="time pa_swap_blocks between the GPU pool and a pinned host pool instead")
    ap.add_argument("--kv-dtype", choices=["native", "e4m3"], default="native",
                    help="pool element type: the config's fp16/bf16, or FP8 E4M3 codes (configs 2-5)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-child", choices=["cpu_baseline", "reference"], default=None,
                    help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.cpu_child is None and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    if args.cpu_child:
        return cpu_child(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.prefill:
        return run_prefill(args)
    if args.swap:
        return run_swap(args)
    if args.hash:
        return run_hash(args)
    return run_gpu(args)


if __name__ == "__main__":
    main()
