"""Paged decode benchmark: fused append + GQA decode over a paged KV cache.

Workload (one step = one decode step of a 36-layer Qwen3-4B-shaped model's
attention): the batch sweep at B=64, Hq=32, Hkv=8, D=128, page 128, prompt
uniform in [64, 512], 36 per-layer K/V pools sharing one block table,
shuffled page layout.  Every step appends one token per row in every layer
and attends over all cached tokens; decode step s (0 <= s < 512) attends
prompt + s + 1 tokens per row.  The K timed steps are spread evenly over the
whole 512-step cycle (timed step i runs decode step floor((i + 1/2) * 512 / K)),
so the timed region measures the cycle's mean whatever K is.  Each step
reads ~5 GB of K/V, far above the 129 MB L2, so no flush is needed between
steps.

Prints one JSON line.  `value` = algorithmic KV-path bytes / device time
(GB/s) over the timed steps; `roofline` = the decode kernel's average
launch (CUDA events around the timed region, which launches nothing else);
`e2e` = the same metric through the C ABI with the step's q / k_new / v_new
copied from pinned host memory and the outputs copied back inside the timed
region.  Also in the line: the same sweep on contiguous pages, the two
single-layer decode workloads (Qwen3-4B-shaped layer, skewed lengths), the
ragged prefill and the two mixed-step workloads.

`--impl reference` times the fp64 CPU oracle on the host cores instead
(bounded samples of the same workload).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode KV-read GB/s (% of HBM peak) and decode tok/s per attn layer"
HQ, HKV, D, P = 32, 8, 128, 128
DECODE_CAPACITY = 512
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_kernel_traffic.txt")
PREFILL_PROFILE_FILE = os.path.join(ROOT, "profiles", "prefill_kernel_counters.txt")


PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def tensor_peak():
    """Dense bf16 TFLOP/s for a kernel timed alone (measured burst, else the
    fallback figure)."""
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["bf16_tflops"]), "measured bf16 burst (cuBLAS)"
    except Exception:
        return 1900.0, "fallback"


def call_bytes(lens: np.ndarray, batch: int, page_size: int = P) -> int:
    """Algorithmic bytes of one fused append + decode call (one layer):
    cached K/V read + q read + out write + new K/V read + append write +
    block-table entries read + seqlens read."""
    kv_read = int(lens.sum()) * 2 * HKV * D * 2
    q_out = 2 * batch * HQ * D * 2
    new_tok = 2 * batch * 2 * HKV * D * 2
    table = 4 * int(((lens + 1 + page_size - 1) // page_size).sum())
    return kv_read + q_out + new_tok + table + 4 * batch


def source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_append_gb300", "csrc")
    for name in ("pkv_decode.cu", "pkv_device.cuh", "pkv_internal.h"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def prefill_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_append_gb300", "csrc")
    for name in ("pkv_prefill.cu", "pkv_tcgen05.cuh", "pkv_device.cuh", "pkv_internal.h"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_prefill_profile():
    """Tensor-pipe share and DRAM bytes of the prefill kernel from the
    committed ncu summary, if it was taken on the current kernel source."""
    try:
        rec = {}
        with open(PREFILL_PROFILE_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    rec[k.strip()] = v.strip()
        if rec.get("source_sha256") != prefill_source_hash():
            return None
        return {"tensor_pipe_pct": float(rec["tensor_pipe_pct"]), "dram_bytes": float(rec["dram_bytes"])}
    except Exception:
        return None


def mixed_bench(kind: str, reps: int, warmup: int, decode_max_qlen, dev=None) -> dict:
    """One mixed step (pkv_mixed_attn: append + decode kernel + prefill
    kernel) per timed iteration on the Qwen3-4B-shaped layer: speculative
    decode (B=32 rows of 4 tokens on U[512,1024]) or a chunked-prefill step
    (4 chunks of 496 tokens on prefixes U[0,2048] + 60 decode rows on
    U[512,1024]).  CUDA events around each call, L2 flushed by a 512 MiB write
    before it.  Prints one JSON line: GB/s of the step's algorithmic bytes and
    TFLOP/s of its causal pairs, against the measured peaks.  Returns the
    line as a dict."""
    import paged_kv_decode_append_gb300 as pkv
    from paged_kv_decode_append_gb300 import workloads as wl

    if dev is None:
        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
    case = (wl.spec_decode if kind == "spec" else wl.chunked_mix)(device=dev)
    q, kn, vn = case.q, case.k_new.to(dev), case.v_new.to(dev)
    T, Hq, Dh = q.shape
    B = case.batch
    ql = np.diff(case.qo_indptr).astype(np.int64)
    L = case.cache_seqlens.astype(np.int64)
    max_qlen = int(ql.max())
    # decode_max_qlen is the caller's choice: rows of up to that many queries
    # take the decode kernel.  The chunked step's decode rows hold one token
    # each, so it passes 1 (the one-query instantiation); the library default
    # sizes the decode units for speculative rows of up to 16 / G queries
    if decode_max_qlen is None:
        dq = 1 if kind == "chunked" else pkv.default_decode_max_qlen(Hq, case.num_kv_heads)
    else:
        dq = int(decode_max_qlen)
    qo = torch.as_tensor(case.qo_indptr, device=dev)
    bt = torch.as_tensor(case.block_table, device=dev)
    sl = torch.as_tensor(case.cache_seqlens, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = pkv.mixed_workspace(B, T, case.max_blocks, Hq, max_qlen, dq, pkv.cache_desc(case.k_cache, case.layout),
                             dev)
    # algorithmic bytes: cached K/V read, new K/V read and appended, q read,
    # out write, block-table entries and the two int32 row arrays
    Hkv = case.num_kv_heads
    nbytes = (int(L.sum()) * 2 * Hkv * Dh * 2 + 2 * T * 2 * Hkv * Dh * 2 + 2 * T * Hq * Dh * 2 +
              4 * int(((L + ql + case.page_size - 1) // case.page_size).sum()) + 4 * (2 * B + 1))
    pairs = Hq * int((ql * L + ql * (ql + 1) // 2).sum())  # query i of a row sees L + i + 1 keys
    flops = 4 * Dh * pairs
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        # the same slots are appended to every time (cache_seqlens is not advanced)
        pkv.pkv_mixed_attn(case.k_cache, case.v_cache, q, kn, vn, qo, bt, sl, case.softmax_scale, max_qlen, dq,
                           out=out, lse=lse, workspace=ws, err_flag=err, layout=case.layout)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    times = []
    with ClockSampler(0) as clocks:
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
    if int(err.item()) != 0:
        raise RuntimeError(f"mixed step reported error bits {int(err.item())}")
    times = np.array(times)
    ms = float(np.median(times))
    gbs = nbytes / (ms * 1e-3) / 1e9
    tflops = flops / (ms * 1e-3) / 1e12
    hbm, hbm_kind = peaks()
    tpk, tpk_kind = tensor_peak()
    n_prefill = int((ql > dq).sum())
    launches = 1 + 1 + (2 if max_qlen > dq else 0)
    name = ("speculative decode, Qwen3-4B-shaped layer: B=32 rows of 4 new tokens, Hq=32, Hkv=8, D=128, page 16, "
            "cached lengths U[512,1024], 65,536-page shuffled pool" if kind == "spec" else
            "chunked-prefill step, Qwen3-4B-shaped layer: 4 chunks of 496 tokens on prefixes U[0,2048] + 60 decode "
            "rows on U[512,1024] (2,044 new tokens), Hq=32, Hkv=8, D=128, page 16, 65,536-page shuffled pool")
    return {
        "metric": "mixed-step GB/s (% of HBM peak) and TFLOP/s (% of bf16 peak)", "value": gbs, "unit": "GB/s",
        "n_gpus": 1, "steps": reps, "warmup": warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "batch": B, "total_q": T, "decode_max_qlen": dq,
                   "rows_on_prefill_kernel": n_prefill, "l2": "flushed between calls (512 MiB write)"},
        "pct_of_hbm_peak": 100.0 * gbs / hbm, "tflops": tflops, "pct_of_tensor_peak": 100.0 * tflops / tpk,
        "algorithmic_bytes_per_call": nbytes, "flops_per_call": flops, "flops_formula": "4 * head_dim * causal pairs",
        "ms_best": float(times.min()), "hbm_peak": hbm, "hbm_peak_kind": hbm_kind, "tensor_peak": tpk,
        "tensor_peak_kind": tpk_kind, "clocks": clocks.summary(), "gpu_launches": reps * launches}


def prefill_bench(dev, reps: int, head_dim: int = 256):
    """The ragged causal prefill workload (B=8, Hq=48, Hkv=6, D=256, page 16
    HND; head_dim 128 or 64 for the other kernels, same lengths): one
    pkv_prefill_attn call per timed iteration (plan + kernel), CUDA events
    around it, L2 flushed by a 512 MiB write before each call."""
    import paged_kv_decode_append_gb300 as pkv
    from paged_kv_decode_append_gb300 import workloads as wl

    case = wl.ragged_prefill(device=dev, head_dim=head_dim)
    q = case.q
    T, Hq, Dh = q.shape
    qo = torch.as_tensor(case.qo_indptr, device=dev)
    kvl = torch.as_tensor(case.kv_lens, device=dev)
    btp = torch.as_tensor(case.block_table, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    ws = pkv.prefill_workspace(case.batch, T, Hq, pkv.cache_desc(case.k_cache, case.layout), dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ql = np.diff(case.qo_indptr).astype(np.int64)
    kv = case.kv_lens.astype(np.int64)
    pairs = Hq * int((ql * (2 * kv - ql + 1) // 2).sum())  # visited (query, key, head) triples
    flops = 4 * Dh * pairs
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        pkv.pkv_prefill_attn(case.k_cache, case.v_cache, q, qo, kvl, btp, case.softmax_scale, out=out, lse=lse,
                             workspace=ws, err_flag=err, layout=case.layout)

    for _ in range(3):
        call()
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        call()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    if int(err.item()) != 0:
        raise RuntimeError(f"prefill reported error bits {int(err.item())}")
    times = np.array(times)
    ms = float(np.median(times))
    tflops = flops / (ms * 1e-3) / 1e12
    peak, peak_kind = tensor_peak()
    prof = recorded_prefill_profile() if head_dim == 256 else None
    return {
        "workload": f"ragged causal paged prefill: B=8, Hq=48, Hkv=6, D={head_dim}, page 16 HND, "
                    f"q_len {ql.min()}..{ql.max()}, kv_len {kv.min()}..{kv.max()} (seed 4)",
        "tflops": tflops, "unit": "TFLOP/s", "peak": peak, "peak_kind": peak_kind,
        "frac": tflops / peak, "ms_median": ms, "ms_best": float(times.min()), "reps": reps,
        "flops": flops, "pairs": pairs, "flops_formula": "4 * head_dim * causal pairs",
        "launches_per_call": 2, "l2": "flushed between calls (512 MiB write)",
        "tensor_pipe_pct": None if prof is None else prof["tensor_pipe_pct"],
        "dram_bytes_per_call": None if prof is None else prof["dram_bytes"],
    }


def recorded_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, scaled to
    this workload's launch, if it was taken on the current kernel source."""
    try:
        rec = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    rec[k.strip()] = v.strip()
        if rec.get("source_sha256") != source_hash():
            return None
        return float(rec["dram_bytes_per_algorithmic_byte"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend, device_id=torch.device(f"cuda:{local}") if backend == "nccl" else None)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def timed_decode_steps(n: int) -> list:
    """Decode steps of n timed iterations, spread evenly over the cycle:
    iteration i runs step floor((i + 1/2) * 512 / n) (mod 512), so the mean
    work of any n steps is the cycle's mean."""
    return [int((i + 0.5) * DECODE_CAPACITY / n) % DECODE_CAPACITY for i in range(n)]


def cpu_baseline(sw, steps: list, budget_s: float = 12.0, host_layers: int = 2, max_calls: int = 4000):
    """Times the fp64 oracle (all host cores) on whole layer calls (all rows
    and heads) of the timed decode steps, in order, until `budget_s` of
    oracle time is spent; returns GB/s of the same algorithmic bytes.  Every
    layer call of a step costs the same, so the calls cycle over the first
    `host_layers` layer pools (host copies of those only)."""
    import oracle
    from paged_kv_decode_append_gb300 import workloads as wl

    dev = sw.k_caches[0].device
    rows = list(range(sw.batch))
    need = sw.prompt_lens + DECODE_CAPACITY
    host = []
    for layer in range(host_layers):
        k, v, bt = wl.compact_rows(sw.k_caches[layer], sw.v_caches[layer], sw.block_table, rows, need, P)
        host.append((k, v, bt))
    d = oracle.CacheDesc(host[0][0].shape[0], P, HKV, D, oracle.NHD)
    threads = oracle.max_threads(0)
    done_bytes, elapsed, calls, used = 0, 0.0, 0, []
    for i in range(max_calls):  # the timed steps in order, cyclically, until the budget is spent
        if elapsed >= budget_s:
            break
        step = steps[i % len(steps)]
        lens = (sw.prompt_lens + step).astype(np.int32)
        layer = i % host_layers
        q, kn, vn = (wl.bits(t) for t in wl.sweep_step_inputs(sw, step, dev, layers=layer + 1)[layer])
        k, v, bt = host[layer]
        t0 = time.perf_counter()
        oracle.decode(d, k, v, q, kn, vn, bt, lens, sw.softmax_scale, nthreads=0)
        elapsed += time.perf_counter() - t0
        done_bytes += call_bytes(lens, sw.batch)
        calls += 1
        used.append(step)
    # the same oracle on one host thread: the first two sampled calls
    one_bytes, one_t = 0, 0.0
    for i, step in enumerate(steps[:2]):
        lens = (sw.prompt_lens + step).astype(np.int32)
        layer = i % host_layers
        q, kn, vn = (wl.bits(t) for t in wl.sweep_step_inputs(sw, step, dev, layers=layer + 1)[layer])
        k, v, bt = host[layer]
        t0 = time.perf_counter()
        oracle.decode(d, k, v, q, kn, vn, bt, lens, sw.softmax_scale, nthreads=1)
        one_t += time.perf_counter() - t0
        one_bytes += call_bytes(lens, sw.batch)
    return {"value": done_bytes / elapsed / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "single_thread_value": one_bytes / one_t / 1e9,
            "single_thread_sample": f"one layer call of decode steps {steps[:2]}, one host thread",
            "sample": f"{calls} layer calls (the timed decode steps in turn, steps {min(used)}..{max(used)} of the "
                      f"512-step cycle, of the 36-layer B={sw.batch} workload, all rows and heads), fp64 oracle "
                      f"with OpenMP over (row, head), {elapsed:.1f} s of oracle time"}


def run_reference(args):
    """The reference arm: the fp64 oracle timed on the host cores.  Each
    timed step runs one layer call (all rows and heads) of the same decode
    step the GPU arm times; a step of the 36-layer workload is that call
    times 36 (every layer call of a step does the same work).  Under a
    multi-rank launch rank 0 alone runs and prints; the others exit at once."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    from paged_kv_decode_append_gb300 import workloads as wl

    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    sw = wl.batch_sweep(args.batch, device=dev, contiguous=args.layout == "contiguous", layers=1,
                        data_device=dev, fill_decode=True)
    rows = list(range(sw.batch))
    threads = oracle.max_threads(0)
    k, v, bt = wl.compact_rows(sw.k_caches[0], sw.v_caches[0], sw.block_table, rows,
                               sw.prompt_lens + DECODE_CAPACITY, P)
    d = oracle.CacheDesc(k.shape[0], P, HKV, D, oracle.NHD)
    times, nbytes = [], []
    steps = timed_decode_steps(args.warmup) + timed_decode_steps(args.steps)
    for i, step in enumerate(steps):
        lens = (sw.prompt_lens + step).astype(np.int32)
        q, kn, vn = (wl.bits(t) for t in wl.sweep_step_inputs(sw, step, dev, layers=1)[0])
        t0 = time.perf_counter()
        oracle.decode(d, k, v, q, kn, vn, bt, lens, sw.softmax_scale, nthreads=0)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            nbytes.append(call_bytes(lens, sw.batch))
    total_t = float(sum(times))
    value = sum(nbytes) / total_t / 1e9
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_t / len(times) * args.layers,
        "ms_per_layer_call": 1e3 * total_t / len(times),
        "ms_per_step_basis": f"one layer call timed per step, times {args.layers} layers",
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"one layer call per timed step (layer 0 of the 36, the GPU arm's decode steps), "
                                   f"B={args.batch}, fp64 oracle"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))


def single_layer_bench(kind: str, reps: int, warmup: int):
    """One fused append + decode call per timed iteration on the Qwen3-4B-shaped
    layer (B=32, page 16, lengths U[512,1024]) or the skewed batch (B=64, one
    32,768-token row), CUDA events around each call, L2 flushed by a 512 MiB
    write before it (a call reads 0.1-0.4 GB, about L2's size).  Returns a
    dict in the main line's format (plus the streamed form of the call)."""
    import paged_kv_decode_append_gb300 as pkv
    from paged_kv_decode_append_gb300 import workloads as wl

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    case = (wl.qwen3_decode if kind == "qwen3" else wl.skewed_decode)(device=dev)
    B, Hq, Dh = case.q.shape
    bt = torch.as_tensor(case.block_table, device=dev)
    lens = torch.as_tensor(case.cache_seqlens, device=dev)
    out = torch.empty_like(case.q)
    ws = pkv.decode_workspace(B, case.max_blocks, Hq, pkv.cache_desc(case.k_cache, case.layout), dev)
    nbytes = call_bytes(case.cache_seqlens.astype(np.int64), B, case.page_size)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        # the same slot is appended to every time (cache_seqlens is not advanced)
        pkv.pkv_decode_attn(case.k_cache, case.v_cache, case.q, case.k_new, case.v_new, bt, lens,
                            case.softmax_scale, out=out, workspace=ws, layout=case.layout)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    times = []
    with ClockSampler(0) as clocks:
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
    times = np.array(times)
    ms = float(np.median(times))
    value = nbytes / (ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    streamed = streamed_layer_calls(case, bt, lens, out, ws, nbytes, peak, dev)
    name = ("Qwen3-4B-shaped layer decode: B=32, Hq=32, Hkv=8, D=128, page 16, lengths U[512,1024], 65,536-page "
            "shuffled pool" if kind == "qwen3" else
            "skewed-length decode: B=64, Hq=32, Hkv=8, D=128, page 16, one 32,768-token row, others "
            "clip(lognormal(6.5,0.8),128,4096), 65,536-page shuffled pool")
    del case, flush
    torch.cuda.empty_cache()
    return {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1, "steps": reps, "warmup": warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": name, "batch": B, "l2": "flushed between calls (512 MiB write)"},
        "pct_of_hbm_peak": 100.0 * value / peak, "decode_tok_s_per_attn_layer": B / (ms * 1e-3),
        "ms_best": float(times.min()), "algorithmic_bytes_per_call": nbytes, "peak": peak, "peak_kind": peak_kind,
        "clocks": clocks.summary(), "gpu_launches": reps, "streamed": streamed}


def streamed_layer_calls(case, bt, lens, out, ws, nbytes, peak, dev, rounds: int = 5):
    """The same call back to back, as the layers of a model would issue it:
    R copies of the layer's pool (R x the call's bytes >= 4 x L2, so no call
    finds its pages in L2), one call per copy in turn, launched with
    programmatic dependent launch (overlapped prologue, early K/V stream; a
    call appends into its own copy only) and captured in one CUDA graph of
    N calls.  Returns the per-call GB/s over `rounds` replays."""
    import paged_kv_decode_append_gb300 as pkv

    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 << 20)
    copies = max(2, -(-4 * l2 // nbytes))
    pools = [(case.k_cache, case.v_cache)] + [(case.k_cache.clone(), case.v_cache.clone())
                                              for _ in range(copies - 1)]
    n_calls = copies * max(1, 24 // copies)
    flags = pkv.api.DECODE_OVERLAP_PROLOGUE | pkv.api.DECODE_EARLY_KV
    # the calls share cache_seqlens and block_table: the first makes the step plan, the others reuse it
    call_flags = [flags | (pkv.api.DECODE_MAKE_PLAN if i == 0 else pkv.api.DECODE_USE_PLAN) for i in range(n_calls)]
    stream = torch.cuda.Stream(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for i in range(copies):  # warm-up outside the graph (opt-in attributes, first-call set-up)
            k, v = pools[i]
            pkv.pkv_decode_attn(k, v, case.q, case.k_new, case.v_new, bt, lens, case.softmax_scale, out=out,
                                workspace=ws, layout=case.layout, flags=call_flags[i])
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(n_calls):
                k, v = pools[i % copies]
                pkv.pkv_decode_attn(k, v, case.q, case.k_new, case.v_new, bt, lens, case.softmax_scale, out=out,
                                    workspace=ws, layout=case.layout, flags=call_flags[i])
        graph.replay()
        graph.replay()
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(rounds):
            graph.replay()
        b.record(stream)
        b.synchronize()
    ms = a.elapsed_time(b) / (rounds * n_calls)
    del graph, pools
    torch.cuda.empty_cache()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"value": gbs, "unit": "GB/s", "pct_of_hbm_peak": 100.0 * gbs / peak, "ms_per_call": ms,
            "copies": int(copies), "calls_per_graph": int(n_calls), "replays": rounds,
            "launch": "one CUDA graph of back-to-back calls, programmatic dependent launch (overlapped prologue "
                      "and early K/V stream), each call on the next of the rotating pool copies; the first call "
                      "makes the step plan, the others reuse it",
            "l2": f"{copies} rotating copies of the layer pool (copies x call bytes >= 4 x L2)"}


def workload_config(args, layout=None):
    steps = timed_decode_steps(args.steps)
    layout = args.layout if layout is None else layout
    return {"workload": f"paged decode batch sweep B={args.batch} (Qwen3-4B-shaped: Hq=32, Hkv=8, D=128), "
                        f"page 128, {layout} pages, prompt U[64,512] + decode steps of the 512-step cycle, "
                        f"{args.layers} layer caches per step; {args.steps} timed steps spread over the cycle: "
                        f"step floor((i + 1/2) * 512 / {args.steps}) for i < {args.steps} "
                        f"(steps {min(steps)}..{max(steps)})",
            "batch": args.batch, "num_q_heads": HQ, "num_kv_heads": HKV, "head_dim": D, "page_size": P,
            "layers": args.layers, "layout": layout, "decode_steps_timed": [min(steps), max(steps)],
            "l2": "inputs larger than L2: every step streams 36 distinct layer caches (~5 GB)"}


class Sweep:
    """The 36-layer batch-sweep decode of one rank: pools, per-step inputs and
    one CUDA graph per decode step (its layers' launches back to back)."""

    def __init__(self, pkv, wl, args, dev, layout: str, seed: int, flags: int, plan: bool):
        B, L = args.batch, args.layers
        self.pkv, self.args, self.dev, self.B, self.L, self.flags, self.plan = pkv, args, dev, B, L, flags, plan
        self.sw = wl.batch_sweep(B, device=dev, contiguous=layout == "contiguous", layers=L, seed=seed,
                                 fill_decode=True)
        self.bt = torch.as_tensor(self.sw.block_table, device=dev)
        self.lens_all = (self.sw.prompt_lens[None, :] + np.arange(DECODE_CAPACITY)[:, None]).astype(np.int32)
        self.lens_dev = torch.as_tensor(self.lens_all, device=dev)
        desc = pkv.cache_desc(self.sw.k_caches[0])
        self.ws = pkv.decode_workspace(B, self.sw.max_blocks, HQ, desc, dev)
        ring = 8  # distinct per-step input sets, reused round-robin
        self.inputs = [wl.sweep_step_inputs(self.sw, s, dev, layers=L) for s in range(ring)]
        self.outs = [torch.empty(B, HQ, D, dtype=torch.bfloat16, device=dev) for _ in range(L)]
        self.step_bytes = [L * call_bytes(self.lens_all[s], B) for s in range(DECODE_CAPACITY)]

    def step_inputs(self, step):
        return self.inputs[step % len(self.inputs)]

    def layer_flags(self, layer):
        """Launch flags of one layer of a step: with step plans, layer 0 makes
        the plan (one extra small kernel) and every later layer reuses it."""
        if not self.plan:
            return self.flags
        api = self.pkv.api
        return self.flags | (api.DECODE_MAKE_PLAN if layer == 0 else api.DECODE_USE_PLAN)

    def layer_call(self, step, layer, q, kn, vn, flags=None):
        self.pkv.pkv_decode_attn(self.sw.k_caches[layer], self.sw.v_caches[layer], q, kn, vn, self.bt,
                                 self.lens_dev[step], self.sw.softmax_scale, out=self.outs[layer], workspace=self.ws,
                                 flags=self.layer_flags(layer) if flags is None else flags)

    def graph(self, step):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for layer, (q, kn, vn) in enumerate(self.step_inputs(step)):
                self.layer_call(step, layer, q, kn, vn)
        return g

    def timed(self, warm_steps, steps, world, local, clocks=True):
        """Replays the graphs of `warm_steps`, then times `steps` back to back
        (barrier + synchronize on both sides).  Returns (ms, bytes)."""
        warm = [self.graph(s) for s in warm_steps]
        graphs = [self.graph(s) for s in steps]
        torch.cuda.synchronize(self.dev)
        for g in warm:
            g.replay()
        torch.cuda.synchronize(self.dev)
        barrier(world)
        stream = torch.cuda.current_stream(self.dev)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        total = 0
        sampler = ClockSampler(local) if clocks else None
        if sampler is not None:
            sampler.__enter__()
        try:
            torch.cuda.synchronize(self.dev)
            barrier(world)
            torch.cuda.nvtx.range_push("timed")
            start.record(stream)
            for s, g in zip(steps, graphs):
                g.replay()
                total += self.step_bytes[s]
            end.record(stream)
            torch.cuda.nvtx.range_pop()
            torch.cuda.synchronize(self.dev)
            barrier(world)
        finally:
            if sampler is not None:
                sampler.__exit__(None, None, None)
        del warm, graphs
        return start.elapsed_time(end), total, (sampler.summary() if sampler is not None else None)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=DECODE_CAPACITY)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--batch", type=int, default=64)
    ap.add_argument("--layers", type=int, default=36)
    ap.add_argument("--layout", default="shuffled", choices=["shuffled", "contiguous"])
    ap.add_argument("--e2e-steps", type=int, default=DECODE_CAPACITY)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-reps", type=int, default=20, help="timed prefill calls (0 = skip)")
    ap.add_argument("--mixed-reps", type=int, default=20,
                    help="timed mixed-step calls per mixed workload in the default line (0 = skip)")
    ap.add_argument("--layer-reps", type=int, default=20,
                    help="timed single-layer calls per single-layer workload in the default line (0 = skip)")
    ap.add_argument("--no-contiguous", action="store_true",
                    help="skip the contiguous-pages sweep of the default line")
    ap.add_argument("--prefill-only", action="store_true",
                    help="run only the prefill measurement on cuda:0 and print its JSON object")
    ap.add_argument("--workload", default="sweep", choices=["sweep", "qwen3", "skewed", "spec", "chunked"],
                    help="sweep: the 36-layer batch sweep (default); qwen3 / skewed: one decode layer, timed per "
                         "call; spec / chunked: one mixed step (pkv_mixed_attn), timed per call")
    ap.add_argument("--decode-max-qlen", type=int, default=None,
                    help="spec / chunked: longest row on the decode kernel (default: 1 for chunked, whose "
                         "decode rows are single-token; the library's for spec)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="plain launches instead of programmatic dependent launch between layers")
    ap.add_argument("--no-plan", action="store_true",
                    help="every layer plans its work split itself (no step plan shared by the layers)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    if args.impl == "reference":
        run_reference(args)
        return
    if args.workload in ("spec", "chunked"):
        reps = 50 if args.steps == ap.get_default("steps") else args.steps
        print(json.dumps(mixed_bench(args.workload, reps, args.warmup, args.decode_max_qlen)))
        return
    if args.workload != "sweep":
        reps = 50 if args.steps == ap.get_default("steps") else args.steps
        print(json.dumps(single_layer_bench(args.workload, reps, args.warmup)))
        return
    if args.prefill_only:
        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
        print(json.dumps({"prefill": prefill_bench(dev, max(args.prefill_reps, 1))}))
        return

    import paged_kv_decode_append_gb300 as pkv
    from paged_kv_decode_append_gb300 import workloads as wl

    pkv.api._lib.load()
    rank, world, local = dist_setup(args.gpus)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    B, L = args.batch, args.layers
    # layers of one step read different caches: the next layer may stream its
    # K/V while the previous one finishes
    flags = 0 if args.no_overlap else pkv.api.DECODE_OVERLAP_PROLOGUE | pkv.api.DECODE_EARLY_KV
    plan = not args.no_plan
    sweep = Sweep(pkv, wl, args, dev, args.layout, 2 + rank, flags, plan)
    sw = sweep.sw
    steps = timed_decode_steps(args.steps)
    warm_steps = timed_decode_steps(args.warmup)
    stream = torch.cuda.current_stream(dev)

    # The timed region: one CUDA graph per decode step, replayed back to back.
    # It holds the decode kernel's launches (plus, with step plans, one small
    # plan kernel per step that runs beside layer 0), so the decode kernel's
    # average launch duration is the region time over its launches.
    ms, total_bytes, clocks = sweep.timed(warm_steps, steps, world, local)
    n_ev = args.steps * L
    n_launch = n_ev + (args.steps if plan else 0)
    ms_max = max_over_ranks(ms, world, dev)
    all_bytes = sum_over_ranks(float(total_bytes), world, dev)
    value = all_bytes / (ms_max * 1e-3) / 1e9
    launch_bytes = total_bytes / n_ev
    kernel_ms = ms / n_ev
    achieved = launch_bytes / (kernel_ms * 1e-3) / 1e9
    peak, peak_kind = peaks()
    traffic_ratio = recorded_traffic()

    # Diagnostic: each launch alone (plain launch, CUDA events around it) for
    # the first `iso_steps` timed steps, to show the duration of one kernel by itself.
    iso_steps = steps[:min(20, len(steps))]
    iso_ev, iso_bytes = [], []
    for s in iso_steps:
        for layer, (q, kn, vn) in enumerate(sweep.step_inputs(s)):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                sweep.layer_call(s, layer, q, kn, vn, flags=0)
            torch.cuda.synchronize(dev)
            a.record(stream)
            g.replay()
            b.record(stream)
            iso_ev.append((a, b, g))
            iso_bytes.append(call_bytes(sweep.lens_all[s], B))
    torch.cuda.synchronize(dev)
    iso_ms = np.array([a.elapsed_time(b) for a, b, _ in iso_ev])
    iso_gbs = float(np.sum(iso_bytes) / (iso_ms.sum() * 1e-3) / 1e9)
    del iso_ev

    # Without graphs: the same steps as plain stream launches (36 per step).
    eager_steps = steps[:min(20, len(steps))]
    torch.cuda.synchronize(dev)
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    eager_bytes = 0
    ea.record(stream)
    for s in eager_steps:
        for layer, (q, kn, vn) in enumerate(sweep.step_inputs(s)):
            sweep.layer_call(s, layer, q, kn, vn)
        eager_bytes += sweep.step_bytes[s]
    eb.record(stream)
    torch.cuda.synchronize(dev)
    eager_gbs = eager_bytes / (ea.elapsed_time(eb) * 1e-3) / 1e9

    # End to end through the public API: pkv_decode_step graphs (all 36 layers
    # each) captured once over two sets of device input / output buffers.
    # Every step copies that step's q / k_new / v_new of all layers and its
    # cache_seqlens from pinned host memory into one set, launches the graph
    # of that set and copies all its outputs back.  The copies run on their
    # own streams, double-buffered: step s+1's inputs go up while step s
    # computes, step s's outputs come down while step s+1 computes.  The timed
    # region spans the first input copy to the last output copy; the steps are
    # those the device-timed value covers (the first e2e_steps of them).
    e2e_list = steps[:min(args.e2e_steps, len(steps))]
    e2e_steps = len(e2e_list)
    per_layer = [B * HQ * D, B * HKV * D, B * HKV * D]
    layer_elems = sum(per_layer)

    def split(buf, base):
        q_, k_, v_ = torch.split(buf[base:base + layer_elems], per_layer)
        return q_.view(B, HQ, D), k_.view(B, HKV, D), v_.view(B, HKV, D)

    sets = []
    for _ in range(2):
        d_in_all = torch.empty(L * layer_elems, dtype=torch.bfloat16, device=dev)
        d_out_all = torch.empty(L * B * HQ * D, dtype=torch.bfloat16, device=dev)
        d_seq = torch.empty(B, dtype=torch.int32, device=dev)
        d_in = [split(d_in_all, layer * layer_elems) for layer in range(L)]
        d_out = [d_out_all[layer * B * HQ * D:(layer + 1) * B * HQ * D].view(B, HQ, D) for layer in range(L)]
        graph = pkv.DecodeStep(sw.k_caches, sw.v_caches, [t[0] for t in d_in], [t[1] for t in d_in],
                               [t[2] for t in d_in], sweep.bt, d_seq, sw.softmax_scale, d_out, workspace=sweep.ws,
                               flags=flags | (pkv.api.DECODE_USE_PLAN if plan else 0))
        sets.append((d_in_all, d_out_all, d_seq, graph))
    h_in = []
    for r in range(2):  # two pinned input sets, alternated
        h = torch.empty(L * layer_elems, dtype=torch.bfloat16).pin_memory()
        for layer, trip in enumerate(sweep.inputs[r]):
            for dst, t in zip(split(h, layer * layer_elems), trip):
                dst.copy_(t.cpu())
        h_in.append(h)
    h_seq = [torch.as_tensor(sweep.lens_all[s]).pin_memory() for s in e2e_list]
    h_out = [torch.empty(L * B * HQ * D, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = sets[0][0].numel() * 2 + B * 4
    d2h = sets[0][1].numel() * 2
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready = [ev() for _ in range(e2e_steps)]
    done = [ev() for _ in range(e2e_steps)]
    out_read = [ev() for _ in range(e2e_steps)]

    def upload(i):  # step i's inputs into set i % 2, once step i-2 (same set) is read and copied out
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(out_read[i - 2])
            d_in_all, _, d_seq, _ = sets[i % 2]
            d_in_all.copy_(h_in[i % 2], non_blocking=True)
            d_seq.copy_(h_seq[i], non_blocking=True)
            in_ready[i].record(up)

    torch.cuda.synchronize(dev)
    barrier(world)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_bytes = 0
    e_start.record(stream)
    up.wait_stream(stream)
    upload(0)
    for i in range(e2e_steps):
        if i + 1 < e2e_steps:
            upload(i + 1)
        stream.wait_event(in_ready[i])
        sets[i % 2][3].launch()
        done[i].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(done[i])
            h_out[i % 2].copy_(sets[i % 2][1], non_blocking=True)
            out_read[i].record(down)
        e_bytes += sweep.step_bytes[e2e_list[i]]
    stream.wait_stream(down)
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    e_ms = max_over_ranks(e_start.elapsed_time(e_end), world, dev)
    e_all = sum_over_ranks(float(e_bytes), world, dev)
    e2e_value = e_all / (e_ms * 1e-3) / 1e9
    del sets

    prefill = prefill_bench(dev, args.prefill_reps) if args.prefill_reps > 0 else None
    prefill_other = None
    if args.prefill_reps > 0:  # the other prefill kernels on the same lengths
        keep = ("tflops", "frac", "ms_median", "ms_best", "reps", "flops", "workload")
        prefill_other = {f"d{hd}": {k: v for k, v in prefill_bench(dev, args.prefill_reps, hd).items() if k in keep}
                         for hd in (128, 64)}

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(sw, steps)
    del sweep, sw
    torch.cuda.empty_cache()

    contiguous = None
    if not args.no_contiguous:  # the same sweep on sequentially reserved pages
        other = "contiguous" if args.layout == "shuffled" else "shuffled"
        csweep = Sweep(pkv, wl, args, dev, other, 2, flags, plan)
        c_ms, c_bytes, c_clocks = csweep.timed(warm_steps, steps, 1, local)
        c_val = c_bytes / (c_ms * 1e-3) / 1e9
        contiguous = {"layout": other, "value": c_val, "unit": "GB/s", "pct_of_hbm_peak": 100.0 * c_val / peak,
                      "ms_per_step": c_ms / args.steps, "steps": args.steps,
                      "algorithmic_bytes_per_launch": c_bytes / n_ev, "clocks": c_clocks,
                      "gpu_launches": n_launch, "config": workload_config(args, other)}
        del csweep
        torch.cuda.empty_cache()
    single = None
    if args.layer_reps > 0:  # one layer per call: the Qwen3-4B-shaped layer and the skewed batch
        keep = ("value", "unit", "pct_of_hbm_peak", "decode_tok_s_per_attn_layer", "ms_per_step", "ms_best",
                "steps", "config", "algorithmic_bytes_per_call", "clocks", "gpu_launches", "streamed")
        single = {}
        for kind in ("qwen3", "skewed"):
            line = single_layer_bench(kind, args.layer_reps, 3)
            single[kind] = {k: line[k] for k in keep}
    mixed = None
    if args.mixed_reps > 0:  # one mixed step per call: speculative decode and a chunked-prefill step
        keep = ("value", "unit", "pct_of_hbm_peak", "tflops", "pct_of_tensor_peak", "ms_per_step", "ms_best",
                "steps", "config", "algorithmic_bytes_per_call", "flops_per_call", "clocks", "gpu_launches")
        mixed = {}
        for kind in ("spec", "chunked"):
            line = mixed_bench(kind, args.mixed_reps, 3, None, dev)
            mixed[kind] = {k: line[k] for k in keep}
    steps_tok = B / (ms / args.steps / L * 1e-3)  # decode tokens/s per attention layer
    out = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(args),
        "pct_of_hbm_peak": 100.0 * value / peak,
        "decode_tok_s_per_attn_layer": steps_tok * world,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None if traffic_ratio is None else traffic_ratio * launch_bytes,
                     "peak_kind": peak_kind, "kernel": "pkv::decode_kernel<128,4> (layers 1-35 of a step: the instantiation that starts from the step plan)",
                     "algorithmic_bytes_per_launch": launch_bytes, "launch_ms_mean": kernel_ms,
                     "isolated_launch_ms_mean": float(iso_ms.mean()), "isolated_launch_ms_best": float(iso_ms.min()),
                     "isolated_gbs": iso_gbs, "isolated_launches": int(iso_ms.size),
                     "isolated_steps": f"the first {len(iso_steps)} timed decode steps, each launch alone"},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "path": "pkv_decode_step graphs of the 36 layers over two buffer sets; per step pinned H2D of "
                        "all inputs and cache_seqlens, one graph launch, D2H of all outputs; copies on their own "
                        "streams, double-buffered (step s+1's upload and step s-1's download overlap step s)"},
        "eager": {"value": eager_gbs, "unit": "GB/s", "steps": len(eager_steps),
                  "launch": "plain stream launches, no CUDA graph"},
        "gpu_launches": n_launch,
        "launch": "one CUDA graph per decode step (36 decode kernel launches" + (
            "" if args.no_overlap else ", programmatic dependent launch between them, K/V streamed early") + (
            "; layer 0 also launches the step plan kernel and layers 1-35 reuse its plan)" if plan else ")"),
        "cpu_baseline": cpu,
        "contiguous": contiguous,
        "single_layer": single,
        "prefill": prefill,
        "prefill_other": prefill_other,
        "mixed": mixed,
    }
    print(json.dumps(out))


if __name__ == "__main__":
    main()
