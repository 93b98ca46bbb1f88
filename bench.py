#!/usr/bin/env python
"""Benchmark of the paged GQA decode-attention hot path on GB300.

One step = one decode-attention call (the whole hot path: split plan, the
split-K partial kernel with its log-sum-exp merge) over one batch of seeded
synthetic inputs already resident in HBM. Default workload: the long-context
split-K case B=4, Hq 32, Hkv 8, D 128, block 16, context 32768, random
block tables over a 40 GiB K+V pool (512 MiB of KV read per step, 4x the L2,
so consecutive steps do not hit in L2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

Prints one JSON line (rank 0). Under torchrun each rank runs its own batch
(seed + rank) with no data-path collective (weak scaling); the timed region
is bracketed by a barrier and a device synchronize on both sides and the
time is the max over ranks. ``--impl reference`` times the FP64 CPU oracle on
the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "decode tokens/s and KV-read HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0

NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (~8 TB/s)

# DRAM bytes (read + write) per launch from one ncu capture of the workload's
# kernel, and the SHA-256 of the kernel sources that capture ran on. When the
# sources no longer hash to that value the figure is stale and the bench
# reports null traffic.
_CSRC = os.path.join(ROOT, "paged_gqa_decode_attention_gb300", "csrc")
TC_KERNEL_SOURCES = ("partial_tc_kernel.cuh", "ptx.cuh", "split_merge.cuh", "pda_internal.h",
                     "partial_tc_bf16_d128.cu", "partial_launch.cu")
ROPE_KERNEL_SOURCES = ("rope_kv_write.cu", "ptx.cuh", "pda_internal.h")
NCU_TRAFFIC = {
    # workload: (bytes per launch, kernel sources, their SHA-256 at capture)
    "long_b4_l32768": (540_981_760, TC_KERNEL_SOURCES,
                       "9d54b0a72658dbd1b0ed990de896a3e78228f88ebff1598f7b029366fd744473"),
    "rope_prefill_t32768": (768_234_496, ROPE_KERNEL_SOURCES,
                            "fa980a506c38f4a633447bab730832813569500c8a40c5ee3795b4ff6925ceb9"),
}


def sources_digest(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(_CSRC, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def ncu_traffic(workload: str):
    """(bytes per launch or None, note)."""
    entry = NCU_TRAFFIC.get(workload)
    if entry is None:
        return None, "no ncu capture for this workload"
    nbytes, files, digest = entry
    if nbytes is None or digest is None or sources_digest(files) != digest:
        return None, "kernel sources changed since the last ncu capture"
    return nbytes, "ncu dram__bytes_read.sum + dram__bytes_write.sum per launch"


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def make_workload(name: str, seed: int, device):
    from paged_gqa_decode_attention_gb300 import workloads as W
    if name == "long_b4_l32768":
        return W.long_context(seed=seed, batch=4, context=32768, device=device)
    if name == "long_b4_l32768_pool1g":  # same step over a 1 GiB pool (for ncu captures)
        return W.long_context(seed=seed, batch=4, context=32768, num_blocks=16384, device=device)
    if name == "long_b4_l32768_fp8":  # the headline step with an FP8 (E4M3) K/V cache
        return W.long_context(seed=seed, batch=4, context=32768, device=device, kv_fp8=True)
    if name == "long_b8_l32768_fp8":  # FP8 cache, the headline's KV bytes per step
        return W.long_context(seed=seed, batch=8, context=32768, device=device, kv_fp8=True)
    if name == "long_b8_l32768_fp8_pool1g":  # same step over a 1 GiB FP8 pool (for ncu captures)
        return W.long_context(seed=seed, batch=8, context=32768, num_blocks=32768, device=device,
                              kv_fp8=True)
    if name == "long_b1_l32768":
        return W.long_context(seed=seed, batch=1, context=32768, device=device)
    if name == "long_b4_l8192":
        return W.long_context(seed=seed, batch=4, context=8192, device=device)
    if name == "long_b1_l8192":
        return W.long_context(seed=seed, batch=1, context=8192, device=device)
    if name == "long_b4_l32768_bs32":  # same step with 32-token pages (40 GiB pool)
        return W.custom(seed=seed, B=4, Hq=32, Hkv=8, D=128, block_size=32, lens=[32768] * 4,
                        num_blocks=327680, device=device)
    if name == "long_b32_l32768_mqa4":  # same bytes and G as long_b4_l32768, one kv head
        return W.custom(seed=seed, B=32, Hq=4, Hkv=1, D=128, block_size=16, lens=[32768] * 32,
                        num_blocks=4 * 65536, device=device)
    # other GQA geometries (random pages over exactly the pool they need)
    if name == "geo_qwen05b_b64_l8192":  # Qwen2.5-0.5B attention: 14/2 heads, D 64
        return W.custom(seed=seed, B=64, Hq=14, Hkv=2, D=64, block_size=16, lens=[8192] * 64,
                        device=device)
    if name == "geo_qwen7b_b16_l8192":  # Qwen2.5-7B attention: 28/4 heads, D 128 (G = 7)
        return W.custom(seed=seed, B=16, Hq=28, Hkv=4, D=128, block_size=16, lens=[8192] * 16,
                        device=device)
    if name == "geo_d256_b16_l8192":  # 16/8 heads, D 256 (G = 2)
        return W.custom(seed=seed, B=16, Hq=16, Hkv=8, D=256, block_size=16, lens=[8192] * 16,
                        device=device)
    # the headline's bytes (B x L x 8 kv heads) at other group sizes / head dims
    if name == "geo_g1_b4_l32768":  # 8/8 heads (G = 1), D 128
        return W.custom(seed=seed, B=4, Hq=8, Hkv=8, D=128, block_size=16, lens=[32768] * 4,
                        device=device)
    if name == "geo_g2_b4_l32768":  # 16/8 heads (G = 2), D 128
        return W.custom(seed=seed, B=4, Hq=16, Hkv=8, D=128, block_size=16, lens=[32768] * 4,
                        device=device)
    if name == "geo_g8_b4_l32768":  # 64/8 heads (G = 8), D 128
        return W.custom(seed=seed, B=4, Hq=64, Hkv=8, D=128, block_size=16, lens=[32768] * 4,
                        device=device)
    if name == "geo_d64_b8_l32768":  # 32/8 heads, D 64 (B = 8: the same bytes)
        return W.custom(seed=seed, B=8, Hq=32, Hkv=8, D=64, block_size=16, lens=[32768] * 8,
                        device=device)
    if name == "geo_fp8_d64_b16_l32768":  # FP8 cache, 32/8 heads, D 64 (the headline's bytes)
        return W.to_fp8_kv(W.custom(seed=seed, B=16, Hq=32, Hkv=8, D=64, block_size=16,
                                    lens=[32768] * 16, device=device))
    if name == "long_b4_l32768_g16":  # 128/8 heads (G = 16: all 16 MMA columns), the headline's bytes
        return W.custom(seed=seed, B=4, Hq=128, Hkv=8, D=128, block_size=16, lens=[32768] * 4,
                        device=device)
    if name == "long_b8_l32768_fp8_g16":  # FP8 cache, 128/8 heads
        return W.to_fp8_kv(W.custom(seed=seed, B=8, Hq=128, Hkv=8, D=128, block_size=16,
                                    lens=[32768] * 8, device=device))
    if name == "long_b8_l32768_fp8_g8":  # FP8 cache, 64/8 heads
        return W.to_fp8_kv(W.custom(seed=seed, B=8, Hq=64, Hkv=8, D=128, block_size=16,
                                    lens=[32768] * 8, device=device))
    if name == "geo_mqa_b64_l8192":  # MQA: 8 query heads on one kv head, D 128
        return W.custom(seed=seed, B=64, Hq=8, Hkv=1, D=128, block_size=16, lens=[8192] * 64,
                        device=device)
    if name == "serving_b128":
        return W.serving_mix(seed=seed, batch=128, device=device)
    if name == "mid_ragged_b8":
        return W.mid_ragged(seed=seed, device=device)
    if name == "short_b32":
        return W.short_batch(seed=seed, device=device)
    raise SystemExit(f"unknown workload {name}")


WORKLOAD_DESC = {
    "long_b4_l32768": "long-context split-K: B=4, Hq 32, Hkv 8, D 128, block 16, context 32768, "
                      "bf16 N(0,1), random block tables over a 40 GiB K+V pool",
}

# RoPE + paged-KV write workloads: the Qwen2.5-0.5B attention geometry
# (14/2 heads, D 64, theta 1e6) at 1-512 new decode tokens, and a 32768-token
# prefill at 32/8/128 that is large enough to measure HBM bandwidth.
ROPE_WORKLOADS = {
    "rope_qwen05b_t1": dict(tokens=1),
    "rope_qwen05b_t32": dict(tokens=32),
    "rope_qwen05b_t512": dict(tokens=512),
    "rope_prefill_t32768": dict(tokens=32768, Hq=32, Hkv=8, D=128, theta=10000.0,
                                mode="prefill"),
}
ROPE_METRIC = "RoPE + paged-KV write tokens/s and HBM GB/s (% of GB300 peak), 1 GPU"

# KV-cache movement workloads (32/8/128 bf16 caches, block 16, 40 GiB pool):
# gather the headline step's 4 x 32768 tokens into contiguous rows; copy
# 4096 random blocks to other blocks; scatter 32768 rows into random slots.
MOVE_WORKLOADS = ("move_gather_b4_l32768", "move_copy_blocks_4096", "move_scatter_t32768")
MOVE_METRIC = "KV-cache movement GB/s moved (read + write, % of GB300 peak), 1 GPU"


# ---------------------------------------------------------------------------
# distributed helpers (weak scaling, no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def shard_seed(base_seed: int, rank: int) -> int:
    """Each rank decodes its own batch of sequences."""
    return base_seed + 1000 * rank


def reduce_max(x: float, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region (NVML through ctypes; read-only)
# ---------------------------------------------------------------------------

_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """Polls SM clock and clock-event reasons every ``period`` seconds in a
    thread while the timed region runs."""

    def __init__(self, uuid: str | None, period: float = 0.002):
        self.period = period
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._nvml = None
        self._dev = None
        try:
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if nvml.nvmlInit_v2() != 0:
                return
            dev = ctypes.c_void_p()
            ok = -1
            if uuid:
                ok = nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(dev))
            if ok != 0:
                ok = nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(dev))
            if ok != 0:
                return
            mx = ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._nvml, self._dev = nvml, dev
        except OSError:
            pass

    def _reasons(self) -> int:
        r = ctypes.c_ulonglong()
        fn = getattr(self._nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self._nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        return r.value if fn(self._dev, ctypes.byref(r)) == 0 else 0

    def _run(self):
        mhz = ctypes.c_uint()
        while not self._stop.is_set():
            if self._nvml.nvmlDeviceGetClockInfo(self._dev, 1, ctypes.byref(mhz)) == 0:
                self.samples.append((mhz.value, self._reasons()))
            time.sleep(self.period)

    def __enter__(self):
        self._stop.clear()
        if self._nvml is not None:
            self._thr = threading.Thread(target=self._run, daemon=True)
            self._thr.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._nvml is not None:
            self._thr.join()

    def summary(self) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "note": "NVML unavailable"}
        mhz = [m for m, _ in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        reasons = sorted({name for b, name in _REASONS.items() if bits & b})
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples)}


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# CPU baseline: the FP64 oracle on a bounded sample
# ---------------------------------------------------------------------------

def _oracle_rows(wl, q, k, v, bt, cl, rows, threads):
    """The oracle on rows (b, hq) of host arrays from compact_for_rows."""
    import oracle
    dt = oracle.BF16 if wl.q.dtype == torch.bfloat16 else oracle.FP16
    if wl.kv_fp8 or "k_scale" in wl.meta:
        ks, vs = wl.meta.get("k_scale"), wl.meta.get("v_scale")
        return oracle.paged_decode_kv(
            q, k, v, bt, cl, dt, oracle.FP8_E4M3 if wl.kv_fp8 else dt, wl.scale,
            None if ks is None else ks.double().cpu().numpy(),
            None if vs is None else vs.double().cpu().numpy(), rows=rows, threads=threads)
    return oracle.paged_decode_rows(q, k, v, bt, cl, dt, wl.scale, rows, threads=threads)


def oracle_sample(wl, target_s: float = 10.0):
    """Time the FP64 oracle on whole sequences of ``wl`` (all query heads of
    every sequence, passes repeated until about ``target_s`` of wall time).
    Returns (tokens_per_s, sample_description, threads, seconds)."""
    import oracle
    from paged_gqa_decode_attention_gb300 import workloads as W
    threads = os.cpu_count() or 1
    dt = oracle.BF16 if wl.q.dtype == torch.bfloat16 else oracle.FP16
    q, k, v, bt, cl = W.compact_for_rows(wl, list(range(wl.batch)))
    rows = np.array([[b, h] for b in range(q.shape[0]) for h in range(q.shape[1])],
                    dtype=np.int32)
    passes, elapsed = 0, 0.0
    while elapsed < target_s and passes < 1000:
        t0 = time.perf_counter()
        _oracle_rows(wl, q, k, v, bt, cl, rows, threads)
        elapsed += time.perf_counter() - t0
        passes += 1
    seqs = passes * q.shape[0]
    desc = (f"{passes} pass(es) over all {q.shape[0]} sequences x {q.shape[1]} query heads "
            f"({int(cl.sum())} tokens per pass) of the same workload; oracle over {threads} "
            f"threads")
    return seqs / elapsed, desc, threads, elapsed


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    if dev.type == "cpu" and args.workload.startswith("long_"):
        # without a GPU, draw the same shapes over a pool just large enough
        from paged_gqa_decode_attention_gb300 import workloads as W
        B = 8 if "_b8_" in args.workload else (4 if "_b4_" in args.workload else 1)
        L = int(args.workload.split("_l")[-1].split("_")[0])
        wl = W.long_context(seed=args.seed, batch=B, context=L,
                            num_blocks=B * (L // 16) + 64, kv_fp8="fp8" in args.workload)
    else:
        wl = make_workload(args.workload, args.seed, dev)
    import oracle
    from paged_gqa_decode_attention_gb300 import workloads as W
    threads = os.cpu_count() or 1
    dt = oracle.BF16 if wl.q.dtype == torch.bfloat16 else oracle.FP16
    q, k, v, bt, cl = W.compact_for_rows(wl, [0])
    rows = np.array([[0, h] for h in range(q.shape[1])], dtype=np.int32)
    for _ in range(args.warmup):
        _oracle_rows(wl, q, k, v, bt, cl, rows, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_rows(wl, q, k, v, bt, cl, rows, threads)
    el = time.perf_counter() - t0
    value = args.steps / el  # one sequence (all query heads) per step
    sample = (f"per step: sequence 0 (all {q.shape[1]} query heads, {int(cl[0])} tokens) of "
              f"the {args.workload} workload")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "desc": WORKLOAD_DESC.get(args.workload, "")},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def back_to_back_samples(step, dev, samples: int = 7, launches: int = 200) -> list[float]:
    """Per-launch device time (ms) of ``samples`` replays of one CUDA graph of
    ``launches`` calls, CUDA events on the replay stream around each replay
    (consecutive calls overlap their set-up with the previous call's tail)."""
    stream = torch.cuda.current_stream(dev)
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for _ in range(launches):
            step()
    graph.replay()
    torch.cuda.synchronize(dev)
    out = []
    for _ in range(samples):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        out.append(e0.elapsed_time(e1) / launches)
    del graph
    return out


def cold_calls(step, dev, calls: int = 30) -> list[float]:
    """Device time (ms) of ``calls`` single calls, each preceded by an L2
    flush (a write of twice the L2 size, then a read of another such buffer so
    the dirty lines drain before the call), CUDA events around each call on
    the launching stream."""
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    wbuf = torch.empty(2 * max(l2, 1 << 27), dtype=torch.uint8, device=dev)
    rbuf = torch.empty(2 * max(l2, 1 << 27) // 4, dtype=torch.int32, device=dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(calls)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(calls)]
    for i in range(calls):
        wbuf.zero_()
        rbuf.max()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


def sample_summary(ms: list[float], nbytes: int, peak: float, **extra) -> dict:
    med = statistics.median(ms)
    return {**extra, "per_call_ms_median": med, "per_call_ms_min": min(ms),
            "per_call_ms_max": max(ms), "kv_gbs_median": nbytes / (med / 1e3) / 1e9,
            "frac_of_measured_median": nbytes / (med / 1e3) / 1e9 / peak,
            "frac_of_nominal_median": nbytes / (med / 1e3) / 1e9 / NOMINAL_HBM_GBS}


def partial_kernel_label(wl) -> str:
    """Which partial kernel the library runs for this geometry: tensor cores
    for FP8 K/V and for groups of 3..8 at head dim 64/128, CUDA cores
    otherwise (PDA_PARTIAL_KERNEL overrides)."""
    env = os.environ.get("PDA_PARTIAL_KERNEL", "")
    G = wl.num_q_heads // wl.num_kv_heads
    tc = env == "tensor_core" or (env != "cuda_core" and (
        wl.kv_fp8 or (3 <= G <= 8 and wl.head_dim in (64, 128))))
    return ("paged_partial_tc_kernel (tcgen05 split-K partials + fused LSE merge)" if tc else
            "paged_partial_kernel (CUDA-core split-K partials + fused LSE merge)")


def e2e_graph(attn, wl, out, args, ksc, vsc, dev, world):
    """End-to-end tokens/s through the public API with host-resident inputs
    and output: per step one graph (H2D copy of the packed inputs, run, D2H
    copy of out) and a host wait. Falls back to separate copies on the stream
    if graph capture is unavailable. Returns (mode, tokens/s, h2d, d2h)."""
    B = wl.batch
    parts = [wl.q, wl.block_table, wl.context_lens]
    sizes = [t.numel() * t.element_size() for t in parts]
    offs, o = [], 0
    for n in sizes:
        offs.append(o)
        o += (n + 255) // 256 * 256  # keep every view 256-byte aligned
    in_h = torch.empty(o, dtype=torch.uint8).pin_memory()
    in_d = torch.empty(o, dtype=torch.uint8, device=dev)

    def view(buf, i):
        t = parts[i]
        return buf[offs[i]:offs[i] + sizes[i]].view(t.dtype).view(t.shape)

    for i, t in enumerate(parts):
        view(in_h, i).copy_(t.cpu())
    q_d, bt_d, cl_d = view(in_d, 0), view(in_d, 1), view(in_d, 2)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(sizes)
    d2h = out_h.numel() * out_h.element_size()

    def step():
        in_d.copy_(in_h, non_blocking=True)
        attn.run(q_d, wl.k_cache, wl.v_cache, bt_d, cl_d, wl.scale, out=out,
                 num_splits=args.splits, k_scale=ksc, v_scale=vsc)
        out_h.copy_(out, non_blocking=True)

    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    mode = "graph per step: packed H2D copy + run + D2H copy, host wait each step"
    g = None
    try:
        with torch.cuda.stream(s):
            step()
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                step()
        s.synchronize()
    except RuntimeError as exc:  # capture unavailable: same work, submitted op by op
        g = None
        mode = f"stream per step (graph capture failed: {str(exc).splitlines()[0][:80]})"
        torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    with torch.cuda.stream(s):
        for _ in range(args.steps):
            if g is not None:
                g.replay()
            else:
                step()
            s.synchronize()
    e2e_s = reduce_max(time.perf_counter() - t0, dev)
    # the host read back the last step's output: it must be the device's
    if not torch.equal(out_h.view(torch.uint8), out.cpu().view(torch.uint8)):  # bit for bit
        raise RuntimeError("end-to-end output copy does not match the device output")
    return mode, B * world * args.steps / e2e_s, h2d, d2h


def run_ours(args):
    world, rank, local = dist_env()
    import torch.distributed as dist
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)

    from paged_gqa_decode_attention_gb300 import PagedDecodeAttention
    from paged_gqa_decode_attention_gb300 import build as pda_build
    pda_build.build()

    wl = make_workload(args.workload, shard_seed(args.seed, rank), dev)
    B, Hq, D = wl.batch, wl.num_q_heads, wl.head_dim
    attn = PagedDecodeAttention(Hq, wl.num_kv_heads, D, wl.block_size, wl.q.dtype,
                                max_batch=B, max_blocks_per_seq=wl.max_blocks, max_splits=64,
                                device=dev, kv_fp8=wl.kv_fp8)
    ksc, vsc = wl.meta.get("k_scale"), wl.meta.get("v_scale")
    out = torch.empty((B, Hq, D), dtype=wl.q.dtype, device=dev)
    kv_bytes = wl.kv_bytes()
    launch = attn.launch_shape(B, wl.max_blocks, num_splits=args.splits)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    # Inputs of at least twice the L2 size evict each other between steps. For
    # smaller ones the L2 is flushed between steps: a write of a buffer larger
    # than L2, then a read of a second one so that the dirty lines are written
    # back before (not during) the next timed step.
    flush = kv_bytes < 2 * l2
    flush_buf = torch.empty(2 * max(l2, 1 << 27), dtype=torch.uint8, device=dev) if flush else None
    flush_read = torch.empty(2 * max(l2, 1 << 27) // 4, dtype=torch.int32, device=dev) if flush else None
    stream = torch.cuda.current_stream(dev)

    def step():
        attn.run(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.context_lens, wl.scale, out=out,
                 num_splits=args.splits, k_scale=ksc, v_scale=vsc)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)

    # ---- timed region: K steps, inputs resident in HBM ----
    # graph timing (default when no L2 flush is needed): the K calls are
    # captured as CUDA graphs of n_inner calls and replayed back to back, so
    # host-side launch cost cannot leave the GPU idle between steps; one call
    # is one kernel launch, so K / region time is the per-launch duration.
    # eager timing (with L2 flushes): one call per step, CUDA events around
    # each call on the launching stream.
    use_graph = (args.timing == "graph") or (args.timing == "auto" and not flush)
    region0, region1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    if use_graph:
        n_inner = max(d for d in range(1, min(args.steps, 100) + 1) if args.steps % d == 0)
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(n_inner):
                step()
        torch.cuda.synchronize(dev)
        graph.replay()  # warm replay
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        with sampler:
            cpu0 = time.perf_counter()
            region0.record(stream)
            for _ in range(args.steps // n_inner):
                graph.replay()
            region1.record(stream)
            cpu_submit = time.perf_counter() - cpu0
            torch.cuda.synchronize(dev)
        barrier()
        timed_ms = region0.elapsed_time(region1)
        avg_launch_ms = timed_ms / args.steps
        timing_desc = f"CUDA graph of {n_inner} calls replayed {args.steps // n_inner}x"
    else:
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier()
        torch.cuda.synchronize(dev)
        with sampler:
            cpu0 = time.perf_counter()
            region0.record(stream)
            for i in range(args.steps):
                if flush:
                    flush_buf.zero_()
                    flush_read.max()
                starts[i].record(stream)
                step()
                ends[i].record(stream)
            region1.record(stream)
            cpu_submit = time.perf_counter() - cpu0
            torch.cuda.synchronize(dev)
        barrier()
        kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        # with L2 flushing between steps the flush is not part of a step
        timed_ms = sum(kernel_ms) if flush else region0.elapsed_time(region1)
        avg_launch_ms = statistics.mean(kernel_ms)
        timing_desc = "eager calls, CUDA events around each call"
    print(f"[bench] timed {timed_ms:.3f} ms for {args.steps} steps; host submit "
          f"{1e3 * cpu_submit:.3f} ms; {timing_desc}", file=sys.stderr)
    timed_ms_max = reduce_max(timed_ms, dev)

    # ---- repeated samples of the same step, outside the K-step region ----
    # back to back: 7 replays of a 200-call graph; cold: single calls after an
    # L2 flush. The clock sampler keeps running across both.
    with sampler:
        b2b_ms = back_to_back_samples(step, dev)
        cold_ms = cold_calls(step, dev)
    value = (B * world * args.steps) / (timed_ms_max / 1e3)

    # ---- end to end: host buffers, copies inside the timed region ----
    # The step's inputs (q, block_table, context_lens) sit in one pinned host
    # buffer and go to the device in one copy; copy in, run and copy out are
    # submitted as one CUDA graph per step, and the host waits for the result
    # every step. (A serving loop writes the next step's inputs into the same
    # pinned buffer before each replay.)
    e2e_mode, e2e_value, h2d, d2h = e2e_graph(attn, wl, out, args, ksc, vsc, dev, world)

    peak, peak_kind = measured_peaks()
    achieved = kv_bytes / (avg_launch_ms / 1e3) / 1e9
    traffic, traffic_note = ncu_traffic(args.workload)
    unique_bytes = wl.unique_kv_bytes()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": timed_ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 q / fp8-e4m3 kv" if wl.kv_fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "desc": WORKLOAD_DESC.get(args.workload, ""),
                   "batch_per_gpu": B, "global_batch": B * world,
                   "kv_bytes_per_step": kv_bytes,
                   "unique_kv_bytes_per_step": unique_bytes,
                   "l2": "inputs larger than L2 (KV per step >= 2x L2, no flush)" if not flush
                   else ("L2 flushed between steps (write + read of 2x L2, outside the step "
                         "events)" if not use_graph else
                         "graph replay without flush: KV per step < 2x L2, partly L2-resident"),
                   "launch": launch,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "timing": timing_desc},
        "kv_gbs": achieved,
        "kv_frac_of_peak": achieved / peak,
        "kv_frac_of_nominal": achieved / NOMINAL_HBM_GBS,
        "samples": {
            "back_to_back": sample_summary(b2b_ms, kv_bytes, peak, samples=len(b2b_ms),
                                           launches_per_sample=200),
            "cold": sample_summary(cold_ms, kv_bytes, peak, calls=len(cold_ms),
                                   l2="flushed before each call"),
        },
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "traffic_source": traffic_note,
                     "peak_source": f"{peak_kind} (hbm_gbs)",
                     "kernel": partial_kernel_label(wl),
                     "per_launch_ms": avg_launch_ms,
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "nominal_peak": NOMINAL_HBM_GBS},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "mode": e2e_mode},
        "gpu_launches": args.steps * launches_per_step(attn, wl),
        "clocks": sampler.summary(),
    }
    if unique_bytes != kv_bytes:
        # shared prefix pages: bytes of the distinct slots read (aliased pages
        # may be served from L2 for all but their first reader)
        line["kv_gbs_unique"] = unique_bytes / (avg_launch_ms / 1e3) / 1e9
        line["kv_frac_of_peak_unique"] = line["kv_gbs_unique"] / peak
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc, cores, secs = oracle_sample(wl)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": secs}
    if rank == 0:
        print(json.dumps(line), flush=True)
    attn.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_split_sweep(args):
    """The long-context split-count sweep: B in {1, 4} x L in {8192, 32768}
    cut from one full-size pool (random tables over 40 GiB; FP8 workloads use
    B in {1, 8} over the 20 GiB FP8 pool), every split count in 1..64 plus the
    planner's pick. Per (shape, S) one JSON line with the cold per-call time
    (L2 flushed before each call) and the back-to-back time (graph replay)."""
    from paged_gqa_decode_attention_gb300 import PagedDecodeAttention, make_config, plan
    from paged_gqa_decode_attention_gb300 import build as pda_build
    from paged_gqa_decode_attention_gb300 import workloads as W
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    dev = torch.device("cuda", torch.cuda.current_device())
    pda_build.build()
    fp8 = "fp8" in args.workload
    big = 8 if fp8 else 4
    pool = W.long_context(seed=args.seed, batch=big, context=32768, device=dev, kv_fp8=fp8)
    peak, _ = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ksc, vsc = pool.meta.get("k_scale"), pool.meta.get("v_scale")
    for B, L in ((1, 8192), (big, 8192), (1, 32768), (big, 32768)):
        wl = W.leading(pool, B, L)
        attn = PagedDecodeAttention(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                                    wl.q.dtype, max_batch=B, max_blocks_per_seq=wl.max_blocks,
                                    max_splits=64, device=dev, kv_fp8=fp8)
        cfg = make_config(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                          wl.q.dtype, max_batch=B, max_blocks_per_seq=wl.max_blocks,
                          max_splits=64, device=dev.index, kv_fp8=fp8)
        picked = plan(cfg, sms, B, wl.max_blocks)[0]
        out = torch.empty_like(wl.q)
        for S in sorted({1, 2, 4, 8, 16, 32, 64, picked}):
            def step(S=S):
                attn.run(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.context_lens,
                         wl.scale, out=out, num_splits=S, k_scale=ksc, v_scale=vsc)
            for _ in range(max(3, args.warmup)):
                step()
            torch.cuda.synchronize(dev)
            cold = sample_summary(cold_calls(step, dev, 20), wl.kv_bytes(), peak, calls=20)
            b2b = sample_summary(back_to_back_samples(step, dev, 5, 100), wl.kv_bytes(), peak,
                                 samples=5, launches_per_sample=100)
            print(json.dumps({"workload": wl.name, "batch": B, "context": L, "splits": S,
                              "planner_pick": S == picked, "kv_bytes": wl.kv_bytes(),
                              "launch": attn.launch_shape(B, wl.max_blocks, num_splits=S),
                              "cold": cold, "back_to_back": b2b}), flush=True)
        attn.close()
    return 0


def launches_per_step(attn, wl) -> int:
    """Kernels one call launches: the partial kernel, which also merges the
    splits (the last split of each sequence's kv head does it)."""
    return 1


def rope_oracle_sample(wl, target_s: float = 5.0):
    """Time the FP64 oracle on the first <= 4096 tokens of a RoPE workload,
    repeated until about ``target_s``. Returns (tokens_per_s, description)."""
    import oracle
    n = min(wl.num_tokens, 4096)

    def b(t):
        return t[:n].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

    args = (b(wl.q), b(wl.k), b(wl.v), wl.positions[:n].cpu().numpy(),
            wl.slot_mapping[:n].cpu().numpy(), wl.cos_sin.cpu().numpy(), wl.rot_dim, wl.neox,
            oracle.BF16 if wl.qkv.dtype == torch.bfloat16 else oracle.FP16,
            wl.k_cache.cpu().view(torch.int16).numpy().view(np.uint16),
            wl.v_cache.cpu().view(torch.int16).numpy().view(np.uint16))
    passes, elapsed = 0, 0.0
    while elapsed < target_s and passes < 10000:
        t0 = time.perf_counter()
        oracle.rope_kv_write(*args)
        elapsed += time.perf_counter() - t0
        passes += 1
    return passes * n / elapsed, f"{passes} pass(es) over {n} tokens of the workload; 1 thread"


def run_rope(args):
    """One step = one RoPE + paged-KV write call over the workload's tokens."""
    from paged_gqa_decode_attention_gb300 import build as pda_build
    from paged_gqa_decode_attention_gb300 import rope_kv_write
    from paged_gqa_decode_attention_gb300 import workloads as W
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    spec = ROPE_WORKLOADS[args.workload]
    if args.impl == "reference":
        wl = W.rope_batch(seed=args.seed, **spec)
        v, desc = rope_oracle_sample(wl, target_s=max(1.0, 0.2 * args.steps))
        line = {"impl": "reference", "metric": ROPE_METRIC, "value": v, "unit": "tokens/s",
                "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * wl.num_tokens / v, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": args.workload, **spec},
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0
    dev = torch.device("cuda", torch.cuda.current_device())
    pda_build.build()
    wl = W.rope_batch(seed=args.seed, device=dev, **spec)
    T = wl.num_tokens
    q_out = torch.empty((T, wl.num_q_heads, wl.head_dim), dtype=wl.qkv.dtype, device=dev)
    stream = torch.cuda.current_stream(dev)
    moved = wl.moved_bytes()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    # small calls: L2 flushed between eager calls (cold), unless --timing graph
    # asks for back-to-back graph replay (L2-warm, as right after the QKV
    # projection that produces the inputs)
    flush = moved < 2 * l2 and args.timing != "graph"
    flush_buf = torch.empty(2 * max(l2, 1 << 27), dtype=torch.uint8, device=dev) if flush else None
    flush_read = torch.empty(2 * max(l2, 1 << 27) // 4, dtype=torch.int32, device=dev) if flush else None

    def step(qkv=None):
        src = wl if qkv is None else qkv
        rope_kv_write(src.q, src.k, src.v, wl.positions, wl.slot_mapping, wl.cos_sin,
                      wl.k_cache, wl.v_cache, neox=wl.neox, q_out=q_out)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if flush:
        with sampler:
            for i in range(args.steps):
                flush_buf.zero_()
                flush_read.max()
                starts[i].record(stream)
                step()
                ends[i].record(stream)
            torch.cuda.synchronize(dev)
        per_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        timed_ms = sum(per_ms)
        timing_desc = "eager calls, CUDA events around each call, L2 flushed between calls"
    else:
        n_inner = max(d for d in range(1, min(args.steps, 100) + 1) if args.steps % d == 0)
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(n_inner):
                step()
        graph.replay()
        torch.cuda.synchronize(dev)
        with sampler:
            starts[0].record(stream)
            for _ in range(args.steps // n_inner):
                graph.replay()
            ends[0].record(stream)
            torch.cuda.synchronize(dev)
        timed_ms = starts[0].elapsed_time(ends[0])
        per_ms = [timed_ms / args.steps]
        timing_desc = f"CUDA graph of {n_inner} calls replayed {args.steps // n_inner}x"
    avg_ms = statistics.mean(per_ms)
    value = T * args.steps / (timed_ms / 1e3)
    # end to end: fused qkv projection output from pinned host memory, q_out back
    qkv_h = wl.qkv.cpu().pin_memory()
    pos_h = wl.positions.cpu().pin_memory()
    slot_h = wl.slot_mapping.cpu().pin_memory()
    out_h = torch.empty(q_out.shape, dtype=q_out.dtype).pin_memory()
    qkv_d = torch.empty_like(wl.qkv)
    e2e_wl = W.RopeWorkload(wl.name, qkv_d, wl.positions, wl.slot_mapping, wl.cos_sin,
                            wl.k_cache, wl.v_cache, wl.num_q_heads, wl.num_kv_heads,
                            wl.head_dim, wl.neox)
    h2d = qkv_h.numel() * qkv_h.element_size() + pos_h.numel() * 4 + slot_h.numel() * 8
    d2h = out_h.numel() * out_h.element_size()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        qkv_d.copy_(qkv_h, non_blocking=True)
        wl.positions.copy_(pos_h, non_blocking=True)
        wl.slot_mapping.copy_(slot_h, non_blocking=True)
        step(e2e_wl)
        out_h.copy_(q_out, non_blocking=True)
        stream.synchronize()
    e2e_value = T * args.steps / (time.perf_counter() - t0)
    peak, peak_kind = measured_peaks()
    achieved = moved / (avg_ms / 1e3) / 1e9
    line = {
        "metric": ROPE_METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": timed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, **spec, "bytes_per_step": moved,
                   "l2": "L2 flushed between calls" if flush else
                   ("inputs larger than L2 (>= 2x L2 per step, no flush)" if moved >= 2 * l2
                    else "L2-warm: graph replay, no flush"),
                   "timing": timing_desc},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": ncu_traffic(args.workload)[0],
                     "traffic_source": ncu_traffic(args.workload)[1],
                     "peak_source": f"{peak_kind} (hbm_gbs)",
                     "kernel": "rope_kv_write_kernel", "per_launch_ms": avg_ms},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(),
    }
    if not args.no_cpu_baseline:
        v, desc = rope_oracle_sample(wl)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line), flush=True)
    return 0


def run_move(args):
    """One step = one KV-cache movement call (gather, block copy or scatter)."""
    from paged_gqa_decode_attention_gb300 import build as pda_build
    from paged_gqa_decode_attention_gb300 import copy_blocks, gather_kv, scatter_kv
    from paged_gqa_decode_attention_gb300 import workloads as W
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    dev = torch.device("cuda", torch.cuda.current_device())
    pda_build.build()
    wl = W.long_context(seed=args.seed, batch=4, context=32768, device=dev)
    nb, bs = wl.k_cache.shape[0], wl.block_size
    row_bytes = wl.num_kv_heads * wl.head_dim * 2
    rng = np.random.default_rng(args.seed)
    if args.workload == "move_gather_b4_l32768":
        lens = wl.context_lens
        cu = (torch.cumsum(lens.to(torch.int64), 0) - lens.to(torch.int64))
        total = int(lens.sum())
        ko = torch.empty((total, wl.num_kv_heads, wl.head_dim), dtype=torch.bfloat16, device=dev)
        vo = torch.empty_like(ko)
        max_len = int(lens.max())

        def step():
            gather_kv(wl.k_cache, wl.v_cache, wl.block_table, lens, cu, max_len, ko, vo)
        units, unit, moved = total, "tokens/s", 2 * 2 * total * row_bytes
    elif args.workload == "move_copy_blocks_4096":
        perm = rng.permutation(nb)[: 2 * 4096].reshape(4096, 2)
        pairs = torch.from_numpy(perm.astype(np.int64)).to(dev)

        def step():
            copy_blocks(wl.k_cache, wl.v_cache, pairs)
        units, unit, moved = 4096, "blocks/s", 2 * 2 * 4096 * bs * row_bytes
    else:
        n = 32768
        rows_k = torch.randn((n, wl.num_kv_heads, wl.head_dim), device=dev).to(torch.bfloat16)
        rows_v = torch.randn_like(rows_k)
        slots = torch.from_numpy(rng.permutation(nb * bs)[:n].astype(np.int64)).to(dev)

        def step():
            scatter_kv(rows_k, rows_v, slots, wl.k_cache, wl.v_cache)
        units, unit, moved = n, "tokens/s", 2 * 2 * n * row_bytes
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    n_inner = max(d for d in range(1, min(args.steps, 100) + 1) if args.steps % d == 0)
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for _ in range(n_inner):
            step()
    graph.replay()
    torch.cuda.synchronize(dev)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with sampler:
        e0.record(stream)
        for _ in range(args.steps // n_inner):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / args.steps
    peak, peak_kind = measured_peaks()
    achieved = moved / (ms / 1e3) / 1e9
    line = {
        "metric": MOVE_METRIC, "value": units / (ms / 1e3), "unit": unit, "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bytes",
        "data": "synthetic",
        "config": {"workload": args.workload, "bytes_moved_per_step": moved,
                   "l2": "inputs larger than L2 (>= 2x L2 per step, no flush)",
                   "timing": f"CUDA graph of {n_inner} calls replayed {args.steps // n_inner}x"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_kind} (hbm_gbs)", "per_launch_ms": ms},
        "gpu_launches": args.steps, "clocks": sampler.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_b4_l32768")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--timing", choices=["auto", "graph", "eager"], default="auto")
    ap.add_argument("--splits", type=int, default=0, help="split count (0 = the planner's)")
    ap.add_argument("--sweep", action="store_true",
                    help="long-context split-count sweep (one JSON line per shape and count)")
    args = ap.parse_args(argv)
    if args.sweep:
        return run_split_sweep(args)
    if args.workload in ROPE_WORKLOADS:
        return run_rope(args)
    if args.workload in MOVE_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "KV-cache movement has no timed oracle arm (byte copies)"}))
            return 0
        return run_move(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
