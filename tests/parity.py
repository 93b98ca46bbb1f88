"""Shared helpers for the GPU parity tests.

Tolerance (the stated bar is a max abs error of 2e-3 for bf16/fp16 outputs
with fp32 accumulation). Rounding the exact result to bf16 alone moves it by
up to half an output ulp, which is 0.0039 at |out| in [1, 2): an exact
implementation could fail a flat 2e-3. So:
  - fp32 outputs (the kernel's own accuracy) must be within 2e-3 of FP64;
  - bf16/fp16 outputs must be within 2e-3 + half an ulp of the output
    dtype at the FP64 value.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_gqa_decode_attention_gb300 import PagedDecodeAttention, workloads

ABS_TOL = 2e-3


def half_ulp(ref: np.ndarray, dtype_name: str) -> np.ndarray:
    mant = 7 if dtype_name == "bf16" else 10
    emin = -126 if dtype_name == "bf16" else -14
    e = np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** emin)))
    return 0.5 * np.exp2(e - mant)


def assert_close(out: torch.Tensor, ref: np.ndarray, what: str = "") -> float:
    """Compare a GPU output with the FP64 oracle under the tolerance above;
    returns the max abs error."""
    got = out.detach().double().cpu().numpy()
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    if out.dtype == torch.float32:
        tol = ABS_TOL
    else:
        tol = ABS_TOL + half_ulp(ref, "bf16" if out.dtype == torch.bfloat16 else "fp16")
    bad = err > tol
    if bad.any():
        idx = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond tolerance; worst at "
                             f"{idx}: got {got[idx]!r} want {ref[idx]!r} (max err {err.max():.3e})")
    return float(err.max())


def oracle_ref(wl: workloads.Workload) -> np.ndarray:
    dt = oracle.BF16 if wl.q.dtype == torch.bfloat16 else oracle.FP16
    if wl.kv_fp8 or "k_scale" in wl.meta:
        q, k, v, bt, cl = workloads.host_arrays(wl)
        ks = wl.meta.get("k_scale")
        vs = wl.meta.get("v_scale")
        return oracle.paged_decode_kv(
            q, k, v, bt, cl, dt, oracle.FP8_E4M3 if wl.kv_fp8 else dt, wl.scale,
            None if ks is None else ks.double().cpu().numpy().repeat(
                wl.num_kv_heads // ks.numel()),
            None if vs is None else vs.double().cpu().numpy().repeat(
                wl.num_kv_heads // vs.numel()))
    return oracle.paged_decode(*workloads.host_arrays(wl), dt, wl.scale)


def make_attn(wl: workloads.Workload, max_splits: int = 64, max_batch: int | None = None,
              max_blocks: int | None = None) -> PagedDecodeAttention:
    return PagedDecodeAttention(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                                wl.q.dtype, max_batch=max_batch or max(1, wl.batch),
                                max_blocks_per_seq=max_blocks or wl.max_blocks,
                                max_splits=max_splits, device=torch.cuda.current_device(),
                                kv_fp8=wl.kv_fp8)


def run_gpu(attn: PagedDecodeAttention, wl: workloads.Workload, **kw) -> torch.Tensor:
    kw.setdefault("k_scale", wl.meta.get("k_scale"))
    kw.setdefault("v_scale", wl.meta.get("v_scale"))
    out = attn.run(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.context_lens, wl.scale, **kw)
    torch.cuda.synchronize()
    return out
