"""GPU parity: the CUDA path against the FP64 oracle, element by element, on
seeded inputs of every workload family, the split-count sweep, edge cases,
and sampled rows of the full-size long-context workload. Calls go through
the C ABI (ctypes binding)."""
import hashlib

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_attention_gb300 import (PDA_EALIAS, PDA_EINVAL, PagedDecodeAttention,
                                              PDAError, merge, workloads)
from parity import assert_close, make_attn, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda", torch.cuda.current_device())


def check(wl_host, **kw):
    wl = wl_host.to(DEV)
    attn = make_attn(wl)
    out = run_gpu(attn, wl, **kw)
    attn.close()
    return assert_close(out, oracle_ref(wl_host), wl.name)


def test_tiny():
    check(workloads.tiny(seed=0))


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_short_batch(seed, bs, dtype):
    check(workloads.short_batch(seed=seed, block_size=bs, dtype=dtype))


def test_short_and_long_calls_alternate_on_one_handle():
    """Small calls (here: contexts up to 256 tokens, 6 MB of K/V) run on the
    CUDA-core kernel, larger ones on the tensor cores, chosen per call; both
    use the handle's split tickets and the persistent kernel's counters, so
    calls of the two kinds alternate on one handle, each compared with the
    oracle."""
    short = workloads.custom(seed=31, B=6, Hq=32, Hkv=8, D=128, block_size=16,
                             lens=[1, 17, 64, 200, 256, 129], num_blocks=300)
    long_ = workloads.custom(seed=32, B=6, Hq=32, Hkv=8, D=128, block_size=16,
                             lens=[3000, 5, 700, 257, 1, 2048], num_blocks=600)
    assert short.max_blocks * short.block_size <= 256 < long_.max_blocks * long_.block_size
    refs = [oracle_ref(short), oracle_ref(long_)]
    wls = [short.to(DEV), long_.to(DEV)]
    attn = make_attn(wls[1])
    for _ in range(2):
        for wl, ref in zip(wls, refs):
            for splits in (0, 3):
                assert_close(run_gpu(attn, wl, num_splits=splits), ref, f"{wl.name} S={splits}")
    assert attn.check_device_error() == (0, 0)
    attn.close()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_mid_ragged_peaky(seed):
    check(workloads.mid_ragged(seed=seed))


@pytest.mark.parametrize("splits", [1, 2, 3, 4, 5, 8, 16, 32, 64])
def test_long_split_sweep(splits):
    """Every split count gives the same result (ragged 3000-token tail)."""
    wl = workloads.long_context(seed=1, batch=2, context=3000, num_blocks=1024)
    check(wl, num_splits=splits)


@pytest.mark.parametrize("batch,context", [(1, 8192), (4, 8192)])
def test_long_context_heuristic(batch, context):
    check(workloads.long_context(seed=2, batch=batch, context=context, num_blocks=4096))


@pytest.mark.parametrize("batch", [16, 128])
def test_serving_mix(batch):
    check(workloads.serving_mix(seed=0, batch=batch))


def test_fp32_output_mode():
    """The kernel's own accuracy: fp32 out within 2e-3 of FP64 (peaky rows)."""
    err = check(workloads.mid_ragged(seed=0), out_dtype=torch.float32)
    assert err < 1e-4, err  # fp32 accumulation is far inside the bar


@pytest.mark.parametrize("G,Hkv", [(1, 8), (2, 4), (4, 2), (8, 1), (8, 8), (4, 8)])
@pytest.mark.parametrize("bs", [16, 32])
def test_edge_lengths_and_groups(G, Hkv, bs):
    lens = [1, bs - 1, bs, bs + 1, 2 * bs, 63, 64, 65, 0, 257, 1000]
    wl = workloads.custom(seed=G * 10 + Hkv, B=len(lens), Hq=G * Hkv, Hkv=Hkv, D=128,
                          block_size=bs, lens=lens, num_blocks=200)
    for splits in (0, 3, 64):
        check(wl, num_splits=splits)


def test_context_hint_below_actual_is_still_exact():
    wl = workloads.custom(seed=5, B=3, Hq=32, Hkv=8, D=128, block_size=16, lens=[900, 40, 2000])
    check(wl, max_context_len_hint=64)


# The long-context split-K shapes at full size (B in {1, 4} x L in {8192,
# 32768}, random tables over the 40 GiB pool), every split count the sweep
# covers plus the heuristic's (0), every row against the oracle.
LONG_SPLITS = [0, 1, 2, 4, 8, 16, 32, 64]


@pytest.fixture(scope="module")
def long_pool():
    wl = workloads.long_context(seed=0, batch=4, context=32768, device=DEV)
    yield wl
    del wl
    torch.cuda.empty_cache()


@pytest.mark.parametrize("batch,context", [(1, 8192), (4, 8192), (1, 32768), (4, 32768)])
def test_full_size_long_context_every_split_count(long_pool, batch, context):
    wl = workloads.leading(long_pool, batch, context)
    ref = oracle.paged_decode(*workloads.compact_for_rows(wl, range(batch)), oracle.BF16,
                              wl.scale)
    attn = make_attn(wl)
    for splits in LONG_SPLITS:
        out = run_gpu(attn, wl, num_splits=splits)
        assert_close(out, ref, f"{wl.name} splits={splits}")
    err = assert_close(run_gpu(attn, wl, out_dtype=torch.float32), ref, f"{wl.name} fp32 out")
    assert err < 1e-4, err
    attn.close()


def test_full_size_group_16_every_split_count():
    """128/8 heads (G = 16: all 16 MMA columns) at the headline's bytes (B=4,
    L=32768): every row against the oracle at the heuristic's split count and
    across the sweep, and in fp32 output."""
    wl = workloads.custom(seed=7, B=4, Hq=128, Hkv=8, D=128, block_size=16, lens=[32768] * 4,
                          device=DEV)
    ref = oracle.paged_decode(*workloads.compact_for_rows(wl, range(wl.batch)), oracle.BF16,
                              wl.scale)
    attn = make_attn(wl)
    for splits in (0, 1, 4, 16, 64):
        assert_close(run_gpu(attn, wl, num_splits=splits), ref, f"{wl.name} splits={splits}")
    err = assert_close(run_gpu(attn, wl, out_dtype=torch.float32), ref, f"{wl.name} fp32 out")
    assert err < 1e-4, err
    attn.close()
    del wl
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,Hq,Hkv,D,L", [(8, 32, 8, 64, 32768), (64, 14, 2, 64, 8192),
                                          (16, 28, 4, 128, 8192), (64, 8, 1, 128, 8192)])
def test_full_size_other_geometries(B, Hq, Hkv, D, L):
    """The other geometries' bench workloads at full size: 32/8 heads at D 64
    (two producer and two PV warps), Qwen2.5-0.5B (14/2, D 64) and
    Qwen2.5-7B (28/4) attention, MQA (8/1); every row against the oracle at
    the heuristic's split count and one other, and in fp32 output."""
    wl = workloads.custom(seed=Hq + D, B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=16, lens=[L] * B,
                          device=DEV)
    ref = oracle.paged_decode(*workloads.compact_for_rows(wl, range(wl.batch)), oracle.BF16,
                              wl.scale)
    attn = make_attn(wl)
    for splits in (0, 5):
        assert_close(run_gpu(attn, wl, num_splits=splits), ref, f"{wl.name} splits={splits}")
    err = assert_close(run_gpu(attn, wl, out_dtype=torch.float32), ref, f"{wl.name} fp32 out")
    assert err < 1e-4, err
    attn.close()
    del wl
    torch.cuda.empty_cache()


def test_fp32_output_mode_every_config():
    """The kernel's own accuracy (fp32 out) on the tiny, short-batch (both
    dtypes, both block sizes), mid-ragged and serving-mix configs: within the
    flat 2e-3 bar, and in fact below 1e-4."""
    cases = [workloads.tiny(seed=0), workloads.mid_ragged(seed=2),
             workloads.serving_mix(seed=2, batch=128)]
    cases += [workloads.short_batch(seed=5, block_size=bs, dtype=dt)
              for bs in (16, 32) for dt in ("bf16", "fp16")]
    for wl in cases:
        err = check(wl, out_dtype=torch.float32)
        assert err < 1e-4, (wl.name, err)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_merge_entry_point(out_dtype):
    rng = np.random.default_rng(3)
    rows, S, D = 37, 13, 128
    o = rng.standard_normal((rows, S, D))
    lse = rng.standard_normal((rows, S)) * 5
    lse[rng.random((rows, S)) < 0.3] = -np.inf
    lse[5, :] = -np.inf  # a row of empty splits
    o32 = torch.from_numpy(o.astype(np.float32))
    l32 = torch.from_numpy(lse.astype(np.float32))
    ref = oracle.lse_merge(l32.double().numpy(), o32.double().numpy())
    out = merge(o32.to(DEV), l32.to(DEV), out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert_close(out, ref, "merge")
    assert not out[5].any()


def _digest(t):
    return hashlib.sha256(t.detach().contiguous().view(torch.uint8).cpu().numpy().tobytes()).hexdigest()


def test_inputs_unchanged_only_out_written():
    wl = workloads.mid_ragged(seed=1).to(DEV)
    before = [_digest(t) for t in (wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.context_lens)]
    attn = make_attn(wl)
    n = wl.batch * wl.num_q_heads * wl.head_dim
    buf = torch.full((n + 4096,), 7.0, dtype=torch.bfloat16, device=DEV)
    out = buf[:n].view(wl.batch, wl.num_q_heads, wl.head_dim)
    attn.run(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.context_lens, wl.scale, out=out)
    torch.cuda.synchronize()
    after = [_digest(t) for t in (wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.context_lens)]
    assert before == after
    assert bool((buf[n:] == 7.0).all())  # nothing written past out
    attn.close()


def test_handle_reuse_across_workloads():
    a = workloads.custom(seed=7, B=4, Hq=32, Hkv=8, D=128, block_size=16, lens=[100, 2000, 5, 64])
    b = workloads.custom(seed=8, B=2, Hq=32, Hkv=8, D=128, block_size=16, lens=[3000, 17],
                         num_blocks=300)
    attn = PagedDecodeAttention(32, 8, 128, 16, torch.bfloat16, max_batch=8,
                                max_blocks_per_seq=256, max_splits=64)
    for wl_host in (a, b, a):
        wl = wl_host.to(DEV)
        assert_close(run_gpu(attn, wl), oracle_ref(wl_host), wl.name)
    attn.close()


def test_cuda_graph_capture_replay():
    wl = workloads.long_context(seed=3, batch=2, context=2500, num_blocks=512).to(DEV)
    attn = make_attn(wl)
    eager = run_gpu(attn, wl).clone()
    out = torch.empty_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        attn.run(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.context_lens, wl.scale, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    attn.close()


def test_validator_flags_without_faulting():
    wl = workloads.custom(seed=9, B=3, Hq=32, Hkv=8, D=128, block_size=16, lens=[40, 17, 90]).to(DEV)
    attn = make_attn(wl)
    attn.validate(wl.block_table, wl.context_lens, wl.num_blocks)
    assert attn.check_device_error() == (0, 0)
    lens = wl.context_lens.clone()
    lens[1] = wl.max_blocks * 16 + 1
    attn.validate(wl.block_table, lens, wl.num_blocks)
    assert attn.check_device_error() == (1, 1)
    table = wl.block_table.clone()
    table[2, 3] = wl.num_blocks + 5
    attn.validate(table, wl.context_lens, wl.num_blocks)
    assert attn.check_device_error() == (2, 2)
    # the kernel itself stays memory-safe on the bad table: the bad page reads zeros
    out = attn.run(wl.q, wl.k_cache, wl.v_cache, table, wl.context_lens, wl.scale)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    assert attn.check_device_error() == (0, 0)
    attn.close()


def test_abi_errors_on_gpu():
    wl = workloads.tiny(seed=0).to(DEV)
    attn = make_attn(wl)
    with pytest.raises(PDAError) as e:
        attn.run(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.context_lens, wl.scale,
                 out=wl.q)
    assert e.value.status == PDA_EALIAS
    lib = attn.lib
    bad = wl.q.data_ptr() + 2  # misaligned
    st = attn.run_raw(bad, wl.k_cache.data_ptr(), wl.v_cache.data_ptr(), wl.block_table.data_ptr(),
                      wl.context_lens.data_ptr(), 1, wl.max_blocks, wl.num_blocks, wl.scale,
                      torch.empty_like(wl.q).data_ptr())
    assert st == PDA_EINVAL and b"aligned" in lib.paged_decode_attn_last_error()
    st = attn.run_raw(wl.q.data_ptr(), wl.k_cache.data_ptr(), wl.v_cache.data_ptr(),
                      wl.block_table.data_ptr(), wl.context_lens.data_ptr(), 2, wl.max_blocks,
                      wl.num_blocks, wl.scale, torch.empty_like(wl.q).data_ptr())
    assert st == PDA_EINVAL  # batch > max_batch
    # batch 0 is a no-op
    assert attn.run_raw(0, 0, 0, 0, 0, 0, 1, 1, 1.0, 0) == 0
    attn.close()


KERNELS = ["cuda_core", "tensor_core"]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("G,Hkv", [(4, 8), (8, 8), (4, 2), (8, 1)])
@pytest.mark.parametrize("bs", [16, 32])
def test_both_partial_kernels_exact(kernel, G, Hkv, bs, monkeypatch):
    """Both implementations of the partial kernel (CUDA cores; tcgen05 tensor
    cores) are exact on ragged lengths, block sizes 16/32, with and without
    splitting."""
    monkeypatch.setenv("PDA_PARTIAL_KERNEL", kernel)
    wl = workloads.custom(seed=21 + G + bs, B=5, Hq=G * Hkv, Hkv=Hkv, D=128, block_size=bs,
                          lens=[3000, 1, 129, 700, 128], num_blocks=400)
    for splits in (0, 1, 5, 64):
        check(wl, num_splits=splits)


@pytest.mark.parametrize("kernel", KERNELS)
def test_both_partial_kernels_peaky_and_fp16(kernel, monkeypatch):
    monkeypatch.setenv("PDA_PARTIAL_KERNEL", kernel)
    check(workloads.mid_ragged(seed=4))
    check(workloads.short_batch(seed=4, block_size=32, dtype="fp16"))
    check(workloads.serving_mix(seed=1, batch=24))
    err = check(workloads.mid_ragged(seed=5), out_dtype=torch.float32)
    assert err < 1e-4, err


# Other GQA geometries: the Qwen2.5 layouts (14/2 and 28/4 heads: G = 7), odd
# group sizes 3, 5, 6, MQA (Hkv = 1), head dims 64 and 256.
GEOMETRIES = [(14, 2, 64), (28, 4, 128), (12, 2, 128), (40, 8, 128), (24, 8, 128), (7, 1, 128),
              (16, 8, 256), (32, 8, 256), (6, 2, 256), (4, 1, 256), (8, 8, 64), (4, 1, 64),
              (32, 4, 64), (10, 2, 64)]


@pytest.mark.parametrize("Hq,Hkv,D", GEOMETRIES)
@pytest.mark.parametrize("bs", [16, 32])
def test_geometries_exact(Hq, Hkv, D, bs):
    lens = [1, bs + 1, 700, 3000, 64, 129]
    wl = workloads.custom(seed=Hq * 7 + Hkv + D + bs, B=len(lens), Hq=Hq, Hkv=Hkv, D=D,
                          block_size=bs, lens=lens, num_blocks=600)
    for splits in (0, 1, 5, 64):
        check(wl, num_splits=splits)


# Group sizes 9..16 (tensor-core kernel only: the group fills up to all 16
# MMA columns): 128/8 and 64/4 heads (G 16), 96/8 (G 12), 28/2 at D 64
# (G 14), 72/8 (G 9), MQA with 11 query heads, 60/4 (G 15).
LARGE_GROUPS = [(128, 8, 128), (64, 4, 64), (96, 8, 128), (28, 2, 64), (72, 8, 128), (11, 1, 128),
                (60, 4, 64), (40, 4, 128)]


@pytest.mark.parametrize("Hq,Hkv,D", LARGE_GROUPS)
@pytest.mark.parametrize("bs", [16, 32])
def test_large_groups_exact(Hq, Hkv, D, bs):
    lens = [1, bs + 1, 700, 3000, 64, 129]
    wl = workloads.custom(seed=Hq * 3 + Hkv + D + bs, B=len(lens), Hq=Hq, Hkv=Hkv, D=D,
                          block_size=bs, lens=lens, num_blocks=600)
    for splits in (0, 1, 5, 64):
        check(wl, num_splits=splits)


@pytest.mark.parametrize("Hq,Hkv,D", [(128, 8, 128), (28, 2, 64), (72, 8, 128)])
def test_large_groups_fp16_and_fp32_out(Hq, Hkv, D):
    lens = [900, 17, 2048, 300]
    wl = workloads.custom(seed=D + Hq + 5, B=4, Hq=Hq, Hkv=Hkv, D=D, block_size=16, lens=lens,
                          dtype="fp16", num_blocks=300)
    check(wl)
    check(wl, num_splits=3)
    wl = workloads.custom(seed=D + Hq + 6, B=4, Hq=Hq, Hkv=Hkv, D=D, block_size=32, lens=lens)
    err = check(wl, out_dtype=torch.float32)
    assert err < 1e-4, err


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (14, 2, 64), (8, 1, 128), (64, 8, 128),
                                      (16, 8, 128), (16, 8, 256)])
def test_block_size_64(kernel, Hq, Hkv, D, monkeypatch):
    """64-token pages (two per tensor-core chunk, one per CUDA-core stage) on
    both kernels where each supports the geometry: ragged and partial last
    pages, every split count, fp16 inputs and fp32 output."""
    G = Hq // Hkv
    if kernel == "tensor_core" and (G < 3 or D == 256):
        pytest.skip("tensor-core kernel: G 3..16 at head dim 64 or 128")
    monkeypatch.setenv("PDA_PARTIAL_KERNEL", kernel)
    lens = [1, 63, 64, 65, 700, 3000, 129]
    wl = workloads.custom(seed=Hq + D + 64, B=len(lens), Hq=Hq, Hkv=Hkv, D=D, block_size=64,
                          lens=lens, num_blocks=200)
    for splits in (0, 1, 5, 64):
        check(wl, num_splits=splits)
    check(workloads.custom(seed=Hq + D + 65, B=3, Hq=Hq, Hkv=Hkv, D=D, block_size=64,
                           lens=[500, 64, 2000], dtype="fp16"))
    err = check(workloads.custom(seed=Hq + D + 66, B=3, Hq=Hq, Hkv=Hkv, D=D, block_size=64,
                                 lens=[500, 64, 2000]), out_dtype=torch.float32)
    assert err < 1e-4, err


@pytest.mark.parametrize("Hq,Hkv,D", [(14, 2, 64), (16, 8, 256), (28, 4, 128)])
def test_geometries_fp16_and_fp32_out(Hq, Hkv, D):
    lens = [900, 17, 2048, 300]
    wl = workloads.custom(seed=D + Hq, B=4, Hq=Hq, Hkv=Hkv, D=D, block_size=16, lens=lens,
                          dtype="fp16", num_blocks=300)
    check(wl)
    wl = workloads.custom(seed=D + Hq + 1, B=4, Hq=Hq, Hkv=Hkv, D=D, block_size=32, lens=lens)
    err = check(wl, out_dtype=torch.float32)
    assert err < 1e-4, err


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("Hq,Hkv,D", [(14, 2, 64), (28, 4, 128), (24, 8, 128), (40, 8, 128),
                                      (12, 2, 64), (32, 4, 64), (16, 4, 64), (9, 3, 64)])
def test_both_kernels_on_padded_groups(kernel, Hq, Hkv, D, monkeypatch):
    """Group sizes 3..8 at head dims 64 and 128 on both implementations (the
    tensor-core kernel pads the group to 16 MMA columns; at D = 64 it runs a
    64-deep QK^T and an M = 64 PV, with two producer warps per ring at G <= 4)."""
    monkeypatch.setenv("PDA_PARTIAL_KERNEL", kernel)
    lens = [3000, 1, 129, 700, 128, 17]
    for bs in (16, 32):
        wl = workloads.custom(seed=Hq + Hkv + D + bs, B=len(lens), Hq=Hq, Hkv=Hkv, D=D,
                              block_size=bs, lens=lens, num_blocks=700)
        for splits in (0, 1, 5, 64):
            check(wl, num_splits=splits)
    wl = workloads.custom(seed=D, B=3, Hq=Hq, Hkv=Hkv, D=D, block_size=16, lens=[500, 64, 2000],
                          dtype="fp16")
    check(wl)
    err = check(workloads.custom(seed=D + 1, B=3, Hq=Hq, Hkv=Hkv, D=D, block_size=16,
                                 lens=[500, 64, 2000]), out_dtype=torch.float32)
    assert err < 1e-4, err


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (32, 8, 64)])
def test_timed_out_call_reports_and_next_call_is_exact(Hq, Hkv, D, monkeypatch):
    """Failure detection without a GPU fault. PDA_TEST_STALL_RUNS=1 (read when
    the handle is created) makes the handle's first run publish no work unit
    and shortens every pipeline wait to 1 ms: no page load, MMA or store is
    ever issued, so the waits run out with nothing in flight. That run
    records error code 3; the next run of the same handle, with no
    check_device_error in between, is exact (the timed-out CTAs still counted
    themselves done, so the work counters were reset); the error word reports
    the timeout and is clear after the next exact run. Both producer
    layouts of the tensor-core kernel (one and two producer warps per ring)."""
    monkeypatch.setenv("PDA_PARTIAL_KERNEL", "tensor_core")
    monkeypatch.setenv("PDA_TEST_STALL_RUNS", "1")
    wl_host = workloads.custom(seed=D + 3, B=3, Hq=Hq, Hkv=Hkv, D=D, block_size=16,
                               lens=[3000, 17, 900], num_blocks=400)
    ref = oracle_ref(wl_host)
    wl = wl_host.to(DEV)
    attn = make_attn(wl)
    monkeypatch.delenv("PDA_TEST_STALL_RUNS")
    run_gpu(attn, wl, num_splits=4)  # stalled: nothing is written
    assert_close(run_gpu(attn, wl, num_splits=4), ref, "first run after a timed-out run")
    code, _ = attn.check_device_error()
    assert code == 3
    assert_close(run_gpu(attn, wl), ref, "heuristic splits after the error was read")
    assert attn.check_device_error() == (0, 0)
    attn.close()


@pytest.mark.parametrize("cluster", ["1", "0"])
@pytest.mark.parametrize("Hq,Hkv,D,bs", [(8, 1, 128, 16), (14, 2, 64, 32), (32, 8, 128, 16),
                                         (128, 8, 128, 16)])
def test_split_merge_paths(cluster, Hq, Hkv, D, bs, monkeypatch):
    """The splits of a (sequence, kv head) merge either inside one
    thread-block cluster through distributed shared memory (split counts 2..16
    when every (sequence, kv head) pair fits in one wave of clusters) or
    through the workspace and the split tickets (PDA_CLUSTER_MERGE=0, and
    whenever the pairs do not fit). Both are exact, including sequences
    shorter than the split count (empty splits inside a cluster), in 16-bit
    and fp32 output."""
    monkeypatch.setenv("PDA_CLUSTER_MERGE", cluster)
    lens = [1, bs + 1, 700, 3000, 4000, 129]
    wl = workloads.custom(seed=Hq + D + bs, B=len(lens), Hq=Hq, Hkv=Hkv, D=D, block_size=bs,
                          lens=lens, num_blocks=700)
    attn = make_attn(wl)
    shapes = {S: attn.launch_shape(wl.batch, wl.max_blocks, num_splits=S)
              for S in (2, 3, 5, 8, 13, 16)}
    attn.close()
    # pairs of 2 CTAs always fit one wave at these batch sizes
    assert shapes[2]["cluster"] == (2 if cluster == "1" else 1), shapes[2]
    for S, sh in shapes.items():
        assert sh["splits"] == S and sh["cluster"] in (1, S), sh
    for splits in (2, 3, 5, 8, 13, 16):
        check(wl, num_splits=splits)
    err = check(wl, num_splits=16, out_dtype=torch.float32)
    assert err < 1e-4, err
    err = check(wl, num_splits=4, out_dtype=torch.float32)
    assert err < 1e-4, err
