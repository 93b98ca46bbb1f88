"""GPU parity of the FP8 (E4M3) KV-cache path against the FP64 oracle with
per-kv-head (and per-tensor) dequantisation scales, and of scaled 16-bit
caches. Calls go through the C ABI (ctypes binding)."""
import pytest
import torch

import oracle
from paged_gqa_decode_attention_gb300 import PDAError, PDA_EUNSUPPORTED, workloads
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


@pytest.mark.parametrize("G,Hkv", [(1, 8), (2, 4), (4, 8), (7, 4), (8, 1), (8, 8), (3, 2)])
@pytest.mark.parametrize("bs", [16, 32])
def test_fp8_geometries_exact(G, Hkv, bs):
    lens = [1, bs + 1, 700, 3000, 64, 129]
    wl = workloads.to_fp8_kv(workloads.custom(seed=G * 11 + Hkv + bs, B=len(lens), Hq=G * Hkv,
                                              Hkv=Hkv, D=128, block_size=bs, lens=lens,
                                              num_blocks=700))
    for splits in (0, 1, 5, 64):
        check(wl, num_splits=splits)


def test_fp8_per_tensor_and_unit_scales():
    base = workloads.custom(seed=3, B=4, Hq=32, Hkv=8, D=128, block_size=16,
                            lens=[900, 17, 2048, 300])
    wl = workloads.to_fp8_kv(base)
    # one scale for the whole tensor (the largest per-head one)
    wl.meta["k_scale"] = wl.meta["k_scale"].max().reshape(1)
    wl.meta["v_scale"] = wl.meta["v_scale"].max().reshape(1)
    check(wl)
    # no scales at all: the raw E4M3 values
    del wl.meta["k_scale"], wl.meta["v_scale"]
    check(wl)


def test_fp8_peaky_rows_and_fp32_out():
    wl = workloads.to_fp8_kv(workloads.mid_ragged(seed=2))
    check(wl)
    err = check(workloads.to_fp8_kv(workloads.mid_ragged(seed=3)), out_dtype=torch.float32)
    assert err < 2e-3, err


def test_fp8_full_size_long_context_every_split_count():
    """The FP8 bench workload (B=8, L=32768, the headline's bytes, random
    tables over a 20 GiB FP8 pool): every row against the oracle on the
    pages those rows read, at every split count of the sweep and the
    heuristic's, and in fp32 output."""
    wl = workloads.long_context(seed=0, batch=8, context=32768, device=DEV, kv_fp8=True)
    ks = wl.meta["k_scale"].double().cpu().numpy()
    vs = wl.meta["v_scale"].double().cpu().numpy()
    q, k, v, bt, cl = workloads.compact_for_rows(wl, range(wl.batch))
    ref = oracle.paged_decode_kv(q, k, v, bt, cl, oracle.BF16, oracle.FP8_E4M3, wl.scale, ks, vs)
    del q, k, v
    attn = make_attn(wl)
    for splits in (0, 1, 2, 4, 8, 16, 32, 64):
        assert_close(run_gpu(attn, wl, num_splits=splits), ref, f"fp8 splits={splits}")
    err = assert_close(run_gpu(attn, wl, out_dtype=torch.float32), ref, "fp8 fp32 out")
    assert err < 2e-3, err
    attn.close()
    del wl
    torch.cuda.empty_cache()


def test_fp8_full_size_group_16():
    """FP8 K/V at 128/8 heads (G = 16) and the headline's bytes (B=8,
    L=32768): every row against the oracle at three split counts and in fp32
    output."""
    wl = workloads.to_fp8_kv(workloads.custom(seed=8, B=8, Hq=128, Hkv=8, D=128, block_size=16,
                                              lens=[32768] * 8, device=DEV))
    ks = wl.meta["k_scale"].double().cpu().numpy()
    vs = wl.meta["v_scale"].double().cpu().numpy()
    q, k, v, bt, cl = workloads.compact_for_rows(wl, range(wl.batch))
    ref = oracle.paged_decode_kv(q, k, v, bt, cl, oracle.BF16, oracle.FP8_E4M3, wl.scale, ks, vs)
    del q, k, v
    attn = make_attn(wl)
    for splits in (0, 7, 64):
        assert_close(run_gpu(attn, wl, num_splits=splits), ref, f"fp8 g16 splits={splits}")
    err = assert_close(run_gpu(attn, wl, out_dtype=torch.float32), ref, "fp8 g16 fp32 out")
    assert err < 2e-3, err
    attn.close()
    del wl
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,Hq,Hkv,L", [(16, 32, 8, 32768), (128, 14, 2, 8192)])
def test_fp8_full_size_head_dim_64(B, Hq, Hkv, L):
    """FP8 K/V at head dim 64 at full size: the bench's 32/8-head step (B=16,
    L=32768, the headline's bytes) and the Qwen2.5-0.5B geometry (14/2 heads,
    B=128, L=8192): every row against the oracle at the heuristic's split count
    and one other, and in fp32 output."""
    wl = workloads.to_fp8_kv(workloads.custom(seed=Hq + B, B=B, Hq=Hq, Hkv=Hkv, D=64,
                                              block_size=16, lens=[L] * B, device=DEV))
    ks = wl.meta["k_scale"].double().cpu().numpy()
    vs = wl.meta["v_scale"].double().cpu().numpy()
    q, k, v, bt, cl = workloads.compact_for_rows(wl, range(wl.batch))
    ref = oracle.paged_decode_kv(q, k, v, bt, cl, oracle.BF16, oracle.FP8_E4M3, wl.scale, ks, vs)
    del q, k, v
    attn = make_attn(wl)
    for splits in (0, 5):
        assert_close(run_gpu(attn, wl, num_splits=splits), ref, f"fp8 d64 splits={splits}")
    err = assert_close(run_gpu(attn, wl, out_dtype=torch.float32), ref, "fp8 d64 fp32 out")
    assert err < 2e-3, err
    attn.close()
    del wl
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kernel", ["cuda_core", "tensor_core"])
def test_scaled_16bit_caches(kernel, monkeypatch):
    """Dequantisation scales on bf16 caches (both kernels)."""
    monkeypatch.setenv("PDA_PARTIAL_KERNEL", kernel)
    wl = workloads.custom(seed=9, B=3, Hq=32, Hkv=8, D=128, block_size=16, lens=[500, 64, 2000])
    g = torch.Generator().manual_seed(0)
    wl.meta["k_scale"] = torch.rand(8, generator=g) * 2 + 0.25
    wl.meta["v_scale"] = torch.rand(8, generator=g) * 2 + 0.25
    check(wl)
    check(wl, num_splits=7)


@pytest.mark.parametrize("G,Hkv", [(4, 8), (7, 2), (8, 1), (1, 8)])
@pytest.mark.parametrize("bs", [16, 32])
def test_fp8_fp16_queries_exact(G, Hkv, bs):
    """FP8 K/V with fp16 queries (and fp16 output): the q tile is split into
    its two fp8 terms from fp16, per-kv-head scales, every split count."""
    lens = [1, bs + 1, 700, 3000, 64, 129]
    wl = workloads.to_fp8_kv(workloads.custom(seed=G * 13 + Hkv + bs, B=len(lens), Hq=G * Hkv,
                                              Hkv=Hkv, D=128, block_size=bs, lens=lens,
                                              dtype="fp16", num_blocks=700))
    assert wl.q.dtype == torch.float16
    for splits in (0, 1, 5, 64):
        check(wl, num_splits=splits)
    err = check(wl, out_dtype=torch.float32)
    assert err < 2e-3, err


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (14, 2), (8, 8), (16, 2), (6, 2)])
@pytest.mark.parametrize("bs", [16, 32])
def test_fp8_head_dim_64_exact(Hq, Hkv, bs):
    """FP8 K/V at head dim 64 (64-byte swizzled rows, M = 64 PV): the
    Qwen2.5-0.5B layout (14/2 heads) and other group sizes, both block sizes,
    every split count, bf16 and fp16 queries, fp32 output."""
    lens = [1, bs + 1, 700, 3000, 64, 129]
    wl = workloads.to_fp8_kv(workloads.custom(seed=Hq * 5 + Hkv + bs, B=len(lens), Hq=Hq,
                                              Hkv=Hkv, D=64, block_size=bs, lens=lens,
                                              num_blocks=700))
    for splits in (0, 1, 5, 64):
        check(wl, num_splits=splits)
    err = check(wl, out_dtype=torch.float32)
    assert err < 2e-3, err
    wl16 = workloads.to_fp8_kv(workloads.custom(seed=Hq + bs, B=3, Hq=Hq, Hkv=Hkv, D=64,
                                                block_size=bs, lens=[500, 64, 2000],
                                                dtype="fp16"))
    check(wl16)
    check(wl16, num_splits=7)


@pytest.mark.parametrize("Hq,Hkv,D", [(128, 8, 128), (64, 4, 64), (9, 1, 128), (28, 2, 64)])
@pytest.mark.parametrize("bs", [16, 32])
def test_fp8_large_groups_exact(Hq, Hkv, D, bs):
    """FP8 K/V with group sizes 9..16 (up to all 16 MMA columns), bf16 and fp16
    queries, every split count, fp32 output."""
    lens = [1, bs + 1, 700, 3000, 64, 129]
    wl = workloads.to_fp8_kv(workloads.custom(seed=Hq * 11 + Hkv + D + bs, B=len(lens), Hq=Hq,
                                              Hkv=Hkv, D=D, block_size=bs, lens=lens,
                                              num_blocks=700))
    for splits in (0, 1, 5, 64):
        check(wl, num_splits=splits)
    err = check(wl, out_dtype=torch.float32)
    assert err < 2e-3, err
    wl16 = workloads.to_fp8_kv(workloads.custom(seed=Hq + bs + 1, B=3, Hq=Hq, Hkv=Hkv, D=D,
                                                block_size=bs, lens=[500, 64, 2000],
                                                dtype="fp16"))
    check(wl16)
    check(wl16, num_splits=7)


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (14, 2, 64), (64, 8, 128)])
def test_fp8_block_size_64(Hq, Hkv, D):
    """FP8 K/V in 64-token pages: every split count, fp16 queries, fp32 output."""
    lens = [1, 63, 64, 65, 700, 3000, 129]
    wl = workloads.to_fp8_kv(workloads.custom(seed=Hq * 3 + D, B=len(lens), Hq=Hq, Hkv=Hkv,
                                              D=D, block_size=64, lens=lens, num_blocks=200))
    for splits in (0, 1, 5, 64):
        check(wl, num_splits=splits)
    err = check(wl, out_dtype=torch.float32)
    assert err < 2e-3, err
    check(workloads.to_fp8_kv(workloads.custom(seed=Hq + 5, B=3, Hq=Hq, Hkv=Hkv, D=D,
                                               block_size=64, lens=[500, 64, 2000],
                                               dtype="fp16")))


def test_fp8_unsupported_geometries_rejected():
    from paged_gqa_decode_attention_gb300 import PagedDecodeAttention
    for kw in (dict(head_dim=256), dict(num_q_heads=8 * 17)):
        args = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                    dtype=torch.bfloat16)
        args.update(kw)
        with pytest.raises(PDAError) as e:
            PagedDecodeAttention(**args, kv_fp8=True)
        assert e.value.status == PDA_EUNSUPPORTED
