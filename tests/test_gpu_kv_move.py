"""GPU parity of the KV-cache movement calls (block copy, gather, scatter,
table remap) against the oracle: byte-exact, on bf16 and FP8 caches, with
out-of-range ids flagged and skipped. Calls go through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_attention_gb300 import (PagedDecodeAttention, copy_blocks, gather_kv,
                                              remap_table, scatter_kv, workloads)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda", torch.cuda.current_device())


def host(t):
    return workloads.bits(t)


def make(seed, fp8=False, **kw):
    args = dict(B=5, Hq=32, Hkv=8, D=128, block_size=16, lens=[1, 17, 700, 3000, 64],
                num_blocks=600)
    args.update(kw)
    wl = workloads.custom(seed=seed, **args)
    return workloads.to_fp8_kv(wl) if fp8 else wl


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("bs", [16, 32])
def test_gather_exact(fp8, bs):
    wl_h = make(1 + bs, fp8, block_size=bs)
    ref_k, ref_v = oracle.gather_kv(host(wl_h.k_cache), host(wl_h.v_cache),
                                    wl_h.block_table.numpy(), wl_h.context_lens.numpy())
    wl = wl_h.to(DEV)
    k, v = gather_kv(wl.k_cache, wl.v_cache, wl.block_table, wl.context_lens)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(k), ref_k)
    np.testing.assert_array_equal(host(v), ref_v)


@pytest.mark.parametrize("fp8", [False, True])
def test_scatter_exact_with_padding(fp8):
    wl_h = make(3, fp8, D=64, Hq=14, Hkv=2)
    rng = np.random.default_rng(3)
    n = 500
    nslots = wl_h.k_cache.shape[0] * wl_h.k_cache.shape[1]
    slots = rng.permutation(nslots)[:n].astype(np.int64)
    slots[rng.random(n) < 0.1] = -1
    src = make(4, fp8, D=64, Hq=14, Hkv=2, lens=[n], num_blocks=40)
    kr = src.k_cache.reshape(-1, 2, 64)[:n].contiguous()
    vr = src.v_cache.reshape(-1, 2, 64)[:n].contiguous()
    ref_k, ref_v = oracle.scatter_kv(host(kr), host(vr), slots, host(wl_h.k_cache),
                                     host(wl_h.v_cache))
    kc, vc = wl_h.k_cache.to(DEV), wl_h.v_cache.to(DEV)
    scatter_kv(kr.to(DEV), vr.to(DEV), torch.from_numpy(slots).to(DEV), kc, vc)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(kc), ref_k)
    np.testing.assert_array_equal(host(vc), ref_v)


@pytest.mark.parametrize("fp8", [False, True])
def test_compaction_copy_and_remap(fp8):
    """Move every live block to a free one and remap the table: bytes match
    the oracle and decode attention is unchanged."""
    wl_h = make(5, fp8, lens=[300, 17, 900], B=3, num_blocks=200)
    bs = wl_h.block_size
    bt = wl_h.block_table.numpy()
    lens = wl_h.context_lens.numpy()
    used = sorted({int(x) for b in range(3) for x in bt[b, : (lens[b] + bs - 1) // bs]})
    free = [i for i in range(wl_h.k_cache.shape[0]) if i not in used]
    pairs = np.array([[u, free[i]] for i, u in enumerate(used)], dtype=np.int64)
    new_id = np.arange(wl_h.k_cache.shape[0], dtype=np.int32)
    new_id[pairs[:, 0]] = pairs[:, 1]
    ref_k, ref_v = oracle.copy_blocks(host(wl_h.k_cache), host(wl_h.v_cache), pairs)
    ref_t = oracle.remap_table(bt, lens, bs, new_id)
    wl = wl_h.to(DEV)
    kw = dict(k_scale=wl.meta.get("k_scale"), v_scale=wl.meta.get("v_scale"))
    attn = PagedDecodeAttention(32, 8, 128, bs, torch.bfloat16, max_batch=3,
                                max_blocks_per_seq=bt.shape[1], kv_fp8=fp8)
    before = attn.run(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.context_lens, **kw)
    copy_blocks(wl.k_cache, wl.v_cache, torch.from_numpy(pairs).to(DEV))
    remap_table(wl.block_table, wl.context_lens, bs, torch.from_numpy(new_id).to(DEV))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(wl.k_cache), ref_k)
    np.testing.assert_array_equal(host(wl.v_cache), ref_v)
    np.testing.assert_array_equal(wl.block_table.cpu().numpy(), ref_t)
    # wipe the old blocks: the moved cache must not read them
    old = torch.from_numpy(pairs[:, 0]).to(DEV)
    wl.k_cache.view(torch.uint8)[old] = 0x7F
    wl.v_cache.view(torch.uint8)[old] = 0x7F
    after = attn.run(wl.q, wl.k_cache, wl.v_cache, wl.block_table, wl.context_lens, **kw)
    torch.cuda.synchronize()
    assert torch.equal(before, after)
    attn.close()


def test_out_of_range_ids_flagged_not_faulting():
    wl = make(6).to(DEV)
    err = torch.zeros(2, dtype=torch.int32, device=DEV)
    k0, v0 = wl.k_cache.clone(), wl.v_cache.clone()
    pairs = torch.tensor([[0, 1], [wl.k_cache.shape[0], 2]], dtype=torch.int64, device=DEV)
    copy_blocks(wl.k_cache, wl.v_cache, pairs, err=err)
    torch.cuda.synchronize()
    assert err.tolist() == [2, 1]
    assert torch.equal(wl.k_cache[1], k0[0]) and torch.equal(wl.k_cache[2], k0[2])
    err.zero_()
    rows = torch.zeros((3, 8, 128), dtype=torch.bfloat16, device=DEV)
    slots = torch.tensor([5, wl.k_cache.shape[0] * 16, -1], dtype=torch.int64, device=DEV)
    scatter_kv(rows, rows, slots, wl.k_cache, wl.v_cache, err=err)
    torch.cuda.synchronize()
    assert err.tolist() == [5, 1]
    err.zero_()
    table = wl.block_table.clone()
    table[2, 3] = -4
    k, v = gather_kv(wl.k_cache, wl.v_cache, table, wl.context_lens, err=err)
    torch.cuda.synchronize()
    assert err.tolist() == [2, 2]


def test_empty_calls_are_no_ops():
    wl = make(7).to(DEV)
    copy_blocks(wl.k_cache, wl.v_cache, torch.zeros((0, 2), dtype=torch.int64, device=DEV))
    k, v = gather_kv(wl.k_cache, wl.v_cache, wl.block_table[:0], wl.context_lens[:0])
    assert k.shape[0] == 0
    scatter_kv(k, v, torch.zeros(0, dtype=torch.int64, device=DEV), wl.k_cache, wl.v_cache)
    torch.cuda.synchronize()
