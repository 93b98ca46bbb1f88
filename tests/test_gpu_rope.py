"""GPU parity of the RoPE + paged-KV write kernel against the FP64 oracle.

The kernel is exactly rounded, so every comparison is bit for bit: q_out,
and the whole K and V cache pools (the written rows and every row the call
must leave alone). Calls go through the C ABI (ctypes binding)."""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_attention_gb300 import (PDA_EALIAS, PDA_EINVAL, PDAError, load_library,
                                              rope_kv_write, workloads)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda", torch.cuda.current_device())
ORACLE_DT = {torch.bfloat16: oracle.BF16, torch.float16: oracle.FP16}


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def oracle_rope(wl, q_out0=None):
    """The oracle on the host copy of a RoPE workload."""
    return oracle.rope_kv_write(
        bits(wl.q), bits(wl.k), bits(wl.v), wl.positions.cpu().numpy(),
        wl.slot_mapping.cpu().numpy(), wl.cos_sin.cpu().numpy(), wl.rot_dim, wl.neox,
        ORACLE_DT[wl.qkv.dtype], bits(wl.k_cache), bits(wl.v_cache),
        q_out=None if q_out0 is None else bits(q_out0))


def run_and_compare(wl_host, in_place=False, packed=False):
    ref_q, ref_k, ref_v = oracle_rope(wl_host, q_out0=wl_host.q if in_place else None)
    wl = wl_host.to(DEV)
    q, k, v = wl.q, wl.k, wl.v
    if packed:
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    if in_place:
        q_out = rope_kv_write(q, k, v, wl.positions, wl.slot_mapping, wl.cos_sin, wl.k_cache,
                              wl.v_cache, neox=wl.neox, q_out=q)
    else:
        q_out = torch.zeros_like(q, memory_format=torch.contiguous_format)
        rope_kv_write(q, k, v, wl.positions, wl.slot_mapping, wl.cos_sin, wl.k_cache, wl.v_cache,
                      neox=wl.neox, q_out=q_out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(q_out), ref_q, err_msg=f"{wl.name}: q_out")
    np.testing.assert_array_equal(bits(wl.k_cache), ref_k, err_msg=f"{wl.name}: k_cache")
    np.testing.assert_array_equal(bits(wl.v_cache), ref_v, err_msg=f"{wl.name}: v_cache")
    return wl


@pytest.mark.parametrize("tokens", [1, 7, 32, 512])
def test_qwen05b_decode_bit_exact(tokens):
    """Qwen2.5-0.5B geometry (14/2 heads, D 64, theta 1e6), 1-512 new tokens."""
    run_and_compare(workloads.rope_batch(seed=tokens, tokens=tokens))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("geom", [(32, 8, 128, 128), (32, 8, 128, 64), (28, 4, 128, 128),
                                  (8, 1, 256, 128), (4, 4, 16, 16), (12, 2, 128, 0)])
def test_geometries_layouts_dtypes(dtype, neox, geom):
    Hq, Hkv, D, rot = geom
    for mode in ("decode", "prefill"):
        wl = workloads.rope_batch(seed=Hq + D + rot, tokens=300, Hq=Hq, Hkv=Hkv, D=D,
                                  rot_dim=rot, theta=10000.0, max_position=4096, dtype=dtype,
                                  mode=mode, neox=neox, pad_frac=0.1, block_size=16)
        run_and_compare(wl)


def test_in_place_and_packed_views():
    wl = workloads.rope_batch(seed=3, tokens=200, Hq=32, Hkv=8, D=128, rot_dim=64,
                              max_position=8192, pad_frac=0.2)
    run_and_compare(wl, in_place=True)
    run_and_compare(wl, packed=True)


def test_extreme_angles_and_values():
    """Large positions (angles of thousands of radians), values near the
    format's range and subnormals: still bit-exact."""
    wl = workloads.rope_batch(seed=5, tokens=256, Hq=8, Hkv=2, D=128, max_position=1 << 20,
                              theta=10000.0)
    scale = torch.tensor([1e-38, 1e-30, 1.0, 1e30, 1e38]).repeat(1 + wl.qkv.numel() // 5)
    wl.qkv.copy_((wl.qkv.float() * scale[:wl.qkv.numel()].view_as(wl.qkv)).clamp(
        -3.3e38, 3.3e38).to(wl.qkv.dtype))
    run_and_compare(wl)
    wl = workloads.rope_batch(seed=6, tokens=256, Hq=8, Hkv=2, D=128, dtype="fp16",
                              max_position=1 << 20, theta=10000.0)
    scale = torch.tensor([1e-7, 6e-5, 1.0, 3e4, 6e4]).repeat(1 + wl.qkv.numel() // 5)
    wl.qkv.copy_((wl.qkv.float() * scale[:wl.qkv.numel()].view_as(wl.qkv)).clamp(
        -65504, 65504).to(wl.qkv.dtype))
    run_and_compare(wl)


def test_large_prefill_full_size():
    """The bandwidth workload (32/8/128, 32768-token prefill), every output."""
    run_and_compare(workloads.rope_batch(seed=0, tokens=32768, Hq=32, Hkv=8, D=128,
                                         theta=10000.0, mode="prefill"))


def test_bad_positions_and_slots_flagged_without_faulting():
    wl_host = workloads.rope_batch(seed=9, tokens=64, max_position=1024)
    pos = wl_host.positions.clone()
    pos[5] = 1024      # one past the table
    pos[9] = -3
    slots = wl_host.slot_mapping.clone()
    slots[20] = wl_host.k_cache.shape[0] * wl_host.k_cache.shape[1]  # one past the pool
    wl_host.positions, wl_host.slot_mapping = pos, slots
    ref_q, ref_k, ref_v = oracle_rope(wl_host)
    wl = wl_host.to(DEV)
    err = torch.zeros(2, dtype=torch.int32, device=DEV)
    q_out = torch.zeros_like(wl.q, memory_format=torch.contiguous_format)
    rope_kv_write(wl.q, wl.k, wl.v, wl.positions, wl.slot_mapping, wl.cos_sin, wl.k_cache,
                  wl.v_cache, q_out=q_out, err=err)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(q_out), ref_q)
    np.testing.assert_array_equal(bits(wl.k_cache), ref_k)
    np.testing.assert_array_equal(bits(wl.v_cache), ref_v)
    code, detail = err.tolist()
    assert (code, detail) in {(4, 5), (4, 9), (5, 20)}
    assert not q_out[5].any() and not q_out[9].any() and q_out[20].any()


def test_zero_tokens_and_abi_errors():
    wl = workloads.rope_batch(seed=1, tokens=8).to(DEV)
    lib = load_library()
    empty = wl.q[:0]
    out = rope_kv_write(empty, wl.k[:0], wl.v[:0], wl.positions[:0], wl.slot_mapping[:0],
                        wl.cos_sin, wl.k_cache, wl.v_cache)
    assert out.shape[0] == 0
    with pytest.raises(PDAError) as e:  # k cache overlapping v cache
        rope_kv_write(wl.q, wl.k, wl.v, wl.positions, wl.slot_mapping, wl.cos_sin, wl.k_cache,
                      wl.k_cache)
    assert e.value.status == PDA_EALIAS
    with pytest.raises(PDAError) as e:  # q_out partially overlapping q
        rope_kv_write(wl.q, wl.k, wl.v, wl.positions, wl.slot_mapping, wl.cos_sin, wl.k_cache,
                      wl.v_cache, q_out=wl.qkv.view(-1)[64:64 + wl.q.numel()].view(wl.q.shape))
    assert e.value.status == PDA_EALIAS
    st = lib.paged_decode_attn_rope_kv_write(
        wl.q.data_ptr() + 2, 0, wl.k.data_ptr(), 0, wl.v.data_ptr(), 0, wl.positions.data_ptr(),
        wl.slot_mapping.data_ptr(), wl.cos_sin.data_ptr(), 32768, 64, 1, 8, 14, 2, 64, 0,
        torch.empty_like(wl.q.contiguous()).data_ptr(), 0, wl.k_cache.data_ptr(),
        wl.v_cache.data_ptr(), 1024, None, DEV.index or 0, None)
    assert st == PDA_EINVAL and b"aligned" in lib.paged_decode_attn_last_error()


def test_written_cache_is_read_by_decode_attention():
    """End to end: new tokens rotated and written by this kernel, then decode
    attention over sequences that end in them, against the oracle run on the
    oracle's own write."""
    from paged_gqa_decode_attention_gb300 import PagedDecodeAttention
    from parity import assert_close
    bs, Hq, Hkv, D = 16, 32, 8, 128
    B, L = 4, 200
    rng = np.random.default_rng(0)
    num_blocks = 64
    table = rng.permutation(num_blocks)[: B * 16].reshape(B, 16).astype(np.int32)
    wl = workloads.rope_batch(seed=2, tokens=B, Hq=Hq, Hkv=Hkv, D=D, theta=10000.0,
                              max_position=4096, num_blocks=num_blocks, block_size=bs)
    # token b is position L-1 of sequence b
    wl.positions = torch.full((B,), L - 1, dtype=torch.int32)
    wl.slot_mapping = torch.as_tensor(table[:, (L - 1) // bs] * bs + (L - 1) % bs,
                                      dtype=torch.int64)
    ref_q, ref_k, ref_v = oracle_rope(wl)
    lens = np.full(B, L, dtype=np.int32)
    scale = D ** -0.5
    ref = oracle.paged_decode(ref_q, ref_k, ref_v, table, lens, oracle.BF16, scale)
    g = wl.to(DEV)
    q_out = rope_kv_write(g.q, g.k, g.v, g.positions, g.slot_mapping, g.cos_sin, g.k_cache,
                          g.v_cache)
    attn = PagedDecodeAttention(Hq, Hkv, D, bs, torch.bfloat16, max_batch=B,
                                max_blocks_per_seq=16)
    out = attn.run(q_out, g.k_cache, g.v_cache, torch.as_tensor(table).to(DEV),
                   torch.as_tensor(lens).to(DEV), scale)
    torch.cuda.synchronize()
    attn.close()
    assert_close(out, ref, "rope then decode")


def test_graph_capture_replay():
    wl = workloads.rope_batch(seed=4, tokens=64).to(DEV)
    q_out = torch.empty_like(wl.q, memory_format=torch.contiguous_format)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rope_kv_write(wl.q, wl.k, wl.v, wl.positions, wl.slot_mapping, wl.cos_sin, wl.k_cache,
                      wl.v_cache, q_out=q_out, stream=s)
    g.replay()
    torch.cuda.synchronize()
    eager = rope_kv_write(wl.q, wl.k, wl.v, wl.positions, wl.slot_mapping, wl.cos_sin,
                          wl.k_cache.clone(), wl.v_cache.clone())
    torch.cuda.synchronize()
    assert torch.equal(eager, q_out)
