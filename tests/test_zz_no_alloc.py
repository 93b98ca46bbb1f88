"""The allocation-free entry point, paged_decode_attn_run_noalloc.

Some callers may not allocate device memory at all (code running where
cudaMalloc is forbidden, or a runtime whose own pool owns every byte of
device memory); they cannot create a handle, because creating one allocates
the split-K workspace. This entry point serves them from scratch compiled
into the library. Here it is called through the C ABI and its output is
compared with the handle-based entry point's and with the FP64 oracle on the
same inputs, for two calls in a row (the second call finds the first call's
leftovers in the shared scratch). The file sorts last so that a run stopping
at the first failure has already run every other test.
"""
import pytest
import torch

from paged_gqa_decode_attention_gb300 import (PDA_EINVAL, PDA_OK, load_library, make_config, plan,
                                              workloads)
from parity import assert_close, make_attn, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda", torch.cuda.current_device())
DT = {torch.bfloat16: 0, torch.float16: 1}
# built-in scratch: 2^21 fp32 partial values
PARTIAL_FLOATS = 1 << 21


def noalloc(lib, wl, out, num_splits=0):
    return lib.paged_decode_attn_run_noalloc(
        wl.q.data_ptr(), wl.k_cache.data_ptr(), wl.v_cache.data_ptr(), wl.block_table.data_ptr(),
        wl.context_lens.data_ptr(), wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
        wl.block_size, DT[wl.q.dtype], wl.max_blocks, wl.num_blocks, float(wl.scale),
        out.data_ptr(), num_splits, DEV.index, torch.cuda.current_stream().cuda_stream)


def heuristic_splits(wl):
    cfg = make_config(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, wl.q.dtype,
                      max_batch=wl.batch, max_blocks_per_seq=wl.max_blocks, max_splits=64,
                      device=DEV.index)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    return plan(cfg, sms, wl.batch, wl.max_blocks)[0]


def test_noalloc_matches_handle_path_two_calls_in_a_row():
    lib = load_library()
    cases = [workloads.long_context(seed=11, batch=2, context=3000, num_blocks=1024),
             workloads.custom(seed=12, B=5, Hq=64, Hkv=8, D=128, block_size=32,
                              lens=[4000, 33, 1700, 1, 2500], num_blocks=400)]
    oracles = [oracle_ref(wl) for wl in cases]
    cases = [wl.to(DEV) for wl in cases]
    for wl in cases:  # both cases split their sequences, so the scratch is really used
        assert heuristic_splits(wl) > 1, wl.name
    refs = []
    for wl in cases:
        attn = make_attn(wl)
        refs.append(run_gpu(attn, wl).double().cpu().numpy())
        attn.close()
    outs = [torch.full_like(wl.q, float("nan")) for wl in cases]
    for wl, out in zip(cases, outs):  # two calls back to back on one stream
        assert noalloc(lib, wl, out) == PDA_OK, lib.paged_decode_attn_last_error()
    torch.cuda.synchronize()
    for wl, out, ref, ref64 in zip(cases, outs, refs, oracles):
        assert_close(out, ref, f"noalloc {wl.name} vs handle path")
        assert_close(out, ref64, f"noalloc {wl.name} vs oracle")


def test_noalloc_split_requests_and_the_scratch_bound():
    """An explicit request is judged by the split count it really runs as:
    64 sequences x 32 heads x 128 dims leave room for 8 splits; num_splits 16
    over 4 pages runs as 4 splits and is accepted, num_splits 16 over 64 pages
    needs 16 and is rejected with a message naming that count. The heuristic's
    pick stays within the scratch on its own (its units fill at most two waves
    of the GPU, far below the bound) and is exact."""
    lib = load_library()
    B = 64
    fit = PARTIAL_FLOATS // (B * 32 * 128)
    assert fit == 8
    short = workloads.long_context(seed=14, batch=B, context=64, num_blocks=300)
    ref64 = oracle_ref(short)
    short = short.to(DEV)
    assert short.max_blocks == 4
    out = torch.full_like(short.q, float("nan"))
    assert noalloc(lib, short, out, num_splits=16) == PDA_OK, lib.paged_decode_attn_last_error()
    torch.cuda.synchronize()
    assert_close(out, ref64, "noalloc num_splits=16 over 4 pages (runs as 4 splits)")

    wl_host = workloads.long_context(seed=13, batch=B, context=1024, num_blocks=4200)
    wl = wl_host.to(DEV)
    assert wl.max_blocks == 64
    out = torch.empty_like(wl.q)
    assert noalloc(lib, wl, out, num_splits=16) == PDA_EINVAL
    msg = lib.paged_decode_attn_last_error()
    assert b"scratch" in msg and b"16 splits" in msg and b"at most 8" in msg, msg
    assert noalloc(lib, wl, out, num_splits=8) == PDA_OK, lib.paged_decode_attn_last_error()
    torch.cuda.synchronize()
    ref64 = oracle_ref(wl_host)
    assert_close(out, ref64, "noalloc num_splits=8 (the most that fit)")
    out.fill_(float("nan"))
    assert noalloc(lib, wl, out) == PDA_OK, lib.paged_decode_attn_last_error()
    torch.cuda.synchronize()
    assert heuristic_splits(wl) <= fit
    assert_close(out, ref64, "noalloc heuristic within scratch")
