"""The allocation-free entry point, paged_decode_attn_run_noalloc.

Some callers may not allocate device memory at all (code running where
cudaMalloc is forbidden, or a runtime whose own pool owns every byte of
device memory); they cannot create a handle, because creating one allocates
the split-K workspace. This entry point serves them from scratch compiled
into the library. Here it is called through the C ABI and its output is
compared with the handle-based entry point's on the same inputs, for two
calls in a row (the second call finds the first call's leftovers in the
shared scratch). The file sorts last so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

from paged_gqa_decode_attention_gb300 import (PDA_EINVAL, PDA_OK, load_library, workloads)
from parity import assert_close, make_attn, run_gpu

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

DEV = torch.device("cuda", torch.cuda.current_device())
DT = {torch.bfloat16: 0, torch.float16: 1}


def noalloc(lib, wl, out, num_splits=0):
    return lib.paged_decode_attn_run_noalloc(
        wl.q.data_ptr(), wl.k_cache.data_ptr(), wl.v_cache.data_ptr(), wl.block_table.data_ptr(),
        wl.context_lens.data_ptr(), wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
        wl.block_size, DT[wl.q.dtype], wl.max_blocks, wl.num_blocks, float(wl.scale),
        out.data_ptr(), num_splits, DEV.index, torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_handle_path_two_calls_in_a_row():
    lib = load_library()
    # both cases split their sequences, so the scratch is really used
    cases = [workloads.long_context(seed=11, batch=2, context=3000, num_blocks=1024).to(DEV),
             workloads.custom(seed=12, B=5, Hq=64, Hkv=8, D=128, block_size=32,
                              lens=[4000, 33, 1700, 1, 2500], num_blocks=400).to(DEV)]
    refs = []
    for wl in cases:
        attn = make_attn(wl)
        refs.append(run_gpu(attn, wl).double().cpu().numpy())
        attn.close()
    outs = [torch.full_like(wl.q, float("nan")) for wl in cases]
    for wl, out in zip(cases, outs):  # two calls back to back on one stream
        assert noalloc(lib, wl, out) == PDA_OK, lib.paged_decode_attn_last_error()
    torch.cuda.synchronize()
    for wl, out, ref in zip(cases, outs, refs):
        assert_close(out, ref, f"noalloc {wl.name}")


def test_noalloc_rejects_split_request_beyond_scratch():
    lib = load_library()
    wl = workloads.long_context(seed=13, batch=64, context=4096, num_blocks=16384).to(DEV)
    out = torch.empty_like(wl.q)
    # 64 sequences x 32 heads x 64 splits x 128 dims of fp32 partials > 8 MiB
    assert noalloc(lib, wl, out, num_splits=64) == PDA_EINVAL
    assert b"scratch" in lib.paged_decode_attn_last_error()
    # the heuristic lowers the split count to what fits and stays exact
    assert noalloc(lib, wl, out) == PDA_OK
    torch.cuda.synchronize()
    attn = make_attn(wl)
    ref = run_gpu(attn, wl).double().cpu().numpy()
    attn.close()
    assert_close(out, ref, "noalloc heuristic within scratch")
