"""The C ABI without a GPU: the library builds and loads, exports every
symbol the header declares, rejects bad arguments with the documented codes
before touching CUDA, and the split planner's host logic."""
import ctypes
import os
import re

import pytest

import paged_gqa_decode_attention_gb300 as pda
from paged_gqa_decode_attention_gb300 import build as pda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pda_build.build()
    return pda.load_library()


def header_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*(?:[\w\*]+\s+)+\**(paged_decode_attn_\w+)\s*\(", text,
                                    re.M))
    return names


def test_exports_every_header_function(lib):
    declared = header_functions()
    assert declared, "no declarations parsed"
    assert declared == set(pda.EXPORTS), declared ^ set(pda.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_abi_version(lib):
    assert lib.paged_decode_attn_abi_version() == pda.ABI_VERSION == 2


def test_library_needs_no_driver_to_load(lib):
    out = os.popen(f"ldd {pda_build.LIB_PATH}").read()
    assert "libcuda.so" not in out and "libcudart" not in out


@pytest.mark.parametrize("field,value,status", [
    ("num_q_heads", 0, pda.PDA_EINVAL),
    ("num_q_heads", 30, pda.PDA_EINVAL),        # not a multiple of Hkv = 8
    ("num_q_heads", 8 * 17, pda.PDA_EUNSUPPORTED),  # group size 17
    ("head_dim", 96, pda.PDA_EUNSUPPORTED),
    ("head_dim", 0, pda.PDA_EINVAL),
    ("block_size", 8, pda.PDA_EUNSUPPORTED),
    ("dtype", 7, pda.PDA_EINVAL),
    ("max_batch", 0, pda.PDA_EINVAL),
    ("max_batch", 70000, pda.PDA_EINVAL),
    ("max_splits", 65, pda.PDA_EINVAL),
    ("max_blocks_per_seq", 0, pda.PDA_EINVAL),
    ("device", -1, pda.PDA_EINVAL),
])
def test_create_rejects_bad_config_before_cuda(lib, field, value, status):
    cfg = pda.make_config(32, 8, 128, 16)
    setattr(cfg, field, value)
    h = ctypes.c_void_p(123)
    assert lib.paged_decode_attn_create(ctypes.byref(cfg), ctypes.byref(h)) == status
    assert h.value is None
    assert lib.paged_decode_attn_last_error()


@pytest.mark.parametrize("Hq,Hkv,D,ok", [(14, 2, 64, True), (28, 4, 128, True), (40, 8, 128, True),
                                         (24, 8, 128, True), (8, 1, 256, False), (16, 8, 256, True),
                                         (32, 8, 256, True), (12, 2, 256, False), (8, 8, 64, True),
                                         (4, 1, 64, True), (128, 8, 128, True), (72, 8, 64, True),
                                         (16, 1, 128, True), (136, 8, 128, False),
                                         (17, 1, 64, False), (40, 8, 256, False)])
def test_create_geometries_before_cuda(lib, Hq, Hkv, D, ok):
    """Group sizes 1..16 at head dims 64 and 128, 1..4 at 256: accepted by the
    config checks (creation then needs a GPU), others are unsupported."""
    cfg = pda.make_config(Hq, Hkv, D, 16)
    h = ctypes.c_void_p()
    st = lib.paged_decode_attn_create(ctypes.byref(cfg), ctypes.byref(h))
    if ok:
        assert st != pda.PDA_EUNSUPPORTED and st != pda.PDA_EINVAL, lib.paged_decode_attn_last_error()
        if st == pda.PDA_OK:
            lib.paged_decode_attn_destroy(h)
    else:
        assert st == pda.PDA_EUNSUPPORTED


@pytest.mark.parametrize("Hq,Hkv,D,bs,ok", [(32, 8, 128, 64, True), (14, 2, 64, 64, True),
                                            (16, 8, 256, 64, True), (128, 8, 128, 64, False),
                                            (32, 8, 128, 128, False), (32, 8, 128, 8, False)])
def test_create_block_sizes_before_cuda(lib, Hq, Hkv, D, bs, ok):
    """Block sizes 16 and 32 everywhere, 64 at group sizes up to 8."""
    cfg = pda.make_config(Hq, Hkv, D, bs)
    h = ctypes.c_void_p()
    st = lib.paged_decode_attn_create(ctypes.byref(cfg), ctypes.byref(h))
    if ok:
        assert st != pda.PDA_EUNSUPPORTED and st != pda.PDA_EINVAL, lib.paged_decode_attn_last_error()
        if st == pda.PDA_OK:
            lib.paged_decode_attn_destroy(h)
    else:
        assert st == pda.PDA_EUNSUPPORTED


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.paged_decode_attn_create(None, ctypes.byref(h)) == pda.PDA_EINVAL
    cfg = pda.make_config(32, 8)
    assert lib.paged_decode_attn_create(ctypes.byref(cfg), None) == pda.PDA_EINVAL
    assert lib.paged_decode_attn_run(None, 0, 0, 0, 0, 0, 1, 1, 1, 1.0, 0, 0) == pda.PDA_EINVAL
    lib.paged_decode_attn_destroy(None)  # NULL-safe
    assert lib.paged_decode_attn_validate(None, 0, 0, 1, 1, 1, 0) == pda.PDA_EINVAL
    code = ctypes.c_int()
    assert lib.paged_decode_attn_check_device_error(None, ctypes.byref(code), ctypes.byref(code),
                                                    0) == pda.PDA_EINVAL


def test_merge_rejects_bad_arguments_before_cuda(lib):
    assert lib.paged_decode_attn_merge(0, 0, 1, 0, 128, 0, 0, 0, 0) == pda.PDA_EINVAL  # S = 0
    assert lib.paged_decode_attn_merge(0, 0, 1, 65, 128, 0, 0, 0, 0) == pda.PDA_EINVAL
    assert lib.paged_decode_attn_merge(0, 0, 1, 4, 130, 0, 0, 0, 0) == pda.PDA_EINVAL
    assert lib.paged_decode_attn_merge(0, 0, 1, 4, 128, 0, 9, 0, 0) == pda.PDA_EINVAL
    assert lib.paged_decode_attn_merge(0, 0, 0, 4, 128, 0, 0, 0, 0) == pda.PDA_OK  # no rows
    assert lib.paged_decode_attn_merge(0, 0, 2, 4, 128, 0, 0, 0, 0) == pda.PDA_EINVAL  # NULL


# --------------------------- split planner --------------------------------

def plan(B, max_blocks, hint=0, Hq=32, Hkv=8, bs=16, sms=152, max_splits=64):
    cfg = pda.make_config(Hq, Hkv, 128, bs, max_batch=max(1, B), max_blocks_per_seq=max_blocks,
                          max_splits=max_splits)
    return pda.plan(cfg, sms, B, max_blocks, hint)


@pytest.mark.parametrize("B,pages", [(1, 2), (1, 512), (4, 2048), (32, 4), (8, 64), (128, 128),
                                     (1, 1), (3, 1000), (64, 4096)])
def test_plan_covers_every_page(lib, B, pages):
    S, chunk = plan(B, pages)
    assert 1 <= S <= 64 and chunk >= 1
    assert S * chunk >= pages > (S - 1) * chunk  # S splits of chunk pages cover all, none empty


def test_plan_no_split_when_grid_is_full(lib):
    assert plan(128, 128, Hq=64, bs=32)[0] == 1       # 1024 CTAs already
    assert plan(32, 4)[0] == 1                         # short contexts
    assert plan(1, 2)[0] == 1                          # tiny


def test_plan_splits_long_contexts_to_fill_the_gpu(lib):
    # the 16-bit tensor-core kernel plans one wave over 27/32 of the SMs (128 of 152)
    S1, _ = plan(1, 512)    # B=1, L=8192: 8 CTAs without splitting
    S4, _ = plan(4, 2048)   # B=4, L=32768
    assert S1 * 8 >= 128 and S4 * 32 >= 128
    assert S1 * 8 <= 152 and S4 * 32 <= 152    # one wave: no CTA takes a second unit
    assert plan(1, 2048)[0] >= plan(4, 2048)[0]


def test_plan_slots_by_kernel(lib):
    """The 16-bit tensor-core kernel plans one wave over 128 of 152 SMs; FP8
    caches (limited per SM) and the CUDA-core kernel (G 1, 2) plan over every
    SM and CTA slot."""
    B, pages = 8, 2048                    # 64 (sequence, kv head) pairs, L = 32768
    S16, _ = plan(B, pages)
    assert S16 * 64 <= 128
    cfg8 = pda.make_config(32, 8, 128, 16, max_batch=B, max_blocks_per_seq=pages, kv_fp8=True)
    S8, _ = pda.plan(cfg8, 152, B, pages)
    assert S8 * 64 > 152                  # several units per SM, balanced dynamically
    Sg2, _ = plan(4, pages, Hq=16)        # G = 2: CUDA-core kernel, 2 CTAs per SM
    assert Sg2 * 32 > 128


def test_plan_respects_hint_and_caps(lib):
    assert plan(1, 2048, hint=64)[0] <= 4
    assert plan(1, 4096, max_splits=8)[0] <= 8
    cfg = pda.make_config(32, 8)
    with pytest.raises(pda.PDAError):
        pda.plan(cfg, 0, 1, 16)           # no SMs
    with pytest.raises(pda.PDAError):
        pda.plan(cfg, 152, 1, 10 ** 6)    # max_blocks beyond the config


# --------------------------- RoPE + KV write -------------------------------

def rope_call(lib, **kw):
    a = dict(q=16, qs=0, k=32, ks=0, v=48, vs=0, pos=64, slots=80, cs=96, max_pos=10,
             rot=64, neox=1, T=4, Hq=14, Hkv=2, D=64, dtype=0, qo=1 << 30, qos=0,
             kc=1 << 31, vc=1 << 32, nslots=100, err=None, dev=0, stream=None)
    a.update(kw)
    return lib.paged_decode_attn_rope_kv_write(
        a["q"], a["qs"], a["k"], a["ks"], a["v"], a["vs"], a["pos"], a["slots"], a["cs"],
        a["max_pos"], a["rot"], a["neox"], a["T"], a["Hq"], a["Hkv"], a["D"], a["dtype"],
        a["qo"], a["qos"], a["kc"], a["vc"], a["nslots"], a["err"], a["dev"], a["stream"])


@pytest.mark.parametrize("kw", [dict(T=-1), dict(Hq=0), dict(D=72), dict(D=0), dict(rot=72),
                                dict(rot=80), dict(dtype=2), dict(qs=100), dict(ks=8),
                                dict(nslots=-1), dict(q=0), dict(cs=0), dict(q=18),
                                dict(dev=-1)])
def test_rope_kv_write_rejects_bad_arguments_before_cuda(lib, kw):
    assert rope_call(lib, **kw) == pda.PDA_EINVAL
    assert lib.paged_decode_attn_last_error()


def test_rope_kv_write_aliasing_and_no_op(lib):
    assert rope_call(lib, T=0, q=0, k=0) == pda.PDA_OK  # nothing to do
    assert rope_call(lib, vc=1 << 31) == pda.PDA_EALIAS             # k_cache == v_cache
    assert rope_call(lib, qo=16 + 64) == pda.PDA_EALIAS             # q_out inside q
    assert rope_call(lib, kc=16) == pda.PDA_EALIAS                  # cache over q
    assert rope_call(lib, qo=96) == pda.PDA_EALIAS                  # q_out over the table


def test_rope_kv_write_fused_views_are_not_aliases(lib):
    """q, k, v as views into one fused [T, (Hq + 2 Hkv) * D] buffer, rotated
    in place: the row sets interleave without sharing a byte, so the call
    passes the alias checks (and reaches CUDA, absent here)."""
    row = (14 + 4) * 64
    base = 1 << 20
    st = rope_call(lib, q=base, qs=row, k=base + 14 * 64 * 2, ks=row, v=base + 16 * 64 * 2,
                   vs=row, qo=base, qos=row)
    assert st == pda.PDA_ECUDA, lib.paged_decode_attn_last_error()
    # q_out as the k part of the same rows does overlap
    st = rope_call(lib, q=base, qs=row, k=base + 14 * 64 * 2, ks=row, v=base + 16 * 64 * 2,
                   vs=row, qo=base + 14 * 64 * 2, qos=row)
    assert st == pda.PDA_EALIAS
