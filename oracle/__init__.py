"""FP64 CPU oracle for paged MQA/GQA decode attention (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it, and it
imports nothing from the CUDA library's package.

The arithmetic lives in ``paged_attn_oracle.c`` (plain C, double precision,
loops that state the definition of the operator). This module compiles it
with gcc on first use and marshals numpy arrays into it. Inputs are the raw
16-bit storage patterns of bf16/fp16 tensors (numpy ``uint16``), so the
conversion to double is the oracle's own exact decode.

Parity pins (all in ``tests/test_oracle_*.py``): brute-force dense attention
in arbitrary precision on tiny inputs, closed forms (one token, constant V,
constant logits, two tokens), invariance under block-table permutation and
block size, GQA reductions (MHA, MQA, duplicated heads), split-K merge equal
to the unsplit result, exact RNE rounding against numpy/torch conversions,
and a mutation test that plants plausible mistakes in a copy of the C source
and checks that the pins catch each one.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

BF16 = 0
FP16 = 1
FP8_E4M3 = 2  # K/V cache elements only

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None

# -ffp-contract=off: no fused multiply-add contraction, so the double
# arithmetic is the same on x86_64 and aarch64 hosts.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle's C source into a shared library at ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-o", tmp, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def _needs_build() -> bool:
    if not os.path.exists(_LIB_PATH):
        return True
    return os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_paged_decode.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, i32,
                                        f64, P, i32]
    lib.oracle_paged_decode.restype = i32
    lib.oracle_paged_decode_rows.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64,
                                             i32, f64, P, i64, P, i32]
    lib.oracle_paged_decode_rows.restype = i32
    lib.oracle_split_partials.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, i32,
                                          f64, i32, i32, P, P]
    lib.oracle_split_partials.restype = i32
    lib.oracle_lse_merge.argtypes = [P, P, i64, i32, i32, P]
    lib.oracle_lse_merge.restype = i32
    lib.oracle_round_array.argtypes = [P, i64, i32, P, P]
    lib.oracle_round_array.restype = None
    lib.oracle_decode_array.argtypes = [P, i64, i32, P]
    lib.oracle_decode_array.restype = None
    lib.oracle_paged_decode_kv.argtypes = [P, P, P, i32, P, P, P, P, i32, i32, i32, i32, i32,
                                           i32, i64, i32, f64, P, i64, P, i32]
    lib.oracle_paged_decode_kv.restype = i32
    lib.oracle_decode_e4m3_array.argtypes = [P, i64, P]
    lib.oracle_decode_e4m3_array.restype = None
    lib.oracle_copy_blocks.argtypes = [P, P, i64, i64, P, i64]
    lib.oracle_copy_blocks.restype = i32
    lib.oracle_gather_kv.argtypes = [P, P, i64, i32, i64, P, i32, P, i32, P, P]
    lib.oracle_gather_kv.restype = i32
    lib.oracle_scatter_kv.argtypes = [P, P, i64, i64, P, P, P, i64]
    lib.oracle_scatter_kv.restype = i32
    lib.oracle_remap_table.argtypes = [P, i32, i32, P, i32, P, i64]
    lib.oracle_remap_table.restype = i32
    lib.oracle_rope_kv_write.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                         i64, i32, P, P, P]
    lib.oracle_rope_kv_write.restype = i32
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building if needed) the oracle library. ``path`` loads another
    build of it (used by the mutation test)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build():
                compile_oracle()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _as_bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected raw 16-bit patterns (uint16), got {a.dtype}")
    return a


def _as_i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


_ERRORS = {-1: "invalid argument", -2: "index or length out of range", -3: "out of memory"}


def _check(status: int, what: str):
    if status != 0:
        raise ValueError(f"oracle {what}: {_ERRORS.get(status, status)}")


def default_threads() -> int:
    return os.cpu_count() or 1


def paged_decode(q, k_cache, v_cache, block_table, context_lens, dtype: int, scale: float,
                 threads: int | None = None, lib=None) -> np.ndarray:
    """out[B, Hq, D] (float64) of softmax(scale * q . K^T) . V over each
    sequence's paged K/V.

    q: uint16 [B, Hq, D]; k_cache/v_cache: uint16 [num_blocks, bs, Hkv, D];
    block_table: int32 [B, max_blocks]; context_lens: int32 [B].
    """
    lib = lib or load()
    q, k, v = _as_bits(q), _as_bits(k_cache), _as_bits(v_cache)
    bt, cl = _as_i32(block_table), _as_i32(context_lens)
    B, Hq, D = q.shape
    nb, bs, Hkv, Dk = k.shape
    assert Dk == D and v.shape == k.shape and bt.shape[0] == B and cl.shape == (B,)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    st = lib.oracle_paged_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(cl), B, Hq, Hkv, D,
                                 bs, bt.shape[1], nb, dtype, float(scale), _ptr(out),
                                 threads or default_threads())
    _check(st, "paged_decode")
    return out


def paged_decode_rows(q, k_cache, v_cache, block_table, context_lens, dtype: int, scale: float,
                      rows, threads: int | None = None, lib=None) -> np.ndarray:
    """Like :func:`paged_decode` for the (b, hq) pairs in ``rows`` only;
    returns float64 [len(rows), D]."""
    lib = lib or load()
    q, k, v = _as_bits(q), _as_bits(k_cache), _as_bits(v_cache)
    bt, cl = _as_i32(block_table), _as_i32(context_lens)
    rows = _as_i32(rows).reshape(-1, 2)
    B, Hq, D = q.shape
    nb, bs, Hkv, _ = k.shape
    out = np.zeros((rows.shape[0], D), dtype=np.float64)
    st = lib.oracle_paged_decode_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(cl), B, Hq, Hkv,
                                      D, bs, bt.shape[1], nb, dtype, float(scale), _ptr(rows),
                                      rows.shape[0], _ptr(out), threads or default_threads())
    _check(st, "paged_decode_rows")
    return out


def split_partials(q, k_cache, v_cache, block_table, context_lens, dtype: int, scale: float,
                   chunk_pages: int, num_splits: int, lib=None):
    """(lse[B, Hq, S], o[B, Hq, S, D]) of split-K partials; split s covers
    pages [s*chunk_pages, (s+1)*chunk_pages) of each sequence."""
    lib = lib or load()
    q, k, v = _as_bits(q), _as_bits(k_cache), _as_bits(v_cache)
    bt, cl = _as_i32(block_table), _as_i32(context_lens)
    B, Hq, D = q.shape
    nb, bs, Hkv, _ = k.shape
    lse = np.zeros((B, Hq, num_splits), dtype=np.float64)
    o = np.zeros((B, Hq, num_splits, D), dtype=np.float64)
    st = lib.oracle_split_partials(_ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(cl), B, Hq, Hkv, D,
                                   bs, bt.shape[1], nb, dtype, float(scale), chunk_pages,
                                   num_splits, _ptr(lse), _ptr(o))
    _check(st, "split_partials")
    return lse, o


def lse_merge(lse, o, lib=None) -> np.ndarray:
    """Merge partials: lse[..., S], o[..., S, D] -> out[..., D] (float64)."""
    lib = lib or load()
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    o = np.ascontiguousarray(o, dtype=np.float64)
    S, D = o.shape[-2], o.shape[-1]
    lead = o.shape[:-2]
    assert lse.shape == lead + (S,)
    n = int(np.prod(lead)) if lead else 1
    out = np.zeros(lead + (D,), dtype=np.float64)
    _check(lib.oracle_lse_merge(_ptr(lse), _ptr(o), n, S, D, _ptr(out)), "lse_merge")
    return out


def round_to(x, dtype: int, lib=None):
    """Round float64 values to bf16/fp16 with ties to even, directly from
    double. Returns (bits uint16, rounded float64)."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    bits = np.zeros(x.shape, dtype=np.uint16)
    rounded = np.zeros(x.shape, dtype=np.float64)
    lib.oracle_round_array(_ptr(x), x.size, dtype, _ptr(bits), _ptr(rounded))
    return bits, rounded


def decode(bits, dtype: int, lib=None) -> np.ndarray:
    """Exact float64 values of raw bf16/fp16 patterns."""
    lib = lib or load()
    bits = _as_bits(bits)
    out = np.zeros(bits.shape, dtype=np.float64)
    lib.oracle_decode_array(_ptr(bits), bits.size, dtype, _ptr(out))
    return out


def rope_kv_write(q, k, v, positions, slot_mapping, cos_sin, rot_dim: int, neox: bool,
                  dtype: int, k_cache, v_cache, q_out=None, lib=None):
    """RoPE on q and k plus the paged cache write (test infrastructure).

    q: uint16 [T, Hq, D]; k, v: uint16 [T, Hkv, D]; positions int32 [T];
    slot_mapping int64 [T]; cos_sin float32 [max_position, rot_dim];
    k_cache/v_cache uint16 [num_blocks, block_size, Hkv, D] (copied, not
    modified); q_out: uint16 [T, Hq, D] starting contents (zeros when None;
    tokens the call skips keep them). Returns (q_out, k_cache, v_cache)."""
    lib = lib or load()
    q, k, v = _as_bits(q), _as_bits(k), _as_bits(v)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    cs = np.ascontiguousarray(cos_sin, dtype=np.float32)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    q_out = np.zeros_like(q) if q_out is None else np.array(q_out, dtype=np.uint16, copy=True)
    num_slots = kc.shape[0] * kc.shape[1]
    st = lib.oracle_rope_kv_write(_ptr(q), _ptr(k), _ptr(v), _ptr(pos), _ptr(slots), _ptr(cs), T,
                                  Hq, Hkv, D, rot_dim, cs.shape[0], int(bool(neox)), num_slots,
                                  dtype, _ptr(q_out), _ptr(kc), _ptr(vc))
    _check(st, "rope_kv_write")
    return q_out, kc, vc


def decode_e4m3(bits, lib=None) -> np.ndarray:
    """Exact float64 values of FP8 E4M3 storage bytes (numpy uint8)."""
    lib = lib or load()
    b = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.zeros(b.shape, dtype=np.float64)
    lib.oracle_decode_e4m3_array(_ptr(b), b.size, _ptr(out))
    return out


def paged_decode_kv(q, k_cache, v_cache, block_table, context_lens, q_dtype: int, kv_dtype: int,
                    scale: float, k_scale=None, v_scale=None, rows=None,
                    threads: int | None = None, lib=None) -> np.ndarray:
    """Decode attention with K/V of any element type and per-kv-head
    dequantisation scales: k_t = k_scale[h] * k_cache[...], likewise v.

    q: uint16 [B, Hq, D]; k_cache/v_cache: uint8 (FP8_E4M3) or uint16
    [num_blocks, bs, Hkv, D]; k_scale/v_scale: [Hkv] or None (1). Returns
    float64 [B, Hq, D], or [len(rows), D] for the (b, hq) pairs in rows."""
    lib = lib or load()
    q = _as_bits(q)
    kdt = np.uint8 if kv_dtype == FP8_E4M3 else np.uint16
    k = np.ascontiguousarray(k_cache)
    v = np.ascontiguousarray(v_cache)
    if k.dtype != kdt or v.dtype != kdt:
        raise TypeError(f"caches must be {np.dtype(kdt).name} storage for kv_dtype {kv_dtype}")
    bt, cl = _as_i32(block_table), _as_i32(context_lens)
    B, Hq, D = q.shape
    nb, bs, Hkv, _ = k.shape
    ks = None if k_scale is None else np.ascontiguousarray(k_scale, dtype=np.float64).reshape(Hkv)
    vs = None if v_scale is None else np.ascontiguousarray(v_scale, dtype=np.float64).reshape(Hkv)
    if rows is None:
        out = np.zeros((B, Hq, D), dtype=np.float64)
        rp, nr = None, 0
    else:
        rows = _as_i32(rows).reshape(-1, 2)
        out = np.zeros((rows.shape[0], D), dtype=np.float64)
        rp, nr = _ptr(rows), rows.shape[0]
    st = lib.oracle_paged_decode_kv(_ptr(q), _ptr(k), _ptr(v), kv_dtype,
                                    None if ks is None else _ptr(ks),
                                    None if vs is None else _ptr(vs), _ptr(bt), _ptr(cl), B, Hq,
                                    Hkv, D, bs, bt.shape[1], nb, q_dtype, float(scale), rp, nr,
                                    _ptr(out), threads or default_threads())
    _check(st, "paged_decode_kv")
    return out


def _raw_rows(cache) -> np.ndarray:
    """Any numpy cache [num_blocks, bs, Hkv, D] as contiguous bytes."""
    return np.ascontiguousarray(cache).view(np.uint8)


def copy_blocks(k_cache, v_cache, pairs, lib=None):
    """Copies of the caches with block pairs[i][1] := block pairs[i][0]."""
    lib = lib or load()
    k = np.array(k_cache, copy=True, order="C")
    v = np.array(v_cache, copy=True, order="C")
    nb = k.shape[0]
    block_bytes = k.nbytes // max(nb, 1)
    pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    _check(lib.oracle_copy_blocks(_ptr(k.view(np.uint8)), _ptr(v.view(np.uint8)), nb,
                                  block_bytes, _ptr(pr), pr.shape[0]), "copy_blocks")
    return k, v


def gather_kv(k_cache, v_cache, block_table, lens, lib=None):
    """(k_out, v_out) [sum(lens), Hkv, D]: each sequence's tokens in order."""
    lib = lib or load()
    k, v = np.ascontiguousarray(k_cache), np.ascontiguousarray(v_cache)
    nb, bs = k.shape[0], k.shape[1]
    row_shape = k.shape[2:]
    row_bytes = k.nbytes // max(nb * bs, 1)
    bt, cl = _as_i32(block_table), _as_i32(lens)
    total = int(cl.sum())
    ko = np.zeros((total,) + row_shape, dtype=k.dtype)
    vo = np.zeros((total,) + row_shape, dtype=k.dtype)
    _check(lib.oracle_gather_kv(_ptr(_raw_rows(k)), _ptr(_raw_rows(v)), nb, bs, row_bytes,
                                _ptr(bt), bt.shape[1], _ptr(cl), cl.shape[0],
                                _ptr(ko.view(np.uint8)), _ptr(vo.view(np.uint8))), "gather_kv")
    return ko, vo


def scatter_kv(k_rows, v_rows, slot_mapping, k_cache, v_cache, lib=None):
    """Copies of the caches with row t written to slot slot_mapping[t] (< 0 skipped)."""
    lib = lib or load()
    kr, vr = np.ascontiguousarray(k_rows), np.ascontiguousarray(v_rows)
    k = np.array(k_cache, copy=True, order="C")
    v = np.array(v_cache, copy=True, order="C")
    n = kr.shape[0]
    row_bytes = kr.nbytes // max(n, 1) if n else k.nbytes // max(k.shape[0] * k.shape[1], 1)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    _check(lib.oracle_scatter_kv(_ptr(kr.view(np.uint8)), _ptr(vr.view(np.uint8)), n, row_bytes,
                                 _ptr(sm), _ptr(k.view(np.uint8)), _ptr(v.view(np.uint8)),
                                 k.shape[0] * k.shape[1]), "scatter_kv")
    return k, v


def remap_table(block_table, lens, block_size: int, new_id, lib=None) -> np.ndarray:
    """A copy of the table with every used entry e replaced by new_id[e]."""
    lib = lib or load()
    bt = np.array(block_table, dtype=np.int32, copy=True, order="C")
    cl = _as_i32(lens)
    nid = _as_i32(new_id)
    _check(lib.oracle_remap_table(_ptr(bt), bt.shape[0], bt.shape[1], _ptr(cl), block_size,
                                  _ptr(nid), nid.shape[0]), "remap_table")
    return bt
