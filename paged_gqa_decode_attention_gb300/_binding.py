"""ctypes binding of the C ABI in include/paged_decode_attn.h.

Argument marshalling only: torch tensors are checked for dtype, shape,
device and contiguity and passed as raw device pointers together with the
current CUDA stream. Every step of the computation runs in the CUDA library;
there is no fallback. If the library is missing the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

PDA_OK, PDA_EINVAL, PDA_EUNSUPPORTED, PDA_ENOMEM, PDA_ECUDA, PDA_EALIAS, PDA_EDEVICE = (
    0, -1, -2, -3, -4, -5, -6)
PDA_BF16, PDA_FP16, PDA_F32 = 0, 1, 2
ABI_VERSION = 2

_STATUS_NAMES = {0: "PDA_OK", -1: "PDA_EINVAL", -2: "PDA_EUNSUPPORTED", -3: "PDA_ENOMEM",
                 -4: "PDA_ECUDA", -5: "PDA_EALIAS", -6: "PDA_EDEVICE"}
_DT = {torch.bfloat16: PDA_BF16, torch.float16: PDA_FP16, torch.float32: PDA_F32}

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpaged_decode_attn.so")

# Every function the header declares (tests check the library exports them).
EXPORTS = [
    "paged_decode_attn_abi_version",
    "paged_decode_attn_last_error",
    "paged_decode_attn_create",
    "paged_decode_attn_destroy",
    "paged_decode_attn_run",
    "paged_decode_attn_run_ex",
    "paged_decode_attn_run_scaled",
    "paged_decode_attn_plan",
    "paged_decode_attn_launch_shape",
    "paged_decode_attn_merge",
    "paged_decode_attn_validate",
    "paged_decode_attn_check_device_error",
    "paged_decode_attn_run_noalloc",
    "paged_decode_attn_rope_kv_write",
    "paged_decode_attn_copy_blocks",
    "paged_decode_attn_gather_kv",
    "paged_decode_attn_scatter_kv",
    "paged_decode_attn_remap_table",
]


class PDAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("block_size", ctypes.c_int),
                ("dtype", ctypes.c_int), ("max_batch", ctypes.c_int),
                ("max_blocks_per_seq", ctypes.c_int), ("max_splits", ctypes.c_int),
                ("device", ctypes.c_int), ("kv_fp8", ctypes.c_int)]


_lib = None
_lock = threading.Lock()


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library (built by ``paged_gqa_decode_attention_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"CUDA library {p} is missing: run paged_gqa_decode_attention_gb300.build.build()")
        lib = ctypes.CDLL(p)
        P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.paged_decode_attn_abi_version.argtypes = []
        lib.paged_decode_attn_abi_version.restype = I
        lib.paged_decode_attn_last_error.argtypes = []
        lib.paged_decode_attn_last_error.restype = ctypes.c_char_p
        lib.paged_decode_attn_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(P)]
        lib.paged_decode_attn_create.restype = I
        lib.paged_decode_attn_destroy.argtypes = [P]
        lib.paged_decode_attn_destroy.restype = None
        lib.paged_decode_attn_run.argtypes = [P, P, P, P, P, P, I, I, I64, F, P, P]
        lib.paged_decode_attn_run.restype = I
        lib.paged_decode_attn_run_ex.argtypes = [P, P, P, P, P, P, I, I, I64, F, P, P, I, I, I]
        lib.paged_decode_attn_run_ex.restype = I
        lib.paged_decode_attn_run_scaled.argtypes = [P, P, P, P, P, P, I, I, I64, F, P, P, I, P,
                                                     P, I, I, I]
        lib.paged_decode_attn_run_scaled.restype = I
        lib.paged_decode_attn_plan.argtypes = [ctypes.POINTER(Config), I, I, I, I,
                                               ctypes.POINTER(I), ctypes.POINTER(I)]
        lib.paged_decode_attn_plan.restype = I
        lib.paged_decode_attn_launch_shape.argtypes = [P, I, I, I, I] + [ctypes.POINTER(I)] * 4
        lib.paged_decode_attn_launch_shape.restype = I
        lib.paged_decode_attn_merge.argtypes = [P, P, I, I, I, P, I, I, P]
        lib.paged_decode_attn_merge.restype = I
        lib.paged_decode_attn_validate.argtypes = [P, P, P, I, I, I64, P]
        lib.paged_decode_attn_validate.restype = I
        lib.paged_decode_attn_check_device_error.argtypes = [P, ctypes.POINTER(I),
                                                             ctypes.POINTER(I), P]
        lib.paged_decode_attn_check_device_error.restype = I
        lib.paged_decode_attn_run_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I64, F,
                                                      P, I, I, P]
        lib.paged_decode_attn_run_noalloc.restype = I
        lib.paged_decode_attn_rope_kv_write.argtypes = [P, I64, P, I64, P, I64, P, P, P, I, I, I,
                                                        I, I, I, I, I, P, I64, P, P, I64, P, I,
                                                        P]
        lib.paged_decode_attn_rope_kv_write.restype = I
        lib.paged_decode_attn_copy_blocks.argtypes = [P, P, I64, I64, P, I, P, I, P]
        lib.paged_decode_attn_copy_blocks.restype = I
        lib.paged_decode_attn_gather_kv.argtypes = [P, P, I64, I, I64, P, I, P, P, I, I, P, P, P,
                                                    I, P]
        lib.paged_decode_attn_gather_kv.restype = I
        lib.paged_decode_attn_scatter_kv.argtypes = [P, P, I64, I64, P, P, P, I64, P, I, P]
        lib.paged_decode_attn_scatter_kv.restype = I
        lib.paged_decode_attn_remap_table.argtypes = [P, I, I, P, I, P, I64, P, I, P]
        lib.paged_decode_attn_remap_table.restype = I
        if lib.paged_decode_attn_abi_version() != ABI_VERSION:
            raise RuntimeError("ABI version mismatch between binding and library")
        if path is None:
            _lib = lib
        return lib


def _check(lib, status: int):
    if status != PDA_OK:
        raise PDAError(status, lib.paged_decode_attn_last_error().decode())


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _dev_ptr(t: torch.Tensor, name: str, dtype=None) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def make_config(num_q_heads: int, num_kv_heads: int, head_dim: int = 128, block_size: int = 16,
                dtype=torch.bfloat16, max_batch: int = 256, max_blocks_per_seq: int = 4096,
                max_splits: int = 64, device: int = 0, kv_fp8: bool = False) -> Config:
    return Config(num_q_heads, num_kv_heads, head_dim, block_size, _DT[dtype], max_batch,
                  max_blocks_per_seq, max_splits, device, int(bool(kv_fp8)))


def plan(config: Config, num_sms: int, batch: int, max_blocks: int,
         max_context_len_hint: int = 0) -> tuple[int, int]:
    """(num_splits, chunk_pages) the split heuristic picks (host only)."""
    lib = load_library()
    s, c = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib, lib.paged_decode_attn_plan(ctypes.byref(config), num_sms, batch, max_blocks,
                                           max_context_len_hint, ctypes.byref(s),
                                           ctypes.byref(c)))
    return s.value, c.value


class PagedDecodeAttention:
    """One library handle: fixed geometry, owns the split-K workspace."""

    def __init__(self, num_q_heads: int, num_kv_heads: int, head_dim: int = 128,
                 block_size: int = 16, dtype=torch.bfloat16, max_batch: int = 256,
                 max_blocks_per_seq: int = 4096, max_splits: int = 64, device=None,
                 kv_fp8: bool = False):
        self.lib = load_library()
        if device is None:
            device = torch.cuda.current_device()
        if isinstance(device, torch.device):
            device = device.index if device.index is not None else torch.cuda.current_device()
        self.device = int(device)
        self.dtype = dtype
        self.kv_fp8 = bool(kv_fp8)
        self.config = make_config(num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                                  max_batch, max_blocks_per_seq, max_splits, self.device,
                                  self.kv_fp8)
        h = ctypes.c_void_p(None)
        _check(self.lib, self.lib.paged_decode_attn_create(ctypes.byref(self.config),
                                                           ctypes.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            self.lib.paged_decode_attn_destroy(self.handle)
            self.handle = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def run(self, q, k_cache, v_cache, block_table, context_lens, scale: float | None = None,
            out=None, num_splits: int = 0, max_context_len_hint: int = 0, out_dtype=None,
            stream=None, k_scale=None, v_scale=None):
        """out[B, Hq, D] = paged decode attention; asynchronous on ``stream``
        (default: torch's current stream). With FP8 caches (kv_fp8), k_cache
        and v_cache are torch.float8_e4m3fn (or uint8) tensors; k_scale and
        v_scale are fp32 device tensors of Hkv (per kv head) or 1 values."""
        c = self.config
        B = q.shape[0]
        if scale is None:
            scale = 1.0 / math.sqrt(c.head_dim)
        if out_dtype is None:
            out_dtype = self.dtype
        if out is None:
            out = torch.empty((B, c.num_q_heads, c.head_dim), dtype=out_dtype, device=q.device)
        if self.kv_fp8:
            for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
                if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
                    raise ValueError(f"{name} must be float8_e4m3fn or uint8 for an FP8 cache")
            kp, vp = _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache")
        else:
            kp = _dev_ptr(k_cache, "k_cache", self.dtype)
            vp = _dev_ptr(v_cache, "v_cache", self.dtype)
        per_head = 0
        for t in (k_scale, v_scale):
            if t is not None:
                if t.numel() not in (1, c.num_kv_heads):
                    raise ValueError("k_scale / v_scale must hold 1 or Hkv values")
                per_head = int(t.numel() == c.num_kv_heads and c.num_kv_heads > 1)
        if (k_scale is not None and v_scale is not None and
                k_scale.numel() != v_scale.numel()):
            raise ValueError("k_scale and v_scale must have the same size")
        args = (self.handle,
                _dev_ptr(q, "q", self.dtype), kp, vp,
                _dev_ptr(block_table, "block_table", torch.int32),
                _dev_ptr(context_lens, "context_lens", torch.int32),
                B, block_table.shape[1], k_cache.shape[0], float(scale),
                _dev_ptr(k_scale, "k_scale", torch.float32) if k_scale is not None else None,
                _dev_ptr(v_scale, "v_scale", torch.float32) if v_scale is not None else None,
                per_head, _dev_ptr(out, "out", out_dtype), _stream_ptr(stream),
                int(num_splits), int(max_context_len_hint), _DT[out_dtype])
        _check(self.lib, self.lib.paged_decode_attn_run_scaled(*args))
        return out

    def run_raw(self, q_ptr: int, k_ptr: int, v_ptr: int, table_ptr: int, lens_ptr: int,
                batch: int, max_blocks: int, num_blocks: int, scale: float, out_ptr: int,
                stream: int = 0) -> int:
        """paged_decode_attn_run on raw device pointers; returns the status."""
        return self.lib.paged_decode_attn_run(self.handle, q_ptr, k_ptr, v_ptr, table_ptr,
                                              lens_ptr, batch, max_blocks, num_blocks,
                                              float(scale), out_ptr, stream)

    def launch_shape(self, batch: int, max_blocks: int, num_splits: int = 0,
                     max_context_len_hint: int = 0) -> dict:
        """How a run with these sizes is launched: splits, chunk_pages, ctas,
        cluster (CTAs per thread-block cluster; 1 = no clusters)."""
        out = [ctypes.c_int(0) for _ in range(4)]
        _check(self.lib, self.lib.paged_decode_attn_launch_shape(
            self.handle, batch, max_blocks, max_context_len_hint, num_splits,
            *[ctypes.byref(o) for o in out]))
        return dict(zip(("splits", "chunk_pages", "ctas", "cluster"), (o.value for o in out)))

    def validate(self, block_table, context_lens, num_blocks: int, stream=None):
        B = context_lens.shape[0]
        _check(self.lib, self.lib.paged_decode_attn_validate(
            self.handle, _dev_ptr(block_table, "block_table", torch.int32),
            _dev_ptr(context_lens, "context_lens", torch.int32), B, block_table.shape[1],
            int(num_blocks), _stream_ptr(stream)))

    def check_device_error(self, stream=None) -> tuple[int, int]:
        code, detail = ctypes.c_int(0), ctypes.c_int(0)
        _check(self.lib, self.lib.paged_decode_attn_check_device_error(
            self.handle, ctypes.byref(code), ctypes.byref(detail), _stream_ptr(stream)))
        return code.value, detail.value


def merge(partial_o: torch.Tensor, partial_lse: torch.Tensor, out_dtype=torch.float32,
          out=None, stream=None) -> torch.Tensor:
    """LSE merge: partial_o [rows, S, D] fp32, partial_lse [rows, S] fp32
    (natural log, -inf = empty split) -> out [rows, D]."""
    lib = load_library()
    rows, S, D = partial_o.shape
    if out is None:
        out = torch.empty((rows, D), dtype=out_dtype, device=partial_o.device)
    dev = partial_o.device.index if partial_o.device.index is not None else 0
    _check(lib, lib.paged_decode_attn_merge(
        _dev_ptr(partial_o, "partial_o", torch.float32),
        _dev_ptr(partial_lse, "partial_lse", torch.float32), rows, S, D,
        _dev_ptr(out, "out", out_dtype), _DT[out_dtype], dev, _stream_ptr(stream)))
    return out


def _token_rows(t: torch.Tensor, name: str, dtype) -> tuple[int, int]:
    """Pointer and token stride (elements) of a [T, H, D] tensor whose heads
    are contiguous within a token (a packed tensor or a view into a fused
    projection output)."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != 3:
        raise ValueError(f"{name} must be [tokens, heads, head_dim]")
    T, H, D = t.shape
    if t.stride(2) != 1 or (H > 1 and t.stride(1) != D):
        raise ValueError(f"{name}: heads must be contiguous within a token")
    return t.data_ptr(), (t.stride(0) if T > 1 else H * D)


def rope_kv_write(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, positions: torch.Tensor,
                  slot_mapping: torch.Tensor, cos_sin_cache: torch.Tensor,
                  k_cache: torch.Tensor, v_cache: torch.Tensor, neox: bool = True,
                  q_out: torch.Tensor | None = None, err: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """RoPE on q and k plus the paged-cache write of k and v, one launch.

    q [T, Hq, D], k/v [T, Hkv, D] (bf16/fp16; token-strided views allowed),
    positions [T] int32, slot_mapping [T] int64 (< 0: no cache write),
    cos_sin_cache [max_position, rot_dim] fp32 (cosines then sines),
    k_cache/v_cache [num_blocks, block_size, Hkv, D]. Returns q_out (a new
    tensor, or ``q_out``; pass ``q_out=q`` to rotate in place). ``err`` is an
    optional int32 [2] device tensor receiving the first bad token."""
    lib = load_library()
    dt = q.dtype
    qp, qs = _token_rows(q, "q", dt)
    kp, ks = _token_rows(k, "k", dt)
    vp, vs = _token_rows(v, "v", dt)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, D) or v.shape != (T, Hkv, D):
        raise ValueError("k and v must be [T, Hkv, D] with q's T and D")
    if q_out is None:
        q_out = torch.empty((T, Hq, D), dtype=dt, device=q.device)
    qop, qos = _token_rows(q_out, "q_out", dt)
    if q_out.shape != q.shape:
        raise ValueError("q_out must have q's shape")
    if k_cache.shape != v_cache.shape or k_cache.dim() != 4 or k_cache.shape[2:] != (Hkv, D):
        raise ValueError("caches must be [num_blocks, block_size, Hkv, D]")
    if cos_sin_cache.dim() != 2:
        raise ValueError("cos_sin_cache must be [max_position, rot_dim]")
    max_pos, rot_dim = cos_sin_cache.shape
    if positions.shape != (T,) or slot_mapping.shape != (T,):
        raise ValueError("positions and slot_mapping must be [T]")
    dev = q.device.index if q.device.index is not None else 0
    _check(lib, lib.paged_decode_attn_rope_kv_write(
        qp, qs, kp, ks, vp, vs, _dev_ptr(positions, "positions", torch.int32),
        _dev_ptr(slot_mapping, "slot_mapping", torch.int64),
        _dev_ptr(cos_sin_cache, "cos_sin_cache", torch.float32), max_pos, rot_dim,
        int(bool(neox)), T, Hq, Hkv, D, _DT[dt], qop, qos, _dev_ptr(k_cache, "k_cache", dt),
        _dev_ptr(v_cache, "v_cache", dt), k_cache.shape[0] * k_cache.shape[1],
        _dev_ptr(err, "err", torch.int32) if err is not None else None, dev,
        _stream_ptr(stream)))
    return q_out


# ------------------------------ KV-cache movement ------------------------------

def _cache_geometry(k_cache: torch.Tensor, v_cache: torch.Tensor):
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype or k_cache.dim() != 4:
        raise ValueError("k_cache and v_cache must be [num_blocks, block_size, Hkv, D] alike")
    nb, bs = k_cache.shape[0], k_cache.shape[1]
    row_bytes = k_cache.shape[2] * k_cache.shape[3] * k_cache.element_size()
    return nb, bs, row_bytes


def _opt_err(err):
    return _dev_ptr(err, "err", torch.int32) if err is not None else None


def _device_of(t: torch.Tensor) -> int:
    return t.device.index if t.device.index is not None else torch.cuda.current_device()


def copy_blocks(k_cache, v_cache, pairs: torch.Tensor, err=None, stream=None):
    """Block pairs[i, 1] := block pairs[i, 0] in both caches (in place);
    pairs is an int64 [n, 2] device tensor."""
    lib = load_library()
    nb, bs, row_bytes = _cache_geometry(k_cache, v_cache)
    n = pairs.shape[0] if pairs.numel() else 0
    _check(lib, lib.paged_decode_attn_copy_blocks(
        _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), nb, bs * row_bytes,
        _dev_ptr(pairs, "pairs", torch.int64) if n else None, n, _opt_err(err),
        _device_of(k_cache), _stream_ptr(stream)))


def gather_kv(k_cache, v_cache, block_table, lens, cu_rows=None, max_len: int | None = None,
              k_out=None, v_out=None, err=None, stream=None):
    """Each sequence's tokens, in order, into contiguous [rows, Hkv, D] buffers
    (sequence b from row cu_rows[b]; default: exclusive prefix sums of lens,
    computed on the host from lens). Returns (k_out, v_out)."""
    lib = load_library()
    nb, bs, row_bytes = _cache_geometry(k_cache, v_cache)
    B = lens.shape[0]
    if cu_rows is None or max_len is None or k_out is None:
        lens_h = lens.cpu().to(torch.int64)
        if cu_rows is None:
            cu_rows = (torch.cumsum(lens_h, 0) - lens_h).to(k_cache.device)
        if max_len is None:
            max_len = int(lens_h.max()) if B else 0
        total = int(lens_h.sum())
    else:
        total = k_out.shape[0]
    shape = (total,) + tuple(k_cache.shape[2:])
    if k_out is None:
        k_out = torch.empty(shape, dtype=k_cache.dtype, device=k_cache.device)
        v_out = torch.empty(shape, dtype=k_cache.dtype, device=k_cache.device)
    _check(lib, lib.paged_decode_attn_gather_kv(
        _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), nb, bs, row_bytes,
        _dev_ptr(block_table, "block_table", torch.int32), block_table.shape[1],
        _dev_ptr(lens, "lens", torch.int32), _dev_ptr(cu_rows, "cu_rows", torch.int64), B,
        int(max_len), _dev_ptr(k_out, "k_out"), _dev_ptr(v_out, "v_out"), _opt_err(err),
        _device_of(k_cache), _stream_ptr(stream)))
    return k_out, v_out


def scatter_kv(k_rows, v_rows, slot_mapping, k_cache, v_cache, err=None, stream=None):
    """Row r of k_rows / v_rows ([n, Hkv, D]) into cache slot slot_mapping[r]
    (int64; < 0 skips), in place."""
    lib = load_library()
    nb, bs, row_bytes = _cache_geometry(k_cache, v_cache)
    if k_rows.dtype != k_cache.dtype or v_rows.dtype != k_cache.dtype:
        raise ValueError("rows and caches must share a dtype")
    n = k_rows.shape[0]
    _check(lib, lib.paged_decode_attn_scatter_kv(
        _dev_ptr(k_rows, "k_rows"), _dev_ptr(v_rows, "v_rows"), n, row_bytes,
        _dev_ptr(slot_mapping, "slot_mapping", torch.int64), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), nb * bs, _opt_err(err), _device_of(k_cache),
        _stream_ptr(stream)))


def remap_table(block_table, lens, block_size: int, new_id, err=None, stream=None):
    """In place: every used entry e of block_table becomes new_id[e]."""
    lib = load_library()
    _check(lib, lib.paged_decode_attn_remap_table(
        _dev_ptr(block_table, "block_table", torch.int32), block_table.shape[0],
        block_table.shape[1], _dev_ptr(lens, "lens", torch.int32), int(block_size),
        _dev_ptr(new_id, "new_id", torch.int32), new_id.shape[0], _opt_err(err),
        _device_of(block_table), _stream_ptr(stream)))
