"""Seeded synthetic inputs for paged decode attention.

This module only draws random numbers and arranges them into the paged
layout; it holds none of the attention arithmetic. Both the CUDA path and the
FP64 oracle consume what it returns, so it is the one piece they share.

Layout of every workload (the contract of the C ABI):
  q            [B, Hq, D]                     bf16 | fp16
  k_cache      [num_blocks, block_size, Hkv, D]  same dtype
  v_cache      [num_blocks, block_size, Hkv, D]  same dtype
  block_table  [B, max_blocks]                int32
  context_lens [B]                            int32

Integers (lengths, tables, masks) come from numpy's PCG64 so they are the
same on every host; floating values come from ``torch.randn`` with a seeded
generator on the device that holds the tensor, drawn in float32 and rounded
to the storage dtype with round-to-nearest-even.

The five workload families follow the shapes the Loom Kernels pages
benchmark (benchmark page, "Reproduce": the paged-decode attention sweep over
batches 1-8 x contexts 128-1024 at 32/8 heads, D 128, and the backend sweep
over batches 1/8/32 x contexts 16-64 x bf16/f16 x block sizes 16/32) and the
long-context and serving-scale cases this library targets.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclass
class Workload:
    name: str
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_table: torch.Tensor
    context_lens: torch.Tensor
    scale: float
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def num_q_heads(self) -> int:
        return self.q.shape[1]

    @property
    def head_dim(self) -> int:
        return self.q.shape[2]

    @property
    def num_kv_heads(self) -> int:
        return self.k_cache.shape[2]

    @property
    def block_size(self) -> int:
        return self.k_cache.shape[1]

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]

    @property
    def max_blocks(self) -> int:
        return self.block_table.shape[1]

    @property
    def dtype_name(self) -> str:
        return "bf16" if self.q.dtype == torch.bfloat16 else "fp16"

    def lens_list(self) -> list[int]:
        return [int(x) for x in self.context_lens.cpu().tolist()]

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes one call reads: sum_b L_b * 2 * Hkv * D * esz
        (no padding of partial pages, no re-reads, shared pages counted once
        per sequence that reads them)."""
        esz = self.k_cache.element_size()
        return sum(self.lens_list()) * 2 * self.num_kv_heads * self.head_dim * esz

    @property
    def kv_fp8(self) -> bool:
        return self.k_cache.element_size() == 1

    def unique_kv_bytes(self) -> int:
        """KV bytes of the distinct physical token slots read by one call."""
        bs = self.block_size
        seen: dict[int, int] = {}
        bt = self.block_table.cpu().numpy()
        for b, L in enumerate(self.lens_list()):
            pages = (L + bs - 1) // bs
            for p in range(pages):
                blk = int(bt[b, p])
                used = min(bs, L - p * bs)
                seen[blk] = max(seen.get(blk, 0), used)
        esz = self.k_cache.element_size()
        return sum(seen.values()) * 2 * self.num_kv_heads * self.head_dim * esz

    def to(self, device) -> "Workload":
        meta = {k: (v.to(device) if isinstance(v, torch.Tensor) else v)
                for k, v in self.meta.items()}
        return Workload(self.name, self.q.to(device), self.k_cache.to(device),
                        self.v_cache.to(device), self.block_table.to(device),
                        self.context_lens.to(device), self.scale, meta)


# ---------------------------------------------------------------------------
# random helpers
# ---------------------------------------------------------------------------

def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream]))


def _randn(shape, std: float, dtype: torch.dtype, device, seed: int, stream: int,
           row_scale: torch.Tensor | None = None) -> torch.Tensor:
    """N(0, std^2) drawn in float32 and rounded to ``dtype``, in chunks so that
    multi-GiB pools never need a float32 copy of the whole tensor.
    ``row_scale`` (float32, one value per leading-dim row) multiplies rows
    before rounding."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1_000_003 + stream)
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(shape[0], -1)
    rows_per_chunk = max(1, (1 << 26) // max(1, flat.shape[1]))
    for r0 in range(0, flat.shape[0], rows_per_chunk):
        r1 = min(flat.shape[0], r0 + rows_per_chunk)
        x = torch.randn((r1 - r0, flat.shape[1]), generator=gen, device=device,
                        dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        if row_scale is not None:
            x.mul_(row_scale[r0:r1].to(device).view(-1, 1))
        flat[r0:r1].copy_(x)
    return out


def _assemble(name, B, Hq, Hkv, D, bs, num_blocks, tables, lens, dtype, std, seed, device,
              k_row_scale=None, meta=None) -> Workload:
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    q = _randn((B, Hq, D), std, dt, device, seed, 1)
    # K/V are drawn through their [num_blocks * block_size, Hkv * D] view so
    # that ``k_row_scale`` can scale single (block, slot) rows
    k = _randn((num_blocks * bs, Hkv * D), std, dt, device, seed, 2, row_scale=k_row_scale)
    v = _randn((num_blocks * bs, Hkv * D), std, dt, device, seed, 3)
    k = k.view(num_blocks, bs, Hkv, D)
    v = v.view(num_blocks, bs, Hkv, D)
    bt = torch.as_tensor(np.ascontiguousarray(tables, dtype=np.int32)).to(device)
    cl = torch.as_tensor(np.ascontiguousarray(lens, dtype=np.int32)).to(device)
    return Workload(name, q, k, v, bt, cl, 1.0 / math.sqrt(D), dict(meta or {}))


def _tables_without_replacement(rng, lens, bs, max_blocks, num_blocks):
    """Each sequence's pages drawn without replacement from a shuffled pool;
    entries past a sequence's last page hold further (unused) pool entries."""
    need = sum((L + bs - 1) // bs for L in lens)
    if need > num_blocks:
        raise ValueError("pool too small for the requested contexts")
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = np.zeros((len(lens), max_blocks), dtype=np.int32)
    pos = 0
    for b, L in enumerate(lens):
        pages = (L + bs - 1) // bs
        tables[b, :pages] = perm[pos:pos + pages]
        pos += pages
    # fill the unused tail of every row with valid but unread block ids
    filler = rng.integers(0, num_blocks, size=tables.shape, dtype=np.int32)
    for b, L in enumerate(lens):
        pages = (L + bs - 1) // bs
        tables[b, pages:] = filler[b, pages:]
    return tables


# ---------------------------------------------------------------------------
# the five workload families
# ---------------------------------------------------------------------------

def tiny(seed: int = 0, device="cpu") -> Workload:
    """B=1, Hq 32, Hkv 8, D 128, block 16, context 32 (2 pages); the table row
    is a random permutation of the 64 physical blocks."""
    rng = _rng(seed, 0)
    B, Hq, Hkv, D, bs, L, nb = 1, 32, 8, 128, 16, 32, 64
    table = rng.permutation(nb).astype(np.int32).reshape(1, nb)
    return _assemble("tiny_b1_l32", B, Hq, Hkv, D, bs, nb, table, [L], "bf16", 1.0, seed,
                     device)


def short_batch(seed: int = 0, block_size: int = 16, dtype: str = "bf16",
                device="cpu") -> Workload:
    """B=32, 32/8/128, context lengths uniform in [16, 64], 4096 physical
    blocks, pages drawn from a shuffled pool."""
    rng = _rng(seed, 1)
    B, Hq, Hkv, D, nb = 32, 32, 8, 128, 4096
    lens = rng.integers(16, 65, size=B).tolist()
    max_blocks = (64 + block_size - 1) // block_size
    tables = _tables_without_replacement(rng, lens, block_size, max_blocks, nb)
    return _assemble(f"short_b32_bs{block_size}_{dtype}", B, Hq, Hkv, D, block_size, nb, tables,
                     lens, dtype, 1.0, seed, device)


def mid_ragged(seed: int = 0, device="cpu") -> Workload:
    """B=8, 32/8/128, block 16, context lengths from {128, 256, 512, 1024};
    the K row of 1% of the (sequence, position) slots is scaled by 3 before
    rounding, which makes the softmax peaky."""
    rng = _rng(seed, 2)
    B, Hq, Hkv, D, bs, nb = 8, 32, 8, 128, 16, 4096
    lens = rng.choice([128, 256, 512, 1024], size=B).tolist()
    max_blocks = 1024 // bs
    tables = _tables_without_replacement(rng, lens, bs, max_blocks, nb)
    scale_rows = np.ones(nb * bs, dtype=np.float32)
    for b, L in enumerate(lens):
        hit = rng.random(L) < 0.01
        for t in np.nonzero(hit)[0]:
            scale_rows[int(tables[b, t // bs]) * bs + int(t % bs)] = 3.0
    # one scale per (block, slot) row of the [nb * bs, Hkv * D] view
    row_scale = torch.from_numpy(scale_rows)
    return _assemble("mid_ragged_b8", B, Hq, Hkv, D, bs, nb, tables, lens, "bf16", 1.0, seed,
                     device, k_row_scale=row_scale,
                     meta={"peaky_slots": int((scale_rows != 1.0).sum())})


LONG_POOL_BLOCKS = 655_360  # 40 GiB of K+V at block 16, Hkv 8, D 128, bf16


def long_context(seed: int = 0, batch: int = 4, context: int = 32768,
                 num_blocks: int = LONG_POOL_BLOCKS, device="cpu",
                 kv_fp8: bool = False) -> Workload:
    """Long-context split-K case: B in {1, 4} x context in {8192, 32768},
    32/8/128, block 16, bf16; random tables over a pool of ``num_blocks``
    blocks (the full-size pool is 40 GiB of K+V, 20 GiB as FP8)."""
    rng = _rng(seed, 3)
    Hq, Hkv, D, bs = 32, 8, 128, 16
    lens = [context] * batch
    max_blocks = (context + bs - 1) // bs
    tables = _tables_without_replacement(rng, lens, bs, max_blocks, num_blocks)
    wl = _assemble(f"long_b{batch}_l{context}", batch, Hq, Hkv, D, bs, num_blocks, tables,
                   lens, "bf16", 1.0, seed, device, meta={"pool_blocks": num_blocks})
    return to_fp8_kv(wl) if kv_fp8 else wl


def leading(wl: Workload, batch: int, context: int) -> Workload:
    """The first ``batch`` sequences of ``wl`` cut to their first ``context``
    tokens, over the same cache pool (views, no copies): the smaller
    long-context shapes taken from one full-size pool."""
    bs = wl.block_size
    pages = (context + bs - 1) // bs
    if batch > wl.batch or pages > wl.max_blocks:
        raise ValueError("leading(): larger than the workload it is cut from")
    lens = torch.clamp(wl.context_lens[:batch], max=context).contiguous()
    name = wl.name.split("_b")[0] + f"_b{batch}_l{context}" + ("_fp8" if wl.kv_fp8 else "")
    return Workload(name, wl.q[:batch].contiguous(), wl.k_cache, wl.v_cache,
                    wl.block_table[:batch, :pages].contiguous(), lens, wl.scale, dict(wl.meta))


def to_fp8_kv(wl: Workload) -> Workload:
    """The same workload with FP8 (E4M3) K/V caches: per kv head h, scale_h =
    max |x| over the pool / 448 (so the largest value maps to the largest
    E4M3 value) and the cache holds RNE(x / scale_h) (torch's saturating
    conversion). The scales go to meta["k_scale"], meta["v_scale"] (fp32
    [Hkv]). Works in row chunks so multi-GiB pools need no fp32 copy."""
    Hkv, D = wl.num_kv_heads, wl.head_dim
    out = {}
    for name, cache in (("k", wl.k_cache), ("v", wl.v_cache)):
        flat = cache.view(-1, Hkv, D)
        rows = flat.shape[0]
        step = max(1, (1 << 26) // (Hkv * D))
        amax = torch.zeros(Hkv, dtype=torch.float32, device=cache.device)
        for r0 in range(0, rows, step):
            amax = torch.maximum(amax, flat[r0:r0 + step].float().abs().amax(dim=(0, 2)))
        sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        q8 = torch.empty(flat.shape, dtype=torch.float8_e4m3fn, device=cache.device)
        for r0 in range(0, rows, step):
            q8[r0:r0 + step] = (flat[r0:r0 + step].float() / sc.view(1, Hkv, 1)).to(
                torch.float8_e4m3fn)
        out[name] = (q8.view(cache.shape), sc)
    meta = dict(wl.meta)
    meta["k_scale"], meta["v_scale"] = out["k"][1], out["v"][1]
    return Workload(wl.name + "_fp8", wl.q, out["k"][0], out["v"][0], wl.block_table,
                    wl.context_lens, wl.scale, meta)


def serving_mix(seed: int = 0, batch: int = 128, max_context: int = 4096,
                device="cpu") -> Workload:
    """B=128, Hq 64, Hkv 8 (G = 8), D 128, block 32; context lengths
    log-uniform in [32, max_context]; values N(0, 0.5^2); every even-indexed
    sequence starts with min(32, floor(L / 32)) pages of one shared prefix
    (aliased block-table entries), the rest of its pages private."""
    rng = _rng(seed, 4)
    Hq, Hkv, D, bs = 64, 8, 128, 32
    lo, hi = math.log(32), math.log(max_context)
    lens = [int(min(max_context, max(32, math.floor(math.exp(u)))))
            for u in rng.uniform(lo, hi, size=batch)]
    max_blocks = (max_context + bs - 1) // bs
    shared = 32
    prefix = [min(shared, L // bs) if b % 2 == 0 else 0 for b, L in enumerate(lens)]
    private = [(L + bs - 1) // bs - p for L, p in zip(lens, prefix)]
    nb = shared + sum(private)
    perm = rng.permutation(nb).astype(np.int32)
    shared_ids, private_ids = perm[:shared], perm[shared:]
    tables = np.zeros((batch, max_blocks), dtype=np.int32)
    pos = 0
    for b in range(batch):
        p = prefix[b]
        tables[b, :p] = shared_ids[:p]
        tables[b, p:p + private[b]] = private_ids[pos:pos + private[b]]
        pos += private[b]
        tables[b, p + private[b]:] = rng.integers(0, nb, size=max_blocks - p - private[b])
    return _assemble(f"serving_b{batch}_g8", batch, Hq, Hkv, D, bs, nb, tables, lens, "bf16",
                     0.5, seed, device, meta={"shared_prefix_pages": prefix})


def custom(seed: int, B: int, Hq: int, Hkv: int, D: int, block_size: int, lens,
           dtype: str = "bf16", num_blocks: int | None = None, std: float = 1.0,
           device="cpu") -> Workload:
    """Any geometry: pages drawn without replacement from a pool of
    ``num_blocks`` (default: exactly the pages needed plus 8)."""
    rng = _rng(seed, 5)
    lens = [int(x) for x in lens]
    max_blocks = max(1, max((L + block_size - 1) // block_size for L in lens) if lens else 1)
    need = sum((L + block_size - 1) // block_size for L in lens)
    nb = num_blocks if num_blocks is not None else need + 8
    tables = _tables_without_replacement(rng, lens, block_size, max_blocks, nb)
    return _assemble(f"custom_b{B}_{Hq}x{Hkv}_d{D}_bs{block_size}", B, Hq, Hkv, D, block_size,
                     nb, tables, lens, dtype, std, seed, device)


# ---------------------------------------------------------------------------
# host views for the oracle (plumbing only: copies and index remapping)
# ---------------------------------------------------------------------------

def bits(t: torch.Tensor) -> np.ndarray:
    """Raw storage patterns: numpy uint16 for bf16/fp16 tensors, uint8 for
    FP8 tensors."""
    t = t.detach().contiguous().cpu()
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def host_arrays(wl: Workload):
    """(q, k, v, block_table, context_lens) as numpy arrays on the host."""
    return (bits(wl.q), bits(wl.k_cache), bits(wl.v_cache),
            wl.block_table.cpu().numpy().astype(np.int32),
            wl.context_lens.cpu().numpy().astype(np.int32))


def compact_for_rows(wl: Workload, seqs) -> tuple:
    """Copy only the pages that sequences ``seqs`` read to the host, with the
    block table remapped to the compacted pool. Returns
    (q, k, v, block_table, context_lens) for those sequences, in that order,
    as numpy arrays. Used to check sampled rows of multi-GiB workloads."""
    seqs = [int(s) for s in seqs]
    bs = wl.block_size
    lens = wl.context_lens.cpu().numpy().astype(np.int64)
    bt = wl.block_table.cpu().numpy()
    used, tables = [], []
    index: dict[int, int] = {}
    for s in seqs:
        pages = int((lens[s] + bs - 1) // bs)
        row = np.zeros(bt.shape[1], dtype=np.int32)
        for p in range(pages):
            blk = int(bt[s, p])
            if blk not in index:
                index[blk] = len(used)
                used.append(blk)
            row[p] = index[blk]
        tables.append(row)
    ids = torch.as_tensor(used if used else [0], dtype=torch.int64, device=wl.k_cache.device)
    k = bits(wl.k_cache.index_select(0, ids))
    v = bits(wl.v_cache.index_select(0, ids))
    q = bits(wl.q[seqs])
    return q, k, v, np.stack(tables).astype(np.int32), lens[seqs].astype(np.int32)


# ---------------------------------------------------------------------------
# RoPE + paged-KV write inputs
# ---------------------------------------------------------------------------

@dataclass
class RopeWorkload:
    """Inputs of one RoPE + paged-KV write call.

    ``qkv`` is the fused projection output [T, (Hq + 2 Hkv) * D]; q, k and v
    are token-strided views into it (the layout a fused QKV projection
    produces). ``cos_sin`` [max_position, rot_dim] float32 holds cos(pos * f_j)
    then sin(pos * f_j) with f_j = theta^(-2j / rot_dim): the usual rotary
    frequency schedule, precomputed once per model like a weight, and an
    input to both the kernel and the oracle."""
    name: str
    qkv: torch.Tensor
    positions: torch.Tensor     # [T] int32
    slot_mapping: torch.Tensor  # [T] int64
    cos_sin: torch.Tensor       # [max_position, rot_dim] float32
    k_cache: torch.Tensor       # [num_blocks, block_size, Hkv, D]
    v_cache: torch.Tensor
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    neox: bool = True
    meta: dict = field(default_factory=dict)

    def _part(self, h0: int, h1: int) -> torch.Tensor:
        D = self.head_dim
        return self.qkv[:, h0 * D:h1 * D].view(-1, h1 - h0, D)

    @property
    def q(self) -> torch.Tensor:
        return self._part(0, self.num_q_heads)

    @property
    def k(self) -> torch.Tensor:
        return self._part(self.num_q_heads, self.num_q_heads + self.num_kv_heads)

    @property
    def v(self) -> torch.Tensor:
        Hq, Hkv = self.num_q_heads, self.num_kv_heads
        return self._part(Hq + Hkv, Hq + 2 * Hkv)

    @property
    def num_tokens(self) -> int:
        return self.qkv.shape[0]

    @property
    def rot_dim(self) -> int:
        return self.cos_sin.shape[1]

    def moved_bytes(self) -> int:
        """Bytes the operation must move: q, k, v read; q_out and the k/v
        cache rows written (padding tokens write no cache rows); one table row
        and the position and slot of every token."""
        esz = self.qkv.element_size()
        T, Hq, Hkv, D = self.num_tokens, self.num_q_heads, self.num_kv_heads, self.head_dim
        written = int((self.slot_mapping >= 0).sum())
        return (T * (Hq + 2 * Hkv) * D * esz + T * Hq * D * esz + written * 2 * Hkv * D * esz
                + T * self.rot_dim * 4 + T * 12)

    def to(self, device) -> "RopeWorkload":
        return RopeWorkload(self.name, self.qkv.to(device), self.positions.to(device),
                            self.slot_mapping.to(device), self.cos_sin.to(device),
                            self.k_cache.to(device), self.v_cache.to(device), self.num_q_heads,
                            self.num_kv_heads, self.head_dim, self.neox, dict(self.meta))


def rope_cos_sin(max_position: int, rot_dim: int, theta: float) -> torch.Tensor:
    """[max_position, rot_dim] float32: cosines then sines of pos * theta^(-2j/rot_dim),
    evaluated in float64 and rounded once."""
    j = np.arange(rot_dim // 2, dtype=np.float64)
    freq = theta ** (-2.0 * j / rot_dim)
    ang = np.arange(max_position, dtype=np.float64)[:, None] * freq[None, :]
    return torch.from_numpy(np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32))


def rope_batch(seed: int = 0, tokens: int = 512, Hq: int = 14, Hkv: int = 2, D: int = 64,
               rot_dim: int | None = None, theta: float = 1.0e6, max_position: int = 32768,
               block_size: int = 16, num_blocks: int | None = None, dtype: str = "bf16",
               mode: str = "decode", neox: bool = True, pad_frac: float = 0.0,
               device="cpu") -> RopeWorkload:
    """Seeded RoPE + KV-write inputs. Defaults: the Qwen2.5-0.5B attention
    geometry (14 query heads, 2 kv heads, D 64, full-width rotate-halves
    rotary with theta 1e6, 32768 positions), bf16 N(0, 1) activations.

    mode "decode": one new token per sequence, positions uniform in
    [0, max_position), distinct random cache slots. mode "prefill": one
    sequence of ``tokens`` tokens at positions 0 .. T-1 stored through a
    random block table. ``pad_frac`` of the tokens get slot -1 (padding).
    The cache pool starts filled with N(0, 1) values."""
    rot_dim = D if rot_dim is None else rot_dim
    dt = DTYPES[dtype]
    rng = _rng(seed, 40)
    T = tokens
    if num_blocks is None:
        num_blocks = max(64, 2 * ((T + block_size - 1) // block_size))
    slots_total = num_blocks * block_size
    if mode == "decode":
        pos = rng.integers(0, max_position, size=T)
        slots = rng.permutation(slots_total)[:T]
    elif mode == "prefill":
        if T > max_position:
            raise ValueError("prefill longer than the position table")
        pos = np.arange(T)
        pages = rng.permutation(num_blocks)[: (T + block_size - 1) // block_size]
        slots = pages[np.arange(T) // block_size] * block_size + np.arange(T) % block_size
    else:
        raise ValueError(mode)
    if T > slots_total:
        raise ValueError("cache pool smaller than the token count")
    slots = slots.astype(np.int64)
    if pad_frac > 0:
        slots[rng.random(T) < pad_frac] = -1
    qkv = _randn((T, (Hq + 2 * Hkv) * D), 1.0, dt, device, seed, 41)
    kc = _randn((num_blocks * block_size, Hkv * D), 1.0, dt, device, seed, 42)
    vc = _randn((num_blocks * block_size, Hkv * D), 1.0, dt, device, seed, 43)
    return RopeWorkload(
        f"rope_{mode}_t{T}_{Hq}x{Hkv}x{D}", qkv,
        torch.as_tensor(pos.astype(np.int32)).to(device), torch.as_tensor(slots).to(device),
        rope_cos_sin(max_position, rot_dim, theta).to(device),
        kc.view(num_blocks, block_size, Hkv, D), vc.view(num_blocks, block_size, Hkv, D),
        Hq, Hkv, D, neox, {"mode": mode, "theta": theta, "block_size": block_size,
                           "dtype": dtype})
