// KV-cache movement (landing page, "Next boundaries": KV-cache movement -
// scheduler-facing block copy, gather, scatter and compact work for prefix
// reuse and preemption). A cache is [num_blocks, block_size, Hkv, D] of any
// element type; these kernels move raw bytes, so every result is an exact
// copy:
//   copy_blocks  block dst := block src for each (src, dst) pair, K and V;
//   gather       each sequence's tokens t < lens[b], through its block
//                table, into contiguous rows starting at cu_rows[b];
//   scatter      contiguous rows into cache slots (slot < 0: skipped);
//   remap_table  table[b, p] := new_id[table[b, p]] for the pages in use
//                (the table update of a compaction).
// Memory-bound streaming: 16-byte vector loads and stores, each thread with
// kVec vectors in flight, grids sized to the work. Out-of-range ids are
// skipped and recorded in an optional error word; nothing faults.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <string>

#include "paged_decode_attn.h"
#include "pda_internal.h"

namespace pda {
namespace {

constexpr int kMoveThreads = 256;
constexpr int kVec = 4;                                    // 16-byte vectors per thread
constexpr int kTileBytes = kMoveThreads * kVec * 16;       // 16 KiB per CTA step

__device__ __forceinline__ void record(int* err, int code, int detail) {
  if (err != nullptr && atomicCAS(err, 0, code) == 0) err[1] = detail;
}

// Copies `bytes` (a multiple of 16) from src to dst; the CTA's threads each
// move up to kVec vectors per step, loads before stores.
__device__ __forceinline__ void copy_span(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                          int64_t n_vec, int64_t v0) {
  uint4 r[kVec];
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const int64_t v = v0 + (int64_t)i * kMoveThreads + threadIdx.x;
    if (v < n_vec) r[i] = __ldcs(src + v);
  }
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const int64_t v = v0 + (int64_t)i * kMoveThreads + threadIdx.x;
    if (v < n_vec) __stcs(dst + v, r[i]);
  }
}

// grid (tiles per block, pairs): blockIdx.y = pair, blockIdx.x = 16 KiB tile
__global__ void __launch_bounds__(kMoveThreads) copy_blocks_kernel(
    uint8_t* k, uint8_t* v, int64_t num_blocks, int64_t block_bytes, const int64_t* pairs,
    int* err) {
  const int64_t src = __ldg(pairs + 2 * (int64_t)blockIdx.y);
  const int64_t dst = __ldg(pairs + 2 * (int64_t)blockIdx.y + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record(err, kErrBlockId, (int)blockIdx.y);
    return;
  }
  const int64_t n_vec = block_bytes / 16;
  const int64_t v0 = (int64_t)blockIdx.x * (kTileBytes / 16);
  copy_span(reinterpret_cast<uint4*>(k + dst * block_bytes),
            reinterpret_cast<const uint4*>(k + src * block_bytes), n_vec, v0);
  copy_span(reinterpret_cast<uint4*>(v + dst * block_bytes),
            reinterpret_cast<const uint4*>(v + src * block_bytes), n_vec, v0);
}

// One warp copies one row of `n_vec` 16-byte vectors, kVec per lane in flight.
__device__ __forceinline__ void copy_row(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                         int64_t n_vec, int lane) {
  for (int64_t w0 = 0; w0 < n_vec; w0 += 32 * kVec) {
    uint4 r[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const int64_t w = w0 + i * 32 + lane;
      if (w < n_vec) r[i] = __ldcs(src + w);
    }
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      const int64_t w = w0 + i * 32 + lane;
      if (w < n_vec) __stcs(dst + w, r[i]);
    }
  }
}

constexpr int kMoveWarps = kMoveThreads / 32;

// grid (token tiles, sequences): a CTA copies rows_per_cta consecutive tokens
// of sequence blockIdx.y to their contiguous rows, one warp per row.
__global__ void __launch_bounds__(kMoveThreads) gather_kernel(
    const uint8_t* k, const uint8_t* v, int64_t num_blocks, int block_size, int64_t row_bytes,
    const int32_t* table, int max_blocks, const int32_t* lens, const int64_t* cu_rows,
    int max_len, int rows_per_cta, uint8_t* ko, uint8_t* vo, int* err) {
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int L = __ldg(lens + b);
  if (L > max_len || L < 0) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record(err, kErrContextLen, b);
    L = L < 0 ? 0 : max_len;
  }
  const int t0 = blockIdx.x * rows_per_cta;
  const int t1 = min(L, t0 + rows_per_cta);
  const int64_t row0 = __ldg(cu_rows + b);
  const int64_t n_vec = row_bytes / 16;
  for (int t = t0 + warp; t < t1; t += kMoveWarps) {
    const int32_t blk = __ldg(table + (int64_t)b * max_blocks + t / block_size);
    if (blk < 0 || blk >= num_blocks) {
      if (lane == 0) record(err, kErrBlockId, b);
      continue;
    }
    const int64_t slot = (int64_t)blk * block_size + t % block_size;
    copy_row(reinterpret_cast<uint4*>(ko + (row0 + t) * row_bytes),
             reinterpret_cast<const uint4*>(k + slot * row_bytes), n_vec, lane);
    copy_row(reinterpret_cast<uint4*>(vo + (row0 + t) * row_bytes),
             reinterpret_cast<const uint4*>(v + slot * row_bytes), n_vec, lane);
  }
}

// grid over tiles of rows_per_cta rows: row r goes to slot slot_mapping[r],
// one warp per row.
__global__ void __launch_bounds__(kMoveThreads) scatter_kernel(
    const uint8_t* kr, const uint8_t* vr, int64_t n_rows, int64_t row_bytes,
    const int64_t* slots, int rows_per_cta, uint8_t* k, uint8_t* v, int64_t num_slots,
    int* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r0 = (int64_t)blockIdx.x * rows_per_cta;
  const int64_t r1 = min(n_rows, r0 + rows_per_cta);
  const int64_t n_vec = row_bytes / 16;
  for (int64_t r = r0 + warp; r < r1; r += kMoveWarps) {
    const int64_t slot = __ldg(slots + r);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (lane == 0) record(err, kErrSlot, (int)r);
      continue;
    }
    copy_row(reinterpret_cast<uint4*>(k + slot * row_bytes),
             reinterpret_cast<const uint4*>(kr + r * row_bytes), n_vec, lane);
    copy_row(reinterpret_cast<uint4*>(v + slot * row_bytes),
             reinterpret_cast<const uint4*>(vr + r * row_bytes), n_vec, lane);
  }
}

__global__ void __launch_bounds__(kMoveThreads) remap_kernel(int32_t* table, int batch,
                                                             int max_blocks, const int32_t* lens,
                                                             int block_size,
                                                             const int32_t* new_id,
                                                             int64_t num_blocks, int* err) {
  const int64_t i = (int64_t)blockIdx.x * kMoveThreads + threadIdx.x;
  if (i >= (int64_t)batch * max_blocks) return;
  const int b = (int)(i / max_blocks), p = (int)(i - (int64_t)b * max_blocks);
  int L = __ldg(lens + b);
  L = L < 0 ? 0 : (L > max_blocks * block_size ? max_blocks * block_size : L);
  if (p >= (L + block_size - 1) / block_size) return;
  const int32_t e = table[i];
  if (e < 0 || e >= num_blocks) {
    record(err, kErrBlockId, b);
    return;
  }
  table[i] = __ldg(new_id + e);
}

int fail(int code, const std::string& msg) { return set_last_error(code, msg.c_str()); }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Selects `device` for the scope and restores the caller's.
struct Dev {
  int prev = -1;
  cudaError_t err = cudaSuccess;
  explicit Dev(int d) {
    err = cudaGetDevice(&prev);
    if (err == cudaSuccess && prev != d) err = cudaSetDevice(d);
    else prev = -1;
  }
  ~Dev() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

int launched(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PDA_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return PDA_OK;
}

}  // namespace
}  // namespace pda

using pda::fail;

extern "C" int paged_decode_attn_copy_blocks(void* k_cache, void* v_cache, int64_t num_blocks,
                                             int64_t block_bytes, const int64_t* pairs,
                                             int n_pairs, int* err, int device, void* stream) {
  if (num_blocks < 0 || block_bytes < 0 || n_pairs < 0 || device < 0)
    return fail(PDA_EINVAL, "negative size or device");
  if (block_bytes % 16) return fail(PDA_EINVAL, "block_bytes must be a multiple of 16");
  if (n_pairs > 65535) return fail(PDA_EINVAL, "at most 65535 pairs per call");
  if (n_pairs == 0 || block_bytes == 0) return PDA_OK;
  if (!k_cache || !v_cache || !pairs) return fail(PDA_EINVAL, "a required pointer is NULL");
  if (!pda::aligned(k_cache, 16) || !pda::aligned(v_cache, 16) || !pda::aligned(pairs, 8))
    return fail(PDA_EINVAL, "caches must be 16-byte aligned, pairs 8-byte aligned");
  if (k_cache == v_cache) return fail(PDA_EALIAS, "k_cache and v_cache are the same buffer");
  pda::Dev guard(device);
  if (guard.err != cudaSuccess) return fail(PDA_ECUDA, "cudaSetDevice failed");
  const int64_t tiles = (block_bytes + pda::kTileBytes - 1) / pda::kTileBytes;
  if (tiles > INT_MAX) return fail(PDA_EINVAL, "block too large");
  pda::copy_blocks_kernel<<<dim3((unsigned)tiles, (unsigned)n_pairs), pda::kMoveThreads, 0,
                            static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache), num_blocks, block_bytes,
      pairs, err);
  return pda::launched("copy_blocks launch");
}

extern "C" int paged_decode_attn_gather_kv(const void* k_cache, const void* v_cache,
                                           int64_t num_blocks, int block_size, int64_t row_bytes,
                                           const int32_t* block_table, int max_blocks,
                                           const int32_t* lens, const int64_t* cu_rows,
                                           int batch, int max_len, void* k_out, void* v_out,
                                           int* err, int device, void* stream) {
  if (num_blocks < 0 || block_size < 1 || row_bytes < 0 || max_blocks < 0 || batch < 0 ||
      max_len < 0 || device < 0)
    return fail(PDA_EINVAL, "negative size, or block_size < 1");
  if (row_bytes % 16) return fail(PDA_EINVAL, "row_bytes must be a multiple of 16");
  if (batch > 65535) return fail(PDA_EINVAL, "batch > 65535");
  if (batch == 0 || max_len == 0 || row_bytes == 0) return PDA_OK;
  if (!k_cache || !v_cache || !block_table || !lens || !cu_rows || !k_out || !v_out)
    return fail(PDA_EINVAL, "a required pointer is NULL");
  if (!pda::aligned(k_cache, 16) || !pda::aligned(v_cache, 16) || !pda::aligned(k_out, 16) ||
      !pda::aligned(v_out, 16) || !pda::aligned(cu_rows, 8) || !pda::aligned(lens, 4) ||
      !pda::aligned(block_table, 4))
    return fail(PDA_EINVAL, "misaligned pointer");
  if ((int64_t)max_len > (int64_t)max_blocks * block_size)
    return fail(PDA_EINVAL, "max_len exceeds max_blocks * block_size");
  pda::Dev guard(device);
  if (guard.err != cudaSuccess) return fail(PDA_ECUDA, "cudaSetDevice failed");
  // about 16 KiB of K (and as much of V) per CTA
  const int rows_per_cta = (int)std::max<int64_t>(1, pda::kTileBytes / row_bytes);
  if ((int64_t)max_len / rows_per_cta + 1 > INT_MAX) return fail(PDA_EINVAL, "max_len too large");
  const int64_t tiles = ((int64_t)max_len + rows_per_cta - 1) / rows_per_cta;
  pda::gather_kernel<<<dim3((unsigned)tiles, (unsigned)batch), pda::kMoveThreads, 0,
                       static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(k_cache), static_cast<const uint8_t*>(v_cache), num_blocks,
      block_size, row_bytes, block_table, max_blocks, lens, cu_rows, max_len, rows_per_cta,
      static_cast<uint8_t*>(k_out), static_cast<uint8_t*>(v_out), err);
  return pda::launched("gather launch");
}

extern "C" int paged_decode_attn_scatter_kv(const void* k_rows, const void* v_rows,
                                            int64_t n_rows, int64_t row_bytes,
                                            const int64_t* slot_mapping, void* k_cache,
                                            void* v_cache, int64_t num_slots, int* err,
                                            int device, void* stream) {
  if (n_rows < 0 || row_bytes < 0 || num_slots < 0 || device < 0)
    return fail(PDA_EINVAL, "negative size or device");
  if (row_bytes % 16) return fail(PDA_EINVAL, "row_bytes must be a multiple of 16");
  if (n_rows == 0 || row_bytes == 0) return PDA_OK;
  if (!k_rows || !v_rows || !slot_mapping || !k_cache || !v_cache)
    return fail(PDA_EINVAL, "a required pointer is NULL");
  if (!pda::aligned(k_rows, 16) || !pda::aligned(v_rows, 16) || !pda::aligned(k_cache, 16) ||
      !pda::aligned(v_cache, 16) || !pda::aligned(slot_mapping, 8))
    return fail(PDA_EINVAL, "misaligned pointer");
  const int rows_per_cta = (int)std::max<int64_t>(1, pda::kTileBytes / row_bytes);
  const int64_t blocks = (n_rows + rows_per_cta - 1) / rows_per_cta;
  if (blocks > INT_MAX) return fail(PDA_EINVAL, "too many rows for one launch");
  pda::Dev guard(device);
  if (guard.err != cudaSuccess) return fail(PDA_ECUDA, "cudaSetDevice failed");
  pda::scatter_kernel<<<(unsigned)blocks, pda::kMoveThreads, 0,
                        static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(k_rows), static_cast<const uint8_t*>(v_rows), n_rows,
      row_bytes, slot_mapping, rows_per_cta, static_cast<uint8_t*>(k_cache),
      static_cast<uint8_t*>(v_cache), num_slots, err);
  return pda::launched("scatter launch");
}

extern "C" int paged_decode_attn_remap_table(int32_t* block_table, int batch, int max_blocks,
                                             const int32_t* lens, int block_size,
                                             const int32_t* new_id, int64_t num_blocks,
                                             int* err, int device, void* stream) {
  if (batch < 0 || max_blocks < 0 || block_size < 1 || num_blocks < 0 || device < 0)
    return fail(PDA_EINVAL, "negative size, or block_size < 1");
  const int64_t n = (int64_t)batch * max_blocks;
  if (n == 0) return PDA_OK;
  if (!block_table || !lens || !new_id) return fail(PDA_EINVAL, "a required pointer is NULL");
  if (!pda::aligned(block_table, 4) || !pda::aligned(lens, 4) || !pda::aligned(new_id, 4))
    return fail(PDA_EINVAL, "misaligned pointer");
  const int64_t blocks = (n + pda::kMoveThreads - 1) / pda::kMoveThreads;
  if (blocks > INT_MAX) return fail(PDA_EINVAL, "table too large");
  pda::Dev guard(device);
  if (guard.err != cudaSuccess) return fail(PDA_ECUDA, "cudaSetDevice failed");
  pda::remap_kernel<<<(unsigned)blocks, pda::kMoveThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      block_table, batch, max_blocks, lens, block_size, new_id, num_blocks, err);
  return pda::launched("remap launch");
}
