// Log-sum-exp merge of split-K partials, and the opt-in input validator.
//
// Merge (Loom Kernels landing page, "Supported now": the split-K/LSE part of
// "Paged MQA/GQA decode"): for a row r with per-split normalised outputs o_s
// and natural-log sums lse_s,
//   M = max_s lse_s,  w_s = exp(lse_s - M),  out = sum_s w_s o_s / sum_s w_s.
// One warp per row; lane i holds lse of splits i and i + 32 (S <= 64) and
// the row's dims are walked four at a time with float4 loads.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "pda_internal.h"

namespace pda {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMergeWarps = 4;

template <typename TOut>
__device__ __forceinline__ void store4(TOut* dst, float4 v) {
  if constexpr (std::is_same_v<TOut, float>) {
    *reinterpret_cast<float4*>(dst) = v;
  } else if constexpr (std::is_same_v<TOut, __half>) {
    __half2 a = __floats2half2_rn(v.x, v.y);
    __half2 b = __floats2half2_rn(v.z, v.w);
    uint2 u;
    memcpy(&u.x, &a, 4);
    memcpy(&u.y, &b, 4);
    *reinterpret_cast<uint2*>(dst) = u;
  } else {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    memcpy(&u.x, &a, 4);
    memcpy(&u.y, &b, 4);
    *reinterpret_cast<uint2*>(dst) = u;
  }
}

template <typename TOut>
__global__ void __launch_bounds__(kMergeWarps * 32) lse_merge_kernel(const MergeParams p) {
  const int row = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.rows) return;
  int S = p.num_splits;
  if (p.context_lens != nullptr) {
    // decode path: the partial kernel wrote `out` itself for 0 or 1 split
    const int b = row / p.Hq;
    int L = __ldg(p.context_lens + b);
    const int maxL = p.max_blocks * p.block_size;
    L = L < 0 ? 0 : (L > maxL ? maxL : L);
    const int n_pages = (L + p.block_size - 1) / p.block_size;
    int sb = (n_pages + p.chunk_pages - 1) / p.chunk_pages;
    if (sb > p.num_splits) sb = p.num_splits;
    if (sb <= 1) return;
    S = sb;
  }
  const float* lse = p.lse + (int64_t)row * p.num_splits;
  const float* o = p.o + (int64_t)row * p.num_splits * p.head_dim;
  TOut* out = static_cast<TOut*>(p.out) + (int64_t)row * p.head_dim;

  const float l0 = lane < S ? lse[lane] : -INFINITY;
  const float l1 = lane + 32 < S ? lse[lane + 32] : -INFINITY;
  float M = fmaxf(l0, l1);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
  if (M == -INFINITY) {  // every split empty
    for (int d4 = lane; d4 < p.head_dim / 4; d4 += 32)
      store4<TOut>(out + d4 * 4, make_float4(0.f, 0.f, 0.f, 0.f));
    return;
  }
  const float w0 = (l0 == -INFINITY) ? 0.f : exp2f((l0 - M) * kLog2e);
  const float w1 = (l1 == -INFINITY) ? 0.f : exp2f((l1 - M) * kLog2e);
  float wsum = w0 + w1;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(kFull, wsum, off);
  const float inv = 1.f / wsum;

  for (int d4 = lane; d4 < p.head_dim / 4; d4 += 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < S; ++s) {
      const float w = __shfl_sync(kFull, s < 32 ? w0 : w1, s & 31);
      if (w != 0.f) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(o + (int64_t)s * p.head_dim) + d4);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
      }
    }
    store4<TOut>(out + d4 * 4, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
  }
}

// One block per sequence: thread 0 checks the context length, all threads
// check the block ids of the pages the sequence reads. The first problem is
// recorded in err[0..1]; nothing traps.
__global__ void validate_kernel(const int32_t* block_table, const int32_t* context_lens,
                                int max_blocks, int block_size, int64_t num_blocks, int* err) {
  const int b = blockIdx.x;
  const int L = context_lens[b];
  const int maxL = max_blocks * block_size;
  if (threadIdx.x == 0 && (L < 0 || L > maxL)) {
    if (atomicCAS(err, 0, kErrContextLen) == 0) err[1] = b;
  }
  const int Lc = L < 0 ? 0 : (L > maxL ? maxL : L);
  const int pages = (Lc + block_size - 1) / block_size;
  for (int pg = threadIdx.x; pg < pages; pg += blockDim.x) {
    const int32_t blk = block_table[(int64_t)b * max_blocks + pg];
    if (blk < 0 || (int64_t)blk >= num_blocks) {
      if (atomicCAS(err, 0, kErrBlockId) == 0) err[1] = b;
      break;
    }
  }
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, int out_dtype, cudaStream_t stream) {
  if (p.rows <= 0) return cudaSuccess;
  const dim3 grid((p.rows + kMergeWarps - 1) / kMergeWarps);
  switch (out_dtype) {
    case 0: lse_merge_kernel<__nv_bfloat16><<<grid, kMergeWarps * 32, 0, stream>>>(p); break;
    case 1: lse_merge_kernel<__half><<<grid, kMergeWarps * 32, 0, stream>>>(p); break;
    case 2: lse_merge_kernel<float><<<grid, kMergeWarps * 32, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_validate(const int32_t* block_table, const int32_t* context_lens, int batch,
                            int max_blocks, int block_size, int64_t num_blocks, int* err,
                            cudaStream_t stream) {
  if (batch <= 0) return cudaSuccess;
  validate_kernel<<<batch, 128, 0, stream>>>(block_table, context_lens, max_blocks, block_size,
                                             num_blocks, err);
  return cudaGetLastError();
}

}  // namespace pda
