// Fused log-sum-exp merge, run by the last CTA of a (sequence, kv head) to
// finish its splits (Loom Kernels landing page, "Supported now": the LSE part
// of "Paged MQA/GQA decode - GQA packing + local split-K/LSE").
//
// Every split CTA writes its normalised partial o_s and natural-log lse_s,
// makes them visible device-wide (__threadfence) and takes a ticket from an
// atomic counter. The CTA that draws the last ticket merges:
//   M = max_s lse_s,  w_s = exp(lse_s - M) / sum_s' exp(lse_s' - M),
//   out = sum_s w_s o_s,
// then resets the counter to zero for the next call. No CTA waits for
// another: there is no spin, only the ticket.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "pda_internal.h"
#include "ptx.cuh"

namespace pda {

template <typename TOut>
__device__ __forceinline__ TOut merge_to_out(float x) {
  if constexpr (std::is_same_v<TOut, float>) {
    return x;
  } else if constexpr (std::is_same_v<TOut, __half>) {
    return __float2half_rn(x);
  } else {
    return __float2bfloat16_rn(x);
  }
}

// Called by kThreads threads (tid 0..kThreads-1) after each has written its
// part of this split's partial (head dim D). `sw` is shared scratch of at
// least one word, `bar_id` a named barrier over exactly these threads.
//
// The merging CTA is on the step's critical path (it finishes last), so the
// merge is one pass of loads with no further barrier: each thread owns
// (head g, 4 consecutive dims) pairs and reads, per group of kChunk splits,
// the splits' log-sum-exps and its four columns of their partials together
// (all in flight at once), folding them with a running maximum:
//   M = max_s lse_s,  out = sum_s e^(lse_s - M) o_s / sum_s e^(lse_s - M).
template <int G, int D, typename TOut, int kChunk = 8, int kThreads = 128>
__device__ __forceinline__ void finish_split(const PartialParams& p, int b, int h, int n_splits_b,
                                             int tid, float* sw, int bar_id) {
  static_assert(D % 4 == 0, "float4 columns");
  constexpr int kCols = D / 4;
  __threadfence();
  named_bar_sync(bar_id, kThreads);
  int* flag = reinterpret_cast<int*>(sw);
  if (tid == 0) {
    const int prev = atomicAdd(p.counters + (int64_t)b * p.Hkv + h, 1);
    *flag = (prev == n_splits_b - 1);
  }
  named_bar_sync(bar_id, kThreads);
  if (!*flag) return;
  __threadfence();
  const int hq0 = h * G;
  const int64_t row0 = (int64_t)b * p.Hq + hq0;
  TOut* out = static_cast<TOut*>(p.out);
  for (int pair = tid; pair < G * kCols; pair += kThreads) {
    const int g = pair / kCols, d4 = (pair - g * kCols) * 4;
    const float* lrow = p.ws_lse + (row0 + g) * p.num_splits;
    const float4* o = reinterpret_cast<const float4*>(p.ws_o + ((row0 + g) * p.num_splits) * D + d4);
    float M = -INFINITY, wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < n_splits_b; s0 += kChunk) {
      const int n = min(kChunk, n_splits_b - s0);
      float l[kChunk];
      float4 v[kChunk];
#pragma unroll
      for (int k = 0; k < kChunk; ++k) {
        if (k < n) {
          l[k] = __ldcg(lrow + s0 + k);
          v[k] = __ldcg(o + (s0 + k) * kCols);
        }
      }
      float mc = -INFINITY;
#pragma unroll
      for (int k = 0; k < kChunk; ++k)
        if (k < n) mc = fmaxf(mc, l[k]);
      const float Mn = fmaxf(M, mc);
      if (Mn == -INFINITY) continue;  // every split so far is empty
      const float r = (M == -INFINITY) ? 0.f : exp2f((M - Mn) * kLog2e);
      wsum *= r;
      acc.x *= r;
      acc.y *= r;
      acc.z *= r;
      acc.w *= r;
      M = Mn;
#pragma unroll
      for (int k = 0; k < kChunk; ++k) {
        if (k < n) {
          const float w = (l[k] == -INFINITY) ? 0.f : exp2f((l[k] - M) * kLog2e);
          wsum += w;
          acc.x = fmaf(w, v[k].x, acc.x);
          acc.y = fmaf(w, v[k].y, acc.y);
          acc.z = fmaf(w, v[k].z, acc.z);
          acc.w = fmaf(w, v[k].w, acc.w);
        }
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    TOut* dst = out + (row0 + g) * D + d4;
    dst[0] = merge_to_out<TOut>(acc.x * inv);
    dst[1] = merge_to_out<TOut>(acc.y * inv);
    dst[2] = merge_to_out<TOut>(acc.z * inv);
    dst[3] = merge_to_out<TOut>(acc.w * inv);
  }
  if (tid == 0) p.counters[(int64_t)b * p.Hkv + h] = 0;  // ready for the next call
}

}  // namespace pda
