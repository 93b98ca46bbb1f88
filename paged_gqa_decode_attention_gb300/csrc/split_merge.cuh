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

// Called by 128 threads (tid 0..127) after each has written its part of this
// split's partial (head dim D). `sw` is shared scratch of at least G * 64 + 1
// floats, `bar_id` a named barrier over exactly these 128 threads.
template <int G, int D, typename TOut>
__device__ __forceinline__ void finish_split(const PartialParams& p, int b, int h, int n_splits_b,
                                             int tid, float* sw, int bar_id) {
  static_assert(D % 4 == 0, "float4 columns");
  constexpr int kCols = D / 4;
  __threadfence();
  named_bar_sync(bar_id, 128);
  int* flag = reinterpret_cast<int*>(sw + G * 64);
  if (tid == 0) {
    const int prev = atomicAdd(p.counters + (int64_t)b * p.Hkv + h, 1);
    *flag = (prev == n_splits_b - 1);
  }
  named_bar_sync(bar_id, 128);
  if (!*flag) return;
  __threadfence();
  const int hq0 = h * G;
  const int64_t row0 = (int64_t)b * p.Hq + hq0;
  for (int i = tid; i < G * n_splits_b; i += 128) {
    const int g = i / n_splits_b, s = i - g * n_splits_b;
    sw[g * 64 + s] = __ldcg(p.ws_lse + (row0 + g) * p.num_splits + s);
  }
  named_bar_sync(bar_id, 128);
  if (tid < G) {
    float* w = sw + tid * 64;
    float M = -INFINITY;
    for (int s = 0; s < n_splits_b; ++s) M = fmaxf(M, w[s]);
    float sum = 0.f;
    for (int s = 0; s < n_splits_b; ++s) {
      const float e = (w[s] == -INFINITY) ? 0.f : exp2f((w[s] - M) * kLog2e);
      w[s] = e;
      sum += e;
    }
    const float inv = 1.f / sum;
    for (int s = 0; s < n_splits_b; ++s) w[s] *= inv;
  }
  named_bar_sync(bar_id, 128);
  // thread -> (head g, 4 consecutive dims): G * D / 4 such pairs over 128
  // threads, float4 loads, 8 splits in flight per step
  TOut* out = static_cast<TOut*>(p.out);
  for (int pair = tid; pair < G * kCols; pair += 128) {
    const int g = pair / kCols, d4 = (pair - g * kCols) * 4;
    const float4* o = reinterpret_cast<const float4*>(p.ws_o + ((row0 + g) * p.num_splits) * D + d4);
    const float* w = sw + g * 64;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int s = 0;
    for (; s + 8 <= n_splits_b; s += 8) {
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = __ldcg(o + (s + k) * kCols);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        acc.x = fmaf(w[s + k], v[k].x, acc.x);
        acc.y = fmaf(w[s + k], v[k].y, acc.y);
        acc.z = fmaf(w[s + k], v[k].z, acc.z);
        acc.w = fmaf(w[s + k], v[k].w, acc.w);
      }
    }
    for (; s < n_splits_b; ++s) {
      const float4 v = __ldcg(o + s * kCols);
      acc.x = fmaf(w[s], v.x, acc.x);
      acc.y = fmaf(w[s], v.y, acc.y);
      acc.z = fmaf(w[s], v.z, acc.z);
      acc.w = fmaf(w[s], v.w, acc.w);
    }
    TOut* dst = out + (row0 + g) * D + d4;
    dst[0] = merge_to_out<TOut>(acc.x);
    dst[1] = merge_to_out<TOut>(acc.y);
    dst[2] = merge_to_out<TOut>(acc.z);
    dst[3] = merge_to_out<TOut>(acc.w);
  }
  if (tid == 0) p.counters[(int64_t)b * p.Hkv + h] = 0;  // ready for the next call
}

}  // namespace pda
