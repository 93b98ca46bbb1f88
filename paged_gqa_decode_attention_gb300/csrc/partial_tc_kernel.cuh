// Split-K partial kernel on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators) for GQA groups of G = 4 or 8 query heads per kv head.
//
// Same method and work decomposition as the CUDA-core kernel
// (partial_kernel.cuh): one CTA per (split, kv head, sequence), split-K with
// a normalised partial and its log-sum-exp per split (Loom Kernels landing
// page, "Supported now": Paged MQA/GQA decode, GQA packing + local
// split-K/LSE). What changes is where the two contractions of a 128-token
// chunk run. With the G query rows packed as the N side of the MMA:
//
//   S^T [128 tokens x 16]  = K_chunk [128 x 128 dims] . Q^T [128 dims x 16]
//   O^T [128 dims   x 16]  = V_chunk^T [128 dims x 128 tokens] . P^T [128 x 16]
//
// (rows G..15 of Q and P are zero). Both are M=128, N=16, K=128 tcgen05.mma
// (kind::f16, fp32 accumulate in TMEM) issued by one thread; the K and V
// tiles are consumed straight from the TMA-written, 128-byte-swizzled stage:
// K as a K-major A operand, V as an MN-major A operand. The probabilities P
// are written to shared memory as two bf16 (or fp16) operands, hi = rn(p) and
// lo = rn(p - hi), both multiplied into O, so P keeps about 16 significant
// bits (one 8-bit operand would cost up to 2^-9 relative error per weight).
//
// Warp roles (192 threads):
//   warps 0-3: softmax and epilogue. Thread t reads TMEM lane t of S (token t
//     of the chunk), scales and masks it, joins a CTA-wide max per head
//     (shuffles + shared memory), writes p_hi/p_lo and, for tokens past the
//     context, zeroes that token's V row (so 0 * stale data never enters the
//     MMA); then reads TMEM lane t of O (dim t) and folds it into a running
//     fp32 accumulator with the online-softmax rescale.
//   warps 4 and 5: producers, TMA page loads of K and of V into two separate
//     3-slot rings (a slot is 128 tokens, 32 KiB): a K slot is released as
//     soon as its QK^T completes, a V slot after its PV, so K loads run ahead.
//   warp 6: allocates 64 TMEM columns (S0, S1, O0, O1, 16 each), issues the
//     MMAs and commits their completion to mbarriers.
// S, O and P are double-buffered by chunk parity so the chunks overlap: the
// MMA warp issues QK^T of chunk c+1 as soon as its K tile lands (while the
// softmax warps work on chunk c), then PV of chunk c once its P is written;
// the softmax warps fold O of chunk c-1 into the running output after
// writing P of chunk c.
// Every wait is bounded; a timed-out CTA records error code 3, stops issuing
// work, still passes every barrier, and frees its TMEM.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "pda_internal.h"
#include "ptx.cuh"
#include "split_merge.cuh"

namespace pda {
namespace tc {

constexpr int kT = 128;                    // tokens per stage = MMA M of QK^T
constexpr int kStages = 3;                 // slots per ring (K and V each)
constexpr int kRowBytes = 128;             // one 64-element half of a 128-dim row
constexpr int kHalf = kT * kRowBytes;      // one half tile: 16 KiB
constexpr int kSlotBytes = 2 * kHalf;      // lo, hi halves of a K or V tile: 32 KiB
constexpr int kN = 16;                     // MMA N: the group's query heads, padded
constexpr int kOpHalf = 2048;              // 16 rows x 128 B of a K-major operand half
constexpr int kOpBytes = 2 * kOpHalf;      // Q, P_hi or P_lo operand
constexpr int kThreads = 224;
constexpr int kWarpProducerK = 4;
constexpr int kWarpProducerV = 5;
constexpr int kWarpMma = 6;
constexpr uint32_t kTmemCols = 64;
constexpr unsigned kFull = 0xffffffffu;

constexpr int kOffK = 0;
constexpr int kOffV = kStages * kSlotBytes;
constexpr int kOffQ = 2 * kStages * kSlotBytes;
constexpr int kOffP = kOffQ + kOpBytes;         // [2 buffers][hi, lo] operands
constexpr int kOffRed = kOffP + 4 * kOpBytes;    // 2 x [4 warps][8] floats (chunk maxima)
constexpr int kOffLred = kOffRed + 2 * 4 * 8 * 4;  // [4 warps][8] floats (final sums)
constexpr int kOffBar = kOffLred + 4 * 8 * 4;
constexpr int kNumBars = 4 * kStages + 10;
constexpr int kOffTmem = kOffBar + kNumBars * 8;
constexpr size_t kSmemBytes = 1024 + kOffTmem + 16;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

template <bool FP16>
struct Half16 {
  using T = std::conditional_t<FP16, __half, __nv_bfloat16>;
  static __device__ __forceinline__ T from(float x) {
    if constexpr (FP16) return __float2half_rn(x); else return __float2bfloat16_rn(x);
  }
  static __device__ __forceinline__ float to(T x) {
    if constexpr (FP16) return __half2float(x); else return __bfloat162float(x);
  }
};

template <typename TOut>
__device__ __forceinline__ TOut to_out(float x) {
  if constexpr (std::is_same_v<TOut, float>) {
    return x;
  } else if constexpr (std::is_same_v<TOut, __half>) {
    return __float2half_rn(x);
  } else {
    return __float2bfloat16_rn(x);
  }
}

// Byte offset of element (row n, column k) of a 16 x 128 K-major operand in
// the 128-byte-swizzled layout: two 64-column halves of 2 KiB, each two
// 8-row atoms of 1 KiB; the 16-byte chunk index is XORed with (row & 7).
__device__ __forceinline__ uint32_t op_offset(int n, int k) {
  const int half = k >> 6, col = k & 63;
  return half * kOpHalf + (n >> 3) * 1024 + (n & 7) * 128 + (((col >> 3) ^ (n & 7)) << 4) +
         (col & 7) * 2;
}

template <int G, int BS, bool FP16, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
    paged_partial_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v, const PartialParams p) {
  static_assert(G == 4 || G == 8, "tensor-core path packs 4 or 8 query heads");
  constexpr int PPS = kT / BS;  // pages per stage
  static_assert(kT % BS == 0 && PPS <= 32, "stage must hold whole pages");
  using TOut = std::conditional_t<OUT_F32, float, std::conditional_t<FP16, __half, __nv_bfloat16>>;
  using H = Half16<FP16>;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const uint32_t bar0 = base_u32 + kOffBar;
  // ring barriers: full/empty per slot, ring r = 0 (K) or 1 (V)
  auto full_bar = [&](int r, int s) { return bar0 + 8u * (r * 2 * kStages + s); };
  auto empty_bar = [&](int r, int s) { return bar0 + 8u * (r * 2 * kStages + kStages + s); };
  // per buffer parity b in {0, 1}
  auto s_full = [&](int b) { return bar0 + 8u * (4 * kStages + 0 + b); };
  auto s_free = [&](int b) { return bar0 + 8u * (4 * kStages + 2 + b); };
  auto p_full = [&](int b) { return bar0 + 8u * (4 * kStages + 4 + b); };
  auto o_full = [&](int b) { return bar0 + 8u * (4 * kStages + 6 + b); };
  auto o_free = [&](int b) { return bar0 + 8u * (4 * kStages + 8 + b); };

  const int split = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int hq0 = h * G;
  TOut* out = static_cast<TOut*>(p.out);

  int L = __ldg(p.context_lens + b);
  const int maxL = p.max_blocks * BS;
  L = L < 0 ? 0 : (L > maxL ? maxL : L);
  const int n_pages = (L + BS - 1) / BS;
  int n_splits_b = (n_pages + p.chunk_pages - 1) / p.chunk_pages;
  if (n_splits_b > p.num_splits) n_splits_b = p.num_splits;

  if (n_splits_b == 0) {  // empty context: zero output rows
    if (split == 0) {
      for (int i = threadIdx.x; i < G * kHeadDim; i += kThreads)
        out[((int64_t)b * p.Hq + hq0) * kHeadDim + i] = to_out<TOut>(0.f);
    }
    return;
  }
  if (split >= n_splits_b) return;

  const int p0 = split * p.chunk_pages;
  const int p1 = (split == n_splits_b - 1) ? n_pages : min(p0 + p.chunk_pages, n_pages);
  const int t0 = p0 * BS;
  const int t1 = min(p1 * BS, L);
  const int n_chunks = (p1 - p0 + PPS - 1) / PPS;

  if (threadIdx.x == 0) {
    for (int r = 0; r < 2; ++r)
      for (int s = 0; s < kStages; ++s) {
        mbar_init(full_bar(r, s), 1);
        mbar_init(empty_bar(r, s), 1);
      }
    for (int b2 = 0; b2 < 2; ++b2) {
      mbar_init(s_full(b2), 1);
      mbar_init(s_free(b2), 4);
      mbar_init(p_full(b2), 4);
      mbar_init(o_full(b2), 1);
      mbar_init(o_free(b2), 4);
    }
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(base_u32 + kOffTmem, kTmemCols);
    tmem_relinquish();
  }
  if (warp < 4) {
    // Q rows of the group as the B operand of QK^T (raw values; the scale is
    // applied to S in fp32), rows G..15 zero; both P operands zeroed.
    const int t = threadIdx.x;
    const uint8_t* qb = static_cast<const uint8_t*>(p.q) + (((int64_t)b * p.Hq + hq0) * kHeadDim) * 2;
    for (int i = t; i < 2 * kN * 8; i += 128) {
      const int half = i >> 7, g = (i >> 3) & 15, c = i & 7;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (g < G) v = __ldg(reinterpret_cast<const uint4*>(qb + (g * kHeadDim + half * 64 + c * 8) * 2));
      *reinterpret_cast<uint4*>(base + kOffQ + half * kOpHalf + (g >> 3) * 1024 + (g & 7) * 128 +
                                ((c ^ (g & 7)) << 4)) = v;
    }
    for (int i = t; i < 4 * kOpBytes / 16; i += 128)
      *reinterpret_cast<uint4*>(base + kOffP + i * 16) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base + kOffTmem);
  auto tS = [&](int b2) { return tmem + (uint32_t)(b2 * kN); };
  auto tO = [&](int b2) { return tmem + (uint32_t)((2 + b2) * kN); };

  bool failed = false;

  if (warp == kWarpProducerK || warp == kWarpProducerV) {
    // ------------------- producers: K ring (warp 4), V ring (warp 5) -------------------
    const int r = warp - kWarpProducerK;
    const CUtensorMap* map = r == 0 ? &tmap_k : &tmap_v;
    if (lane == 0) prefetch_tensormap(map);
    const int32_t* table = p.block_table + (int64_t)b * p.max_blocks;
    int win_base = p0;
    int win_blk = (p0 + lane < p1) ? __ldg(table + p0 + lane) : 0;
    for (int c = 0; c < n_chunks; ++c) {
      const int slot = c % kStages;
      if (c >= kStages) {
        const bool ok = mbar_wait(empty_bar(r, slot), ((c / kStages) - 1) & 1);
        if (!__all_sync(kFull, ok)) {
          failed = true;
          break;
        }
      }
      const int pg0 = p0 + c * PPS;
      const int npg = min(PPS, p1 - pg0);
      if (pg0 + PPS > win_base + 32) {
        win_base = pg0;
        win_blk = (pg0 + lane < p1) ? __ldg(table + pg0 + lane) : 0;
      }
      int blk[PPS];
#pragma unroll
      for (int i = 0; i < PPS; ++i) blk[i] = __shfl_sync(kFull, win_blk, (pg0 + i - win_base) & 31);
      if (lane == 0) {
        const uint32_t fb = full_bar(r, slot);
        mbar_arrive_expect_tx(fb, (uint32_t)npg * BS * 2 * kRowBytes);
        const uint32_t st = base_u32 + (r == 0 ? kOffK : kOffV) + slot * kSlotBytes;
#pragma unroll
        for (int i = 0; i < PPS; ++i) {
          if (i < npg) {
            const int y = blk[i] * BS;
            const uint32_t ro = (uint32_t)(i * BS * kRowBytes);
            tma_load_2d(st + ro, map, h * kHeadDim, y, fb);
            tma_load_2d(st + kHalf + ro, map, h * kHeadDim + 64, y, fb);
          }
        }
      }
      __syncwarp();
    }
  } else if (warp == kWarpMma) {
    // ------------------------------ MMA issue -----------------------------
    constexpr uint32_t idesc_qk = idesc_f16(128, kN, !FP16, false, false);
    constexpr uint32_t idesc_pv = idesc_f16(128, kN, !FP16, true, false);
    const uint32_t q_u32 = base_u32 + kOffQ;
    // S(c) = K(c) . Q^T into S[c & 1]; needs the stage and the softmax's read of S(c-2)
    auto issue_qk = [&](int c) {
      const int slot = c % kStages;
      bool ok = !failed && mbar_wait(full_bar(0, slot), (c / kStages) & 1);
      if (ok && c >= 2) ok = mbar_wait(s_free(c & 1), ((c - 2) >> 1) & 1);
      if (!__all_sync(kFull, ok)) failed = true;
      if (failed) return;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t kb = base_u32 + kOffK + slot * kSlotBytes;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t a = sdesc_sw128(kb + (k >> 2) * kHalf + (k & 3) * 32, 16, 1024);
          const uint64_t bq = sdesc_sw128(q_u32 + (k >> 2) * kOpHalf + (k & 3) * 32, 16, 1024);
          mma_f16_ss(tS(c & 1), a, bq, idesc_qk, k > 0 ? 1u : 0u);
        }
        mma_commit(s_full(c & 1));
        mma_commit(empty_bar(0, slot));  // K slot free once QK^T has read it
      }
      __syncwarp();
    };
    if (n_chunks > 0) issue_qk(0);
    for (int c = 0; c < n_chunks; ++c) {
      if (c + 1 < n_chunks) issue_qk(c + 1);
      // O(c) = V(c)^T . P(c)^T into O[c & 1]; needs P(c) and the fold of O(c-2)
      const int vslot = c % kStages;
      bool ok = !failed && mbar_wait(full_bar(1, vslot), (c / kStages) & 1);
      if (ok) ok = mbar_wait(p_full(c & 1), (c >> 1) & 1);
      if (ok && c >= 2) ok = mbar_wait(o_free(c & 1), ((c - 2) >> 1) & 1);
      if (!__all_sync(kFull, ok)) failed = true;
      if (!failed) {
        tc_fence_after();
        if (lane == 0) {
          const int slot = vslot;
          const uint32_t vb = base_u32 + kOffV + slot * kSlotBytes;
          const uint32_t phi = base_u32 + kOffP + (c & 1) * 2 * kOpBytes;
          const uint32_t plo = phi + kOpBytes;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            // V^T as an MN-major A operand: 64-dim halves kHalf apart (LBO),
            // 8-token row groups 1 KiB apart (SBO); 16 tokens per step
            const uint64_t a = sdesc_sw128(vb + k * 2048, kHalf, 1024);
            const uint32_t po = (k >> 2) * kOpHalf + (k & 3) * 32;
            mma_f16_ss(tO(c & 1), a, sdesc_sw128(phi + po, 16, 1024), idesc_pv, k > 0 ? 1u : 0u);
            mma_f16_ss(tO(c & 1), a, sdesc_sw128(plo + po, 16, 1024), idesc_pv, 1u);
          }
          mma_commit(o_full(c & 1));
          mma_commit(empty_bar(1, slot));
        }
        __syncwarp();
      }
    }
    // Drain the last stages' completion arrivals so that no MMA commit lands
    // on this CTA's shared memory after it exits.
    for (int c = n_chunks > kStages ? n_chunks - kStages : 0; c < n_chunks && !failed; ++c) {
      bool ok = mbar_wait(empty_bar(0, c % kStages), (c / kStages) & 1);
      if (ok) ok = mbar_wait(empty_bar(1, c % kStages), (c / kStages) & 1);
      if (!__all_sync(kFull, ok)) failed = true;
    }
  } else {
    // ------------------------- softmax and epilogue ------------------------
    const int t = threadIdx.x;  // token row of S; output dim of O
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float m_run[G], l_th[G], acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_run[g] = -INFINITY;
      l_th[g] = 0.f;
      acc[g] = 0.f;
    }
    float* red = reinterpret_cast<float*>(base + kOffRed);
    float alpha_prev[G];
    // acc = acc * alpha(c) + O(c), for the chunk before the current one
    auto fold = [&](int c) {
      bool ok = !failed && mbar_wait(o_full(c & 1), (c >> 1) & 1);
      if (!__all_sync(kFull, ok)) failed = true;
      tc_fence_after();
      float o[G];
      if constexpr (G == 4) {
        tmem_ld_x4(tO(c & 1) + lane_base, o);
      } else {
        tmem_ld_x8(tO(c & 1) + lane_base, o);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free(c & 1));
#pragma unroll
      for (int g = 0; g < G; ++g) acc[g] = acc[g] * alpha_prev[g] + o[g];
    };
    for (int c = 0; c < n_chunks; ++c) {
      const int slot = c % kStages;
      const int n_valid = min(kT, t1 - (t0 + c * kT));
      bool ok = !failed && mbar_wait(s_full(c & 1), (c >> 1) & 1);
      if (!__all_sync(kFull, ok)) failed = true;
      tc_fence_after();
      float s[G];
      if constexpr (G == 4) {
        tmem_ld_x4(tS(c & 1) + lane_base, s);
      } else {
        tmem_ld_x8(tS(c & 1) + lane_base, s);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free(c & 1));
#pragma unroll
      for (int g = 0; g < G; ++g) s[g] = (t < n_valid) ? s[g] * p.qscale : -INFINITY;
      float* rb = red + (c & 1) * 32;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float mx = s[g];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
        if (lane == 0) rb[warp * 8 + g] = mx;
      }
      named_bar_sync(1, 128);
      float alpha[G];
      uint8_t* pb = base + kOffP + (c & 1) * 2 * kOpBytes;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float mx = fmaxf(fmaxf(rb[g], rb[8 + g]), fmaxf(rb[16 + g], rb[24 + g]));
        const float mn = fmaxf(m_run[g], mx);  // finite: every chunk holds a valid token
        alpha[g] = exp2f(m_run[g] - mn);
        m_run[g] = mn;
        const float pr = exp2f(s[g] - mn);
        l_th[g] = l_th[g] * alpha[g] + pr;
        const typename H::T hi = H::from(pr);
        const typename H::T lo = H::from(pr - H::to(hi));
        const uint32_t off = op_offset(g, t);
        *reinterpret_cast<typename H::T*>(pb + off) = hi;
        *reinterpret_cast<typename H::T*>(pb + kOpBytes + off) = lo;
      }
      if (n_valid < kT) {
        // keep stale or out-of-context V rows out of the MMA; the V tile of
        // this chunk must have landed first (its last page may be partial)
        ok = !failed && mbar_wait(full_bar(1, slot), (c / kStages) & 1);
        if (!__all_sync(kFull, ok)) failed = true;
      }
      if (t >= n_valid) {
        uint8_t* vrow = base + kOffV + slot * kSlotBytes + t * kRowBytes;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<uint4*>(vrow + hh * kHalf + i * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(c & 1));
      if (c > 0) fold(c - 1);
#pragma unroll
      for (int g = 0; g < G; ++g) alpha_prev[g] = alpha[g];
    }
    if (n_chunks > 0) fold(n_chunks - 1);
    // softmax denominators: sum the per-token partial sums over 128 threads
    float* lred = reinterpret_cast<float*>(base + kOffLred);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float v = l_th[g];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
      if (lane == 0) lred[warp * 8 + g] = v;
    }
    named_bar_sync(1, 128);
    const int d = t;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float Ls = lred[g] + lred[8 + g] + lred[16 + g] + lred[24 + g];
      const float o = acc[g] / Ls;
      const int64_t row = (int64_t)b * p.Hq + hq0 + g;
      if (n_splits_b == 1) {
        out[row * kHeadDim + d] = to_out<TOut>(o);
      } else {
        const int64_t r = row * p.num_splits + split;
        p.ws_o[r * kHeadDim + d] = o;
        if (d == 0) p.ws_lse[r] = (m_run[g] + log2f(Ls)) * kLn2;
      }
    }
    // the last split of this (sequence, kv head) merges all of them into `out`
    // (the P operands are free: every PV has completed)
    if (n_splits_b > 1)
      finish_split<G, TOut>(p, b, h, n_splits_b, d, reinterpret_cast<float*>(base + kOffP), 1);
  }

  if (failed && lane == 0 && atomicCAS(p.err, 0, kErrWaitTimeout) == 0) p.err[1] = split;
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int G, int BS, bool FP16, bool OUT_F32>
cudaError_t launch_one(const CUtensorMap* tk, const CUtensorMap* tv, const PartialParams& p,
                       int batch, cudaStream_t stream) {
  dim3 grid(p.num_splits, p.Hkv, batch);
  paged_partial_tc_kernel<G, BS, FP16, OUT_F32><<<grid, kThreads, kSmemBytes, stream>>>(*tk, *tv,
                                                                                      p);
  return cudaGetLastError();
}

template <int G, int BS, bool FP16, bool OUT_F32>
cudaError_t prepare_one() {
  return cudaFuncSetAttribute(paged_partial_tc_kernel<G, BS, FP16, OUT_F32>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
}

template <int G, int BS, bool FP16>
int occupancy_one() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, paged_partial_tc_kernel<G, BS, FP16, false>, kThreads, kSmemBytes) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

template <bool FP16>
struct Dispatch {
  template <int G, int BS>
  static cudaError_t launch_g(bool f32, const CUtensorMap* tk, const CUtensorMap* tv,
                              const PartialParams& p, int batch, cudaStream_t s) {
    return f32 ? launch_one<G, BS, FP16, true>(tk, tv, p, batch, s)
               : launch_one<G, BS, FP16, false>(tk, tv, p, batch, s);
  }
  static cudaError_t launch(int G, int BS, bool f32, const CUtensorMap* tk, const CUtensorMap* tv,
                            const PartialParams& p, int batch, cudaStream_t s) {
    if (G == 4 && BS == 16) return launch_g<4, 16>(f32, tk, tv, p, batch, s);
    if (G == 4 && BS == 32) return launch_g<4, 32>(f32, tk, tv, p, batch, s);
    if (G == 8 && BS == 16) return launch_g<8, 16>(f32, tk, tv, p, batch, s);
    if (G == 8 && BS == 32) return launch_g<8, 32>(f32, tk, tv, p, batch, s);
    return cudaErrorInvalidValue;
  }
  template <int G, int BS>
  static cudaError_t prepare_g() {
    cudaError_t e = prepare_one<G, BS, FP16, false>();
    return e != cudaSuccess ? e : prepare_one<G, BS, FP16, true>();
  }
  static cudaError_t prepare(int G, int BS) {
    if (G == 4 && BS == 16) return prepare_g<4, 16>();
    if (G == 4 && BS == 32) return prepare_g<4, 32>();
    if (G == 8 && BS == 16) return prepare_g<8, 16>();
    if (G == 8 && BS == 32) return prepare_g<8, 32>();
    return cudaErrorInvalidValue;
  }
  static int occupancy(int G, int BS) {
    if (G == 4) return BS == 16 ? occupancy_one<4, 16, FP16>() : occupancy_one<4, 32, FP16>();
    return BS == 16 ? occupancy_one<8, 16, FP16>() : occupancy_one<8, 32, FP16>();
  }
};

}  // namespace tc
}  // namespace pda
