// Split-K partial kernel for paged MQA/GQA decode attention (sm_103a).
//
// Loom Kernels landing page, "Supported now" ("Paged MQA/GQA decode": GQA
// packing + local split-K/LSE) and benchmark page, "Current qualified
// results" (the D128 long-context split-K/LSE path) name the method; this is
// a GB300 design of it.
//
// One CTA handles one (split s, kv head h, sequence b). It streams the
// split's K/V pages for head h from HBM into shared memory with TMA tiled
// loads (one 64-dim x block_size box per half-row, 128-byte swizzle), through
// a kStages-deep ring of stages guarded by mbarriers:
//   warp kNW (producer): reads block-table entries (32 at a time, shared by
//     shuffles) and issues the TMA loads for the next stage once the
//     consumers have released it;
//   warps 0..kNW-1 (consumers): each owns kTPW tokens of every stage and runs
//     its own online softmax over them for all G query heads of the group:
//       QK: LPT lanes per token, each holding a slice of the G pre-scaled
//           query rows in registers, dot products reduced by xor-shuffles;
//       softmax: chunk max by shuffles, rescale of the running state;
//       PV: each lane owns D / 32 of the output dims for all G heads.
// Head dims D of 64, 128 and 256 (one, two or four 64-dim boxes per row) and
// any group size G up to 8 (up to 4 at D = 256, where the query slice would
// not fit the registers) are instantiated.
// At the end the consumer warps' (max, sum, acc) states are merged through
// shared memory; a sequence handled by a single split writes `out` directly,
// otherwise the split writes its normalised partial and natural-log LSE to
// the workspace and the last split to finish merges them (split_merge.cuh).
//
// Logits are kept in base-2 units (q is pre-multiplied by scale * log2 e) so
// the exponentials are exp2f; the LSE is converted back to natural log.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "pda_internal.h"
#include "ptx.cuh"
#include "split_merge.cuh"

namespace pda {
namespace partial {

constexpr int kNW = 4;                    // consumer warps
constexpr int kTPW = 16;                  // tokens per consumer warp per stage
constexpr int kChunk = kNW * kTPW;        // tokens per stage
constexpr int kStages = 3;                // pipeline depth
constexpr int kRowBytes = 128;            // one 64-element box of a row
constexpr int kHalfBytes = kChunk * kRowBytes;  // one box column of a stage
constexpr int kThreads = (kNW + 1) * 32;
constexpr int kPBufBytes = kNW * kTPW * 8 * 4;  // probabilities, room for G <= 8
constexpr int kBarBytes = 2 * kStages * 8;
constexpr unsigned kFull = 0xffffffffu;

// Bytes of one stage: K and V, D / 64 boxes each.
__host__ __device__ constexpr int stage_bytes(int D) { return 2 * (D / 64) * kHalfBytes; }
__host__ __device__ constexpr size_t smem_bytes(int D) {
  return 1024 + size_t(kStages) * stage_bytes(D) + kPBufBytes + kBarBytes;
}
// Lanes per token in QK: enough that each lane's slice of the G query rows
// (G * D / LPT floats) stays within 128 registers; 8 from G = 4 on, where
// 4 lanes spilled at D = 128.
__host__ __device__ constexpr int lpt_for(int G, int D) {
  return (G >= 4 || G * D / 4 > 128) ? 8 : 4;
}
__host__ __device__ constexpr bool geometry_supported(int G, int D) {
  return G >= 1 && G <= 8 && (D == 64 || D == 128 || D == 256) && G * D / lpt_for(G, D) <= 128;
}

template <bool FP16>
__device__ __forceinline__ void unpack2(uint32_t w, float& lo, float& hi) {
  if constexpr (FP16) {
    __half2 h2;
    memcpy(&h2, &w, 4);
    const float2 f = __half22float2(h2);
    lo = f.x;
    hi = f.y;
  } else {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  }
}

template <bool FP16>
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  unpack2<FP16>(u.x, f[0], f[1]);
  unpack2<FP16>(u.y, f[2], f[3]);
  unpack2<FP16>(u.z, f[4], f[5]);
  unpack2<FP16>(u.w, f[6], f[7]);
}

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

__device__ __forceinline__ void record_error(int* err, int code, int detail) {
  if (atomicCAS(err, 0, code) == 0) err[1] = detail;
}

template <int G, int D, int BS, bool FP16>
__global__ void __launch_bounds__(kThreads, partial_ctas_per_sm_hint(kPartialCudaCore, G, D))
    paged_partial_kernel(const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const PartialParams p) {
  static_assert(geometry_supported(G, D), "unsupported (G, D)");
  constexpr int NB = D / 64;             // 64-dim boxes per row
  constexpr int LPT = lpt_for(G, D);     // lanes per token in QK
  constexpr int TPP = 32 / LPT;          // tokens per QK pass
  constexpr int PASSES = kTPW / TPP;
  constexpr int CPS = 8 / LPT;           // 16-byte chunks per lane per box
  constexpr int DPL = D / 32;            // PV: output dims per lane
  constexpr int PPS = kChunk / BS;       // pages per stage
  constexpr int kStageBytes = stage_bytes(D);
  constexpr int kVOff = NB * kHalfBytes;  // V boxes follow the K boxes in a stage
  static_assert(kChunk % BS == 0 && PPS <= 32, "stage must hold whole pages");
  using TNat = std::conditional_t<FP16, __half, __nv_bfloat16>;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;  // 128B-swizzle atoms need 1 KiB
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  float* pbuf = reinterpret_cast<float*>(base + kStages * kStageBytes);
  const uint32_t bar0 = base_u32 + kStages * kStageBytes + kPBufBytes;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };

  const int split = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int hq0 = h * G;

  // The producer's first block-table window depends only on the split index,
  // so its load is issued before the context length arrives.
  const int p0_spec = split * p.chunk_pages;
  int spec_blk = 0;
  if ((threadIdx.x >> 5) == kNW && p0_spec + (threadIdx.x & 31) < p.max_blocks)
    spec_blk = __ldg(p.block_table + (int64_t)b * p.max_blocks + p0_spec + (threadIdx.x & 31));
  // Context length, clamped to what the block table can address.
  int L = __ldg(p.context_lens + b);
  const int maxL = p.max_blocks * BS;
  L = L < 0 ? 0 : (L > maxL ? maxL : L);
  const int n_pages = (L + BS - 1) / BS;
  int n_splits_b = (n_pages + p.chunk_pages - 1) / p.chunk_pages;
  if (n_splits_b > p.num_splits) n_splits_b = p.num_splits;  // last split takes the rest

  if (n_splits_b == 0) {  // empty context: zero output rows
    if (split == 0) {
      for (int i = threadIdx.x; i < G * D; i += kThreads) {
        const int64_t o = ((int64_t)b * p.Hq + hq0) * D + i;
        if (p.out_f32) static_cast<float*>(p.out)[o] = 0.f;
        else static_cast<TNat*>(p.out)[o] = to_out<TNat>(0.f);
      }
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
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kNW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  bool failed = false;
  float m_run[G], l_run[G], acc[G][DPL];
  // PV: this lane's dims [lane * DPL, lane * DPL + DPL): box, 16-byte chunk
  // within the box, byte offset within the chunk
  const int vbox = (lane * DPL) >> 6;
  const int vch = ((lane * DPL) & 63) >> 3;
  const int vsub = ((lane * DPL) & 7) * 2;

  if (warp == kNW) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    const int32_t* table = p.block_table + (int64_t)b * p.max_blocks;
    // block-table entries in windows of 32 pages, the next window prefetched
    int win_base = p0;
    int win_blk = (p0 + lane < p1) ? spec_blk : 0;
    int nxt_blk = (p0 + 32 + lane < p1) ? __ldg(table + p0 + 32 + lane) : 0;
    for (int c = 0; c < n_chunks; ++c) {
      const int slot = c % kStages;
      if (c >= kStages) {
        const bool ok = mbar_wait(empty_bar(slot), ((c / kStages) - 1) & 1);
        if (!__all_sync(kFull, ok)) {
          failed = true;
          break;
        }
      }
      const int pg0 = p0 + c * PPS;
      const int npg = min(PPS, p1 - pg0);
      if (pg0 + PPS > win_base + 32) {  // pg0 == win_base + 32: PPS divides 32
        win_base += 32;
        win_blk = nxt_blk;
        nxt_blk = (win_base + 32 + lane < p1) ? __ldg(table + win_base + 32 + lane) : 0;
      }
      int blk[PPS];
#pragma unroll
      for (int i = 0; i < PPS; ++i) blk[i] = __shfl_sync(kFull, win_blk, (pg0 + i - win_base) & 31);
      if (lane == 0) {
        const uint32_t fb = full_bar(slot);
        mbar_arrive_expect_tx(fb, (uint32_t)npg * BS * 2 * NB * kRowBytes);
        const uint32_t st = base_u32 + slot * kStageBytes;
#pragma unroll
        for (int i = 0; i < PPS; ++i) {
          if (i < npg) {
            const int y = blk[i] * BS;
            const uint32_t ro = (uint32_t)(i * BS * kRowBytes);
#pragma unroll
            for (int bx = 0; bx < NB; ++bx) {
              tma_load_2d(st + bx * kHalfBytes + ro, &tmap_k, h * D + bx * 64, y, fb);
              tma_load_2d(st + kVOff + bx * kHalfBytes + ro, &tmap_v, h * D + bx * 64, y, fb);
            }
          }
        }
      }
      __syncwarp();
    }
  } else {
    // ------------------------------ consumers -----------------------------
    const int j = lane / LPT;  // token within a QK pass
    const int s = lane % LPT;  // segment: chunks [s*CPS, (s+1)*CPS) of each half-row

    float qf[G][NB][CPS][8];
    {
      // logit scale: softmax scale (base 2) x the kv head's K dequantisation scale
      const float qsc = p.qscale * (p.k_scale ? __ldg(p.k_scale + (p.scale_per_head ? h : 0)) : 1.f);
      const uint8_t* qb = static_cast<const uint8_t*>(p.q) + (((int64_t)b * p.Hq + hq0) * D) * 2;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int hh = 0; hh < NB; ++hh)
#pragma unroll
          for (int i = 0; i < CPS; ++i) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(
                qb + (g * D + hh * 64 + (s * CPS + i) * 8) * 2));
            float t[8];
            unpack8<FP16>(u, t);
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[g][hh][i][e] = t[e] * qsc;
          }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_run[g] = -INFINITY;
      l_run[g] = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[g][e] = 0.f;
    }
    float* pw = pbuf + warp * kTPW * G;

    for (int c = 0; c < n_chunks; ++c) {
      const int slot = c % kStages;
      const bool ok = mbar_wait(full_bar(slot), (c / kStages) & 1);
      if (!__all_sync(kFull, ok)) {
        failed = true;
        break;
      }
      const int n_valid = min(kChunk, t1 - (t0 + c * kChunk));
      const int n_w = min(kTPW, max(0, n_valid - warp * kTPW));
      if (n_w > 0) {
        const uint8_t* kst = base + slot * kStageBytes;
        const uint8_t* vst = kst + kVOff;
        float sc[PASSES][G];
#pragma unroll
        for (int pass = 0; pass < PASSES; ++pass) {
          const int tl = pass * TPP + j;
          const int row = warp * kTPW + tl;
          float a[G];
#pragma unroll
          for (int g = 0; g < G; ++g) a[g] = 0.f;
#pragma unroll
          for (int hh = 0; hh < NB; ++hh)
#pragma unroll
            for (int i = 0; i < CPS; ++i) {
              const int phys = (s * CPS + i) ^ (row & 7);
              const uint4 u = *reinterpret_cast<const uint4*>(kst + hh * kHalfBytes +
                                                              row * kRowBytes + phys * 16);
              float kf[8];
              unpack8<FP16>(u, kf);
#pragma unroll
              for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < 8; ++e) a[g] = fmaf(qf[g][hh][i][e], kf[e], a[g]);
            }
#pragma unroll
          for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int off = 1; off < LPT; off <<= 1) a[g] += __shfl_xor_sync(kFull, a[g], off);
            sc[pass][g] = (tl < n_w) ? a[g] : -INFINITY;
          }
        }
        // online softmax over this warp's tokens of the stage
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float mx = sc[0][g];
#pragma unroll
          for (int pass = 1; pass < PASSES; ++pass) mx = fmaxf(mx, sc[pass][g]);
#pragma unroll
          for (int off = LPT; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
          const float mn = fmaxf(m_run[g], mx);  // finite: n_w > 0
          const float alpha = exp2f(m_run[g] - mn);
          m_run[g] = mn;
          float ls = 0.f;
#pragma unroll
          for (int pass = 0; pass < PASSES; ++pass) {
            sc[pass][g] = exp2f(sc[pass][g] - mn);
            ls += sc[pass][g];
          }
          l_run[g] = l_run[g] * alpha + ls;
#pragma unroll
          for (int e = 0; e < DPL; ++e) acc[g][e] *= alpha;
        }
        if (s == 0) {
#pragma unroll
          for (int pass = 0; pass < PASSES; ++pass)
#pragma unroll
            for (int g = 0; g < G; ++g) pw[(pass * TPP + j) * G + g] = sc[pass][g];
        }
        __syncwarp();
#pragma unroll 4
        for (int t = 0; t < n_w; ++t) {
          const int row = warp * kTPW + t;
          const uint8_t* vp = vst + vbox * kHalfBytes + row * kRowBytes +
                              ((vch ^ (row & 7)) * 16) + vsub;
          float vf[DPL];
          if constexpr (DPL == 2) {
            unpack2<FP16>(*reinterpret_cast<const uint32_t*>(vp), vf[0], vf[1]);
          } else if constexpr (DPL == 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(vp);
            unpack2<FP16>(u.x, vf[0], vf[1]);
            unpack2<FP16>(u.y, vf[2], vf[3]);
          } else {
            unpack8<FP16>(*reinterpret_cast<const uint4*>(vp), vf);
          }
          float pp[G];
          if constexpr (G % 4 == 0) {
#pragma unroll
            for (int g4 = 0; g4 < G / 4; ++g4) {
              const float4 v4 = *reinterpret_cast<const float4*>(pw + t * G + 4 * g4);
              pp[4 * g4 + 0] = v4.x;
              pp[4 * g4 + 1] = v4.y;
              pp[4 * g4 + 2] = v4.z;
              pp[4 * g4 + 3] = v4.w;
            }
          } else {
#pragma unroll
            for (int g = 0; g < G; ++g) pp[g] = pw[t * G + g];
          }
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[g][e] = fmaf(pp[g], vf[e], acc[g][e]);
        }
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(empty_bar(slot));
    }
    // the warp's softmax sum: each token's p is held by its LPT lanes; add
    // over the token lanes only
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int off = LPT; off < 32; off <<= 1) l_run[g] += __shfl_xor_sync(kFull, l_run[g], off);
  }

  if (failed && lane == 0) record_error(p.err, kErrWaitTimeout, split);
  if (warp == kNW) return;

  // ---------------- merge the consumer warps' states ----------------------
  // Scratch aliases the stage ring: every stage has been consumed (all full
  // barriers observed) before the first named barrier.
  named_bar_sync(1, kNW * 32);
  float* mw = reinterpret_cast<float*>(base);  // [kNW][G]
  float* lw = mw + kNW * G;                    // [kNW][G]
  float* aw = lw + kNW * G;                    // [kNW][G][D]
  static_assert(sizeof(float) * kNW * G * (D + 2) <= 2 * (size_t)stage_bytes(D),
                "warp states must fit below the merge scratch");
  if (lane == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      mw[warp * G + g] = m_run[g];
      lw[warp * G + g] = l_run[g];
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < DPL; ++e) aw[(warp * G + g) * D + lane * DPL + e] = acc[g][e];
  named_bar_sync(1, kNW * 32);
  const int tid = threadIdx.x;  // 0 .. 127
  const float vsc = p.v_scale ? __ldg(p.v_scale + (p.scale_per_head ? h : 0)) : 1.f;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kNW; ++w) M = fmaxf(M, mw[w * G + g]);
    float Ls = 0.f;
    float fw[kNW];
#pragma unroll
    for (int w = 0; w < kNW; ++w) {
      const float mwv = mw[w * G + g];
      fw[w] = (mwv == -INFINITY) ? 0.f : exp2f(mwv - M);
      Ls += fw[w] * lw[w * G + g];
    }
    const int64_t row = (int64_t)b * p.Hq + hq0 + g;
    for (int d = tid; d < D; d += kNW * 32) {
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < kNW; ++w) o += fw[w] * aw[(w * G + g) * D + d];
      o = o / Ls * vsc;
      if (n_splits_b == 1) {
        if (p.out_f32) static_cast<float*>(p.out)[row * D + d] = o;
        else static_cast<TNat*>(p.out)[row * D + d] = to_out<TNat>(o);
      } else {
        const int64_t r = row * p.num_splits + split;
        p.ws_o[r * D + d] = o;
        if (d == 0) p.ws_lse[r] = (M + log2f(Ls)) * kLn2;
      }
    }
  }
  // the last split of this (sequence, kv head) merges all of them into `out`
  if (n_splits_b > 1) {
    float* sw = reinterpret_cast<float*>(base + 2 * kStageBytes);
    if (p.out_f32) finish_split<G, D, float>(p, b, h, n_splits_b, tid, sw, 1);
    else finish_split<G, D, TNat>(p, b, h, n_splits_b, tid, sw, 1);
  }
}

template <int G, int D, int BS, bool FP16>
cudaError_t launch_one(const CUtensorMap* tk, const CUtensorMap* tv, const PartialParams& p,
                       int batch, cudaStream_t stream) {
  dim3 grid(p.num_splits, p.Hkv, batch);
  paged_partial_kernel<G, D, BS, FP16><<<grid, kThreads, smem_bytes(D), stream>>>(*tk, *tv, p);
  return cudaGetLastError();
}

template <int G, int D, int BS, bool FP16>
cudaError_t prepare_one() {
  return cudaFuncSetAttribute(paged_partial_kernel<G, D, BS, FP16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes(D));
}

template <int G, int D, int BS, bool FP16>
int occupancy_one() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, paged_partial_kernel<G, D, BS, FP16>,
                                                    kThreads, smem_bytes(D)) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

// Dispatch over (G, block size) for one head dim and input dtype; each
// (D, dtype) pair is instantiated in its own translation unit.
template <int D, bool FP16>
struct Dispatch {
  template <int G>
  static cudaError_t launch_g(int BS, const CUtensorMap* tk, const CUtensorMap* tv,
                              const PartialParams& p, int batch, cudaStream_t s) {
    if constexpr (geometry_supported(G, D)) {
      if (BS == 16) return launch_one<G, D, 16, FP16>(tk, tv, p, batch, s);
      if (BS == 32) return launch_one<G, D, 32, FP16>(tk, tv, p, batch, s);
      if (BS == 64) return launch_one<G, D, 64, FP16>(tk, tv, p, batch, s);
    }
    return cudaErrorInvalidValue;
  }
  template <int G>
  static cudaError_t prepare_g(int BS) {
    if constexpr (geometry_supported(G, D)) {
      if (BS == 16) return prepare_one<G, D, 16, FP16>();
      if (BS == 32) return prepare_one<G, D, 32, FP16>();
      if (BS == 64) return prepare_one<G, D, 64, FP16>();
    }
    return cudaErrorInvalidValue;
  }
  template <int G>
  static int occupancy_g(int BS) {
    if constexpr (geometry_supported(G, D)) {
      return BS == 16   ? occupancy_one<G, D, 16, FP16>()
             : BS == 32 ? occupancy_one<G, D, 32, FP16>()
                        : occupancy_one<G, D, 64, FP16>();
    }
    return 1;
  }
  static cudaError_t launch(int G, int BS, const CUtensorMap* tk, const CUtensorMap* tv,
                            const PartialParams& p, int batch, cudaStream_t s) {
    switch (G) {
      case 1: return launch_g<1>(BS, tk, tv, p, batch, s);
      case 2: return launch_g<2>(BS, tk, tv, p, batch, s);
      case 3: return launch_g<3>(BS, tk, tv, p, batch, s);
      case 4: return launch_g<4>(BS, tk, tv, p, batch, s);
      case 5: return launch_g<5>(BS, tk, tv, p, batch, s);
      case 6: return launch_g<6>(BS, tk, tv, p, batch, s);
      case 7: return launch_g<7>(BS, tk, tv, p, batch, s);
      case 8: return launch_g<8>(BS, tk, tv, p, batch, s);
      default: return cudaErrorInvalidValue;
    }
  }
  static cudaError_t prepare(int G, int BS) {
    switch (G) {
      case 1: return prepare_g<1>(BS);
      case 2: return prepare_g<2>(BS);
      case 3: return prepare_g<3>(BS);
      case 4: return prepare_g<4>(BS);
      case 5: return prepare_g<5>(BS);
      case 6: return prepare_g<6>(BS);
      case 7: return prepare_g<7>(BS);
      case 8: return prepare_g<8>(BS);
      default: return cudaErrorInvalidValue;
    }
  }
  static int occupancy(int G, int BS) {
    switch (G) {
      case 1: return occupancy_g<1>(BS);
      case 2: return occupancy_g<2>(BS);
      case 3: return occupancy_g<3>(BS);
      case 4: return occupancy_g<4>(BS);
      case 5: return occupancy_g<5>(BS);
      case 6: return occupancy_g<6>(BS);
      case 7: return occupancy_g<7>(BS);
      case 8: return occupancy_g<8>(BS);
      default: return 1;
    }
  }
};

}  // namespace partial
}  // namespace pda
