// Split-K partial kernel on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators) for GQA groups of G = 3..16 query heads per kv head (1..16
// with FP8 K/V) and head dims D of 128 or 64.
//
// Same method and work units as the CUDA-core kernel (partial_kernel.cuh):
// a unit is one (split, kv head, sequence), split-K with a normalised partial
// and its log-sum-exp per split (Loom Kernels landing page, "Supported now":
// Paged MQA/GQA decode, GQA packing + local split-K/LSE). Here the kernel is
// persistent: one CTA per SM takes units from a global work counter as it
// goes (so faster SMs take more of them and ragged batches balance), and
// every role streams across unit boundaries, so the TMA rings stay full from
// the first unit to the last. The two contractions of a 128-token chunk
// run on the tensor cores, with the G query rows packed as the N side:
//
//   S^T [128 tokens x 16]  = K_chunk [128 x 128 dims] . Q^T [128 dims x 16]
//   O^T [128 dims   x 32]  = V_chunk^T [128 dims x 128 tokens] . [P_hi; P_lo]^T
//
// (rows G..15 of each 16-row block of Q and P are zero; at D = 64 the QK^T
// contraction is 64 deep and PV is an M = 64 MMA over 16 KiB slots, so the
// rings hold six chunks). Both are tcgen05.mma (kind::f16,
// fp32 accumulate in TMEM) issued by one thread; the K and V tiles are
// consumed straight from the TMA-written, 128-byte-swizzled stage: K as a
// K-major A operand, V as an MN-major A operand. The probabilities P are
// written to shared memory as two bf16 (or fp16) terms, hi = rn(p) and
// lo = rn(p - hi), stacked as one 32-row operand so a single MMA multiplies
// both into O (columns g and 16 + g, added by the softmax); P keeps about
// 16 significant bits (one 8-bit operand would cost up to 2^-9 relative
// error per weight). At these small N an MMA's cost is per instruction,
// not per FLOP: one issuing thread needs ~170-185 cycles per shared-memory
// operand MMA whatever N (16 to 256), while MMAs from two issuing warps
// overlap. So the terms are stacked (half the PV instructions), and QK^T
// and PV are issued by two different warps.
//
// Warp roles (512 threads; 576 with second producers; 32 more with a second
// PV issuer):
//   warps 0-3 and 11-14: softmax, two groups of four that split the G query
//     heads' columns (group 0 the first ceil(G/2), group 1 the rest; G = 1
//     uses one group). Thread t of a group reads TMEM lane t of S (token t of
//     the chunk) for its columns, scales and masks it, joins a CTA-wide max
//     per head (shuffles + shared memory), writes p_hi/p_lo and, in group 0,
//     zeroes the V rows of tokens past the context (so 0 * stale data never
//     enters the MMA); then reads TMEM lane t of O (dim t) for its columns
//     and folds it into a running fp32 accumulator with the online-softmax
//     rescale. The two groups run the same chunk side by side. A unit's last
//     chunk is folded after the next unit's first P is written, so a unit
//     boundary does not wait for the last PV. The unit ring carries each
//     unit decoded, so no role repeats its global loads.
//   warps 4 (K) and 5 (V): producers, TMA page loads of K and of V into two
//     separate 3-slot rings (a slot is 128 tokens, 32 KiB). A K slot is
//     released as soon as its QK^T completes, a V slot after its PV, so K
//     loads run ahead. Warp 4 also takes the work units and loads each
//     unit's G query rows (a TMA box) into one of two Q operand buffers.
//     With FP8 K/V or D 64 (half the bytes per chunk) at G <= 4, warps 16
//     (K) and 17 (V) are second producers and the two warps of a ring take
//     alternate chunks (the CTA has 18 warps then, else 16).
//   warp 6: allocates 256 TMEM columns (S and O, double-buffered), issues
//     the QK^T MMAs and commits their completion to mbarriers; with FP8 K/V
//     it also turns each unit's 16-bit q tile into the two fp8 q terms.
//   warp 15: issues the PV MMAs and commits their completion. At head dim 64
//     (G <= 4, and G 5..8 with 16-bit K/V) it takes the even chunks and a
//     second PV warp the odd ones (warp 18 or 16 at G <= 4; at G 5..8 the
//     epilogue group's warp 10): an M = 64 PV needs as many MMAs per chunk
//     as M = 128 for half the bytes (a second QK^T issuer as well measured
//     no faster). The terms of a split operand (P_hi / P_lo; with FP8, q_hi /
//     q_lo and the three P terms) are stacked along N, so each contraction
//     step is one MMA.
// S, O and P are double-buffered by chunk parity so the chunks overlap:
// QK^T of chunk c+1 is issued as soon as its K tile lands (while the
// softmax warps work on chunk c), PV of chunk c once its P is written; the
// softmax warps fold O of chunk c-1 into the running output after writing P
// of chunk c.
//   warps 7-10 (7-9 when warp 10 issues PV): epilogue. A finished unit's
//     state (accumulators, max, sum) comes through a double-buffered
//     shared-memory slot; this group
//     normalises it, stores the output or the split partial, and runs the
//     split ticket and merge, while the softmax warps go on with the next
//     unit (the unit boundary does not stall the pipeline).
// Every wait is bounded; a timed-out CTA records error code 3, stops issuing
// work, still passes every barrier, counts itself done with the work counter
// (so the counters are reset for the next call) and frees its TMEM.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "pda_internal.h"
#include "ptx.cuh"
#include "split_merge.cuh"

namespace pda {
namespace tc {

constexpr int kT = 128;                    // tokens per stage = MMA M of QK^T
constexpr int kRowBytes = 128;             // one 64-element half of a 128-dim row
constexpr int kHalf = kT * kRowBytes;      // one half tile: 16 KiB
constexpr int kN = 16;                     // MMA N: the group's query heads, padded
constexpr int kOpHalf = 2048;              // 16 rows x 128 B of a K-major operand half
constexpr int kOpBytes = 2 * kOpHalf;      // Q, P_hi or P_lo operand
// Two producer warps per ring for the half-byte chunks (FP8 K/V, D 64) at
// G <= 4, whose per-chunk TMA issue kept one warp per ring busy most of the
// time; elsewhere one warp per ring measured as fast or faster, and the
// extra warps' launch size (and register cap) slowed G >= 7.
__host__ __device__ constexpr bool dual_producers(int G, int D, bool kv8) {
  return (kv8 || D == 64) && G <= 4;
}
// A second PV-issuing warp (alternate chunks) at head dim 64: its PV is an
// M = 64 MMA per 16 tokens, so one issuing thread (~185 cycles per MMA)
// needed ~1480 cycles per 128-token chunk that arrives in ~800. At G <= 4 it
// is an extra warp. At G 5..8 (16-bit K/V) a 17th warp would cut every
// thread's registers from 128 to 96 (one SM sub-partition would hold five
// warps), so it is the epilogue group's last warp (10); the epilogue then
// runs on three warps (its per-dim work needs 64 threads at D 64).
__host__ __device__ constexpr bool dual_pv(int G, int D, bool kv8) {
  return D == 64 && (G <= 4 || (!kv8 && G <= 8));
}
__host__ __device__ constexpr bool pv2_from_epilogue(int G, int D, bool kv8) {
  return dual_pv(G, D, kv8) && G >= 5;
}
__host__ __device__ constexpr int tc_threads(int G, int D, bool kv8) {
  return 512 + (dual_producers(G, D, kv8) ? 64 : 0) +
         (dual_pv(G, D, kv8) && !pv2_from_epilogue(G, D, kv8) ? 32 : 0);
}
constexpr int kWarpProducerK = 4;
constexpr int kWarpProducerV = 5;
constexpr int kWarpMma = 6;                // issues QK^T (and owns the TMEM allocation)
constexpr int kWarpEpi0 = 7;               // warps 7-10 (or 7-9): epilogue group
constexpr int kWarpSmxB0 = 11;             // warps 11-14: second softmax group
constexpr int kWarpMmaPV = 15;             // issues PV
constexpr int kWarpProducerK2 = 16;        // second K producer (odd chunks)
constexpr int kWarpProducerV2 = 17;        // second V producer (odd chunks)
// second PV issuer (odd chunks): the warp after the last producer, or at
// G 5..8 the epilogue group's last warp
__host__ __device__ constexpr int warp_pv2(int G, int D, bool kv8) {
  return pv2_from_epilogue(G, D, kv8) ? 10 : (dual_producers(G, D, kv8) ? 18 : 16);
}
// TMEM columns: S and O, double-buffered. The terms of a split operand are
// stacked along N so one MMA carries all of them (the tensor pipe's cost
// is per instruction at these small N): S holds 16 columns (32 with FP8
// K/V: q_hi and q_lo), O 32 (P_hi, P_lo; 48 with FP8: three P terms); the
// softmax adds the stacked columns of a head.
constexpr uint32_t kTmemCols = 256;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kUnitRing = 4;               // slots of the shared unit queue
// unit ring readers: V producer, both MMA warps, softmax warp 0 (+ the two
// second producers when a ring has two)
constexpr int kUnitConsumers = 4;
constexpr int kUnitInts = 12;              // a unit ring entry: index + decoded Unit
// A finished unit's state, softmax -> epilogue: acc[H][128], max[H], sum[H],
// then the unit index and its sequence's split count (as ints), for H = 8
// query heads (16 for G 9..16). Two slots, so a unit's state can wait while
// the previous one is written out; one for G 9..16 with 16-bit K/V, whose
// rings leave no room for two.
__host__ __device__ constexpr int epi_heads(int G) { return G > 8 ? 16 : 8; }
__host__ __device__ constexpr int epi_floats(int G) { return epi_heads(G) * 128 + 2 * epi_heads(G) + 4; }
__host__ __device__ constexpr int epi_slots(int G, bool kv8) { return G > 8 && !kv8 ? 1 : 2; }
constexpr float kP8Scale = 256.f;          // FP8 K/V: P is split at p * 256

// Shared-memory layout. 16-bit K/V at D 128: 3-slot rings of 32 KiB slots
// (two 64-dim halves of 128 tokens). 16-bit K/V at D 64: 6-slot rings of
// 16 KiB slots (one 64-dim half), the same bytes in flight. FP8 K/V (KV8):
// rings of 80 KiB in slots of one D-byte row per token (5 x 16 KiB at D 128,
// 10 x 8 KiB at D 64 with 64-byte swizzled rows), two fp8 terms of Q next to
// the 16-bit Q tile, three fp8 terms of P in the P buffers.
template <bool KV8, int D = 128, int G = 8>
struct Layout {
  static constexpr int kStages = KV8 ? (D == 64 ? 10 : 5) : (D == 64 ? 6 : 3);
  static constexpr int kSlotBytes = KV8 ? kT * D : (D / 64) * kHalf;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kStages * kSlotBytes;
  static constexpr int kOffQ = 2 * kStages * kSlotBytes;  // [2 buffers] Q tiles (TMA)
  static constexpr int kOffQ8 = kOffQ + 2 * kOpBytes;     // [2 buffers] fp8 Q terms (KV8)
  static constexpr int kOffP = kOffQ8 + (KV8 ? 2 * kOpBytes : 0);  // [2 buffers] P operands
  // [2 buffers][epi_heads(G)] 1/sigma per row (KV8)
  static constexpr int kOffQs = kOffP + 4 * kOpBytes;
  // per softmax group: 2 x [4 warps][8] floats (chunk maxima), [4 warps][8] (final sums)
  static constexpr int kOffRed = kOffQs + 2 * epi_heads(G) * 4;
  static constexpr int kOffLred = kOffRed + 2 * 2 * 4 * 8 * 4;
  static constexpr int kOffBar = kOffLred + 2 * 4 * 8 * 4;
  static constexpr int kNumBars = 4 * kStages + 14 + 2 * kUnitRing + 4 + 2 + 1;
  static constexpr int kOffTmem = kOffBar + kNumBars * 8;
  // [kUnitRing] unit index + decoded unit, so no reader repeats its global loads
  static constexpr int kOffURing = kOffTmem + 16;
  static constexpr int kOffUBcast = kOffURing + kUnitRing * kUnitInts * 4;  // same, softmax warp 0 -> rest
  static constexpr int kOffEpiFlag = kOffUBcast + kUnitInts * 4;  // epilogue group's wait outcome
  static constexpr int kOffEpi = (kOffEpiFlag + 4 + 15) & ~15;
  static constexpr size_t kSmemBytes = 1024 + kOffEpi + epi_slots(G, KV8) * epi_floats(G) * 4;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

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

// Same for a 32 x 128 16-bit operand (two stacked 16-row terms): 64-column
// halves of 4 KiB, each four 8-row atoms.
__device__ __forceinline__ uint32_t op32_offset(int n, int k) {
  const int half = k >> 6, col = k & 63;
  return half * (2 * kOpHalf) + (n >> 3) * 1024 + (n & 7) * 128 +
         (((col >> 3) ^ (n & 7)) << 4) + (col & 7) * 2;
}

// Byte offset of element (row n, column k) of a 16 x 128 K-major fp8 operand
// (one 128-byte row per n, 128-byte swizzle).
__device__ __forceinline__ uint32_t op8_offset(int n, int k) {
  return (n >> 3) * 1024 + (n & 7) * 128 + ((((k >> 4) ^ (n & 7))) << 4) + (k & 15);
}

// Same for a K-major fp8 operand of 64-byte rows (64-byte swizzle: the 16-byte
// chunk index XOR bits 1-2 of the row).
__device__ __forceinline__ uint32_t op8_sw64_offset(int n, int k) {
  return n * 64 + ((((k >> 4) ^ ((n >> 1) & 3))) << 4) + (k & 15);
}

// The fp8 q operand of head dim D: rows of D bytes.
template <int D>
__device__ __forceinline__ uint32_t op8q_offset(int n, int k) {
  if constexpr (D == 64) return op8_sw64_offset(n, k); else return op8_offset(n, k);
}

// Shared-memory descriptor of a swizzled operand whose rows are `row` bytes
// (128 or 64): 8-row groups `8 * row` bytes apart.
template <int kRow>
__device__ __forceinline__ uint64_t sdesc_rows(uint32_t saddr, uint32_t lbo) {
  if constexpr (kRow == 64) return sdesc_sw64(saddr, lbo, 512); else return sdesc_sw128(saddr, lbo, 1024);
}

__device__ __forceinline__ uint8_t to_e4m3(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float e4m3_to_float(uint8_t b) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
  return __half2float(__half(h));
}

// One work unit: (split, kv head, sequence) and its page / token / chunk range.
struct Unit {
  int b, h, split, n_splits_b;
  int p0, p1, t0, t1, n_chunks;
  bool zero_fill;  // an empty context whose output rows this unit writes as zeros
};

// A unit index and its decoded Unit as kUnitInts ints in shared memory
// (written by one thread, read by a whole warp).
__device__ __forceinline__ void unit_put(volatile int* d, int u, const Unit& U) {
  d[0] = u;
  d[1] = U.b;
  d[2] = U.h;
  d[3] = U.split;
  d[4] = U.n_splits_b;
  d[5] = U.p0;
  d[6] = U.p1;
  d[7] = U.t0;
  d[8] = U.t1;
  d[9] = U.n_chunks;
  d[10] = U.zero_fill ? 1 : 0;
}
__device__ __forceinline__ int unit_get(const volatile int* d, Unit& U) {
  U.b = d[1];
  U.h = d[2];
  U.split = d[3];
  U.n_splits_b = d[4];
  U.p0 = d[5];
  U.p1 = d[6];
  U.t0 = d[7];
  U.t1 = d[8];
  U.n_chunks = d[9];
  U.zero_fill = d[10] != 0;
  return d[0];
}

template <int BS>
__device__ __forceinline__ Unit load_unit(const PartialParams& p, int u) {
  constexpr int PPS = kT / BS;
  Unit U;
  U.split = u % p.num_splits;
  const int rest = u / p.num_splits;
  U.h = rest % p.Hkv;
  U.b = rest / p.Hkv;
  int L = __ldg(p.context_lens + U.b);
  const int maxL = p.max_blocks * BS;
  L = L < 0 ? 0 : (L > maxL ? maxL : L);
  const int n_pages = (L + BS - 1) / BS;
  int nsb = (n_pages + p.chunk_pages - 1) / p.chunk_pages;
  if (nsb > p.num_splits) nsb = p.num_splits;  // the last split takes the rest
  U.n_splits_b = nsb;
  U.zero_fill = (nsb == 0 && U.split == 0);
  if (U.split >= nsb) {
    U.p0 = U.p1 = U.t0 = U.t1 = U.n_chunks = 0;
    return U;
  }
  U.p0 = U.split * p.chunk_pages;
  U.p1 = (U.split == nsb - 1) ? n_pages : min(U.p0 + p.chunk_pages, n_pages);
  U.t0 = U.p0 * BS;
  U.t1 = min(U.p1 * BS, L);
  U.n_chunks = (U.p1 - U.p0 + PPS - 1) / PPS;
  return U;
}

// Units that no role has to process: neither pages nor output rows.
__device__ __forceinline__ bool unit_has_work(const Unit& U) { return U.n_chunks > 0 || U.zero_fill; }

// Block-table entries p0 + lane of unit u's sequence, with p0 the unit's first
// page, requested before the unit's context length is known (the entries
// past the sequence's pages are loaded but never used).
__device__ __forceinline__ int unit_first_window(const PartialParams& p, int u, int lane) {
  const int split = u % p.num_splits;
  const int b = u / p.num_splits / p.Hkv;
  const int idx = split * p.chunk_pages + lane;
  return idx < p.max_blocks ? __ldg(p.block_table + (int64_t)b * p.max_blocks + idx) : 0;
}

// Walks a sequence of units with work, chunk by chunk: c counts chunks over
// the whole walk (ring slots and buffer parities follow it), j counts units.
// `next()` of the source yields unit indices in order, -1 at the end; units
// without chunks (empty splits, zero-filled rows) are skipped here.
template <int BS, typename Source>
struct Cursor {
  int u, i, c, j;
  Unit U;
  __device__ __forceinline__ void seek(const PartialParams&, Source& src) {
    while ((u = src.next(U)) >= 0)
      if (U.n_chunks > 0) return;
  }
  __device__ __forceinline__ void start(const PartialParams& p, Source& src) {
    i = c = j = 0;
    seek(p, src);
  }
  __device__ __forceinline__ bool valid() const { return u >= 0; }
  __device__ __forceinline__ void advance(const PartialParams& p, Source& src) {
    ++c;
    if (++i == U.n_chunks) {
      i = 0;
      ++j;
      seek(p, src);
    }
  }
};

template <int G, int D, int BS, bool FP16, bool KV8>
__global__ void __launch_bounds__(tc_threads(G, D, KV8), 1)
    paged_partial_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v,
                            const __grid_constant__ CUtensorMap tmap_q, const PartialParams p) {
  static_assert(G >= 1 && G <= 16, "tensor-core path packs up to 16 query heads (MMA N = 16)");
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  // bytes of one token row of one head in a K/V ring slot (FP8: D, 64-byte
  // swizzled rows at D 64; 16-bit: 128, one 64-dim half)
  constexpr int kKVRow = KV8 ? D : kRowBytes;
  using L = Layout<KV8, D, G>;
  constexpr int kStages = L::kStages;
  constexpr int kSlotBytes = L::kSlotBytes;
  constexpr int kOffK = L::kOffK;
  constexpr int kOffV = L::kOffV;
  constexpr int kOffQ = L::kOffQ;
  constexpr int kOffQ8 = L::kOffQ8;
  constexpr int kOffP = L::kOffP;
  constexpr int kOffQs = L::kOffQs;
  constexpr int kOffRed = L::kOffRed;
  constexpr int kOffLred = L::kOffLred;
  constexpr int kOffBar = L::kOffBar;
  constexpr int kOffTmem = L::kOffTmem;
  constexpr int kOffURing = L::kOffURing;
  constexpr int kOffUBcast = L::kOffUBcast;
  constexpr int kOffEpiFlag = L::kOffEpiFlag;
  constexpr int kOffEpi = L::kOffEpi;
  constexpr int NB = D / 64;    // 64-dim boxes per row
  constexpr int PPS = kT / BS;  // pages per stage
  constexpr int kGroups = G >= 2 ? 2 : 1;  // softmax warp groups (query-head columns split)
  constexpr bool kDual = dual_producers(G, D, KV8);
  constexpr bool kDualPV = dual_pv(G, D, KV8);
  constexpr int kWarpMmaPV2 = warp_pv2(G, D, KV8);
  constexpr int kEpiWarps = pv2_from_epilogue(G, D, KV8) ? 3 : 4;  // epilogue group
  constexpr int kEpiThreads = 32 * kEpiWarps;
  constexpr int kGA = (G + 1) / 2 > 0 ? (G + 1) / 2 : 1;  // columns of group 0 (group 1: G - kGA)
  constexpr int kLd = kGA > 4 ? 8 : 4;      // TMEM columns a softmax thread loads per operand
  constexpr int kGE = epi_heads(G);         // heads of a state slot
  constexpr int kEpiF = epi_floats(G);      // floats of a state slot
  constexpr int kEpiSlots = epi_slots(G, KV8);
  // state slot offsets: per-head maxima, per-head sums, unit index, split count
  constexpr int kStMax = kGE * kHeadDim, kStSum = kStMax + kGE, kStU = kStSum + kGE;
  static_assert(kT % BS == 0 && PPS <= 32, "stage must hold whole pages");
  using TNat = std::conditional_t<FP16, __half, __nv_bfloat16>;
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
  auto q_full = [&](int b) { return bar0 + 8u * (4 * kStages + 10 + b); };
  auto q_empty = [&](int b) { return bar0 + 8u * (4 * kStages + 12 + b); };

  auto uring_full = [&](int s) { return bar0 + 8u * (4 * kStages + 14 + s); };
  auto uring_empty = [&](int s) { return bar0 + 8u * (4 * kStages + 14 + kUnitRing + s); };
  auto ep_full = [&](int s) { return bar0 + 8u * (4 * kStages + 14 + 2 * kUnitRing + s); };
  auto ep_empty = [&](int s) { return bar0 + 8u * (4 * kStages + 16 + 2 * kUnitRing + s); };
  // FP8 K/V: the unit's fp8 Q terms and row scales are ready (buffer b)
  auto q8_full = [&](int b) { return bar0 + 8u * (4 * kStages + 18 + 2 * kUnitRing + b); };
  // cluster launches: every other CTA of the cluster has its split's partial
  // in its state slot (one arrival per other CTA)
  const uint32_t cl_bar = bar0 + 8u * (4 * kStages + 20 + 2 * kUnitRing);
  volatile int* uring = reinterpret_cast<volatile int*>(base + kOffURing);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  bool failed = false;
  const uint64_t wlim = p.wait_ns ? (uint64_t)p.wait_ns : kWaitLimitNs;

  // Work units: CTA i starts with unit i (every role decodes it itself, so the
  // first page loads wait for no counter round trip and no ring hand-off);
  // after that the K-producer warp takes unit indices gridDim.x + k from a
  // global counter (p.sched[0]) and publishes every one that has output to
  // write into the unit ring; the V producer, the MMA warps and softmax warp 0
  // read the ring in order. The CTA that runs out last resets the counters
  // for the next call. (The grid never has more CTAs than units.)
  struct FetchSource {
    const PartialParams* p;
    volatile int* ring;
    uint32_t full0, empty0;
    int lane, k;
    bool* failed;
    uint64_t wlim;
    bool counted;
    bool first;  // the next unit is this CTA's static first unit
    // This CTA takes no more units: count it done exactly once (also after a
    // timed-out wait), so the CTA that finishes last resets the counters and
    // the next call starts from zero.
    __device__ __forceinline__ void done() {
      if (counted) return;
      counted = true;
      if (lane == 0) {
        griddep_launch_dependents();  // no more units: the next grid may start launching
        __threadfence();  // this CTA's last fetch is ordered before its done count
        if (atomicAdd(p->sched + 1, 1) == (int)gridDim.x - 1) {
          p->sched[0] = 0;
          p->sched[1] = 0;
        }
      }
      __syncwarp();
    }
    __device__ __forceinline__ int next(Unit& U) {
      if (p->stall_units) {  // fault injection: publish nothing, let every wait run out
        done();
        return -1;
      }
      if (first) {
        first = false;
        U = load_unit<BS>(*p, (int)blockIdx.x);
        if (unit_has_work(U)) return (int)blockIdx.x;
      }
      while (true) {
        int u = 0;
        if (lane == 0) u = (int)gridDim.x + atomicAdd(p->sched, 1);
        u = __shfl_sync(kFull, u, 0);
        const int pub = u < p->num_units ? u : -1;
        if (pub >= 0) {
          U = load_unit<BS>(*p, pub);
          if (!unit_has_work(U)) continue;  // nothing to do for this unit
        }
        const int slot = k % kUnitRing;
        bool ok = true;
        if (k >= kUnitRing) ok = mbar_wait(empty0 + 8u * slot, ((k / kUnitRing) - 1) & 1, wlim);
        if (!__all_sync(kFull, ok)) {
          *failed = true;
          done();
          return -1;
        }
        if (lane == 0) {
          unit_put(ring + slot * kUnitInts, pub, U);
          mbar_arrive(full0 + 8u * slot);
        }
        __syncwarp();
        ++k;
        if (pub < 0) {
          done();
          return -1;
        }
        return pub;
      }
    }
  };
  struct RingSource {
    const PartialParams* p;
    volatile int* ring;
    uint32_t full0, empty0;
    int lane, k;
    bool* failed;
    uint64_t wlim;
    bool first;  // the next unit is this CTA's static first unit
    __device__ __forceinline__ int next(Unit& U) {
      if (first) {
        first = false;
        if (!p->stall_units && !*failed) {
          U = load_unit<BS>(*p, (int)blockIdx.x);
          if (unit_has_work(U)) return (int)blockIdx.x;
        }
      }
      const int slot = k % kUnitRing;
      const bool ok = !*failed && mbar_wait(full0 + 8u * slot, (k / kUnitRing) & 1, wlim);
      if (!__all_sync(kFull, ok)) {
        *failed = true;
        return -1;
      }
      const int u = unit_get(ring + slot * kUnitInts, U);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8u * slot);
      ++k;
      return u;
    }
  };
  auto ring_source = [&]() {
    return RingSource{&p, uring, uring_full(0), uring_empty(0), lane, 0, &failed, wlim, true};
  };

  if (threadIdx.x == 0) {
    for (int s2 = 0; s2 < kUnitRing; ++s2) {
      mbar_init(uring_full(s2), 1);
      mbar_init(uring_empty(s2), kUnitConsumers + (kDual ? 2 : 0) + (kDualPV ? 1 : 0));
    }
    for (int s2 = 0; s2 < 2; ++s2) {
      mbar_init(ep_full(s2), 4 * kGroups);
      mbar_init(ep_empty(s2), kEpiWarps);
    }
    for (int r = 0; r < 2; ++r)
      for (int s = 0; s < kStages; ++s) {
        mbar_init(full_bar(r, s), 1);
        mbar_init(empty_bar(r, s), 1);
      }
    for (int b2 = 0; b2 < 2; ++b2) {
      mbar_init(s_full(b2), 1);
      mbar_init(s_free(b2), 4 * kGroups);
      mbar_init(p_full(b2), 4 * kGroups);
      mbar_init(o_full(b2), 1);
      mbar_init(o_free(b2), 4 * kGroups);
      mbar_init(q_full(b2), 1);
      // FP8 K/V: also released by each softmax group once it has read the
      // buffer's row scales
      mbar_init(q_empty(b2), KV8 ? 1 + kGroups : 1);
      mbar_init(q8_full(b2), 1);
    }
    if (p.cluster > 1) mbar_init(cl_bar, (uint32_t)(p.cluster - 1));
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(base_u32 + kOffTmem, kTmemCols);
    tmem_relinquish();
  }
  if (warp < 4) {
    // Q operands (rows G..15 stay zero; the TMA box fills rows 0..G-1) and
    // both P operand pairs start zeroed.
    for (int i = threadIdx.x; i < (kOffQs - kOffQ) / 16; i += 128)
      *reinterpret_cast<uint4*>(base + kOffQ + i * 16) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // every CTA of a cluster has initialised its barriers before any other CTA
  // may arrive on them
  if (p.cluster > 1) cluster_sync_all();
  // Everything above touches only this CTA's resources; from here on the
  // kernel reads the inputs and the shared counters, which the previous
  // grid in the stream may still be writing (programmatic dependent launch).
  griddep_wait();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(base + kOffTmem);
  constexpr int kSCols = KV8 ? 2 * kN : kN;  // S columns per buffer
  constexpr int kOCols = KV8 ? 3 * kN : 2 * kN;  // O columns per buffer
  auto tS = [&](int b2) { return tmem + (uint32_t)(b2 * kSCols); };
  auto tO = [&](int b2) { return tmem + (uint32_t)(2 * kSCols + b2 * kOCols); };

  if (!kDual && (warp == kWarpProducerK || warp == kWarpProducerV)) {
    // one producer warp per ring (this loop measured a few percent faster
    // here than the two-warp loop below run with one warp per ring)
    // ------------------- producers: K ring (warp 4), V ring (warp 5) -------------------
    const int r = warp - kWarpProducerK;
    const CUtensorMap* map = r == 0 ? &tmap_k : &tmap_v;
    if (lane == 0) {
      prefetch_tensormap(map);
      if (r == 0) prefetch_tensormap(&tmap_q);
    }
    FetchSource fetch{&p, uring, uring_full(0), uring_empty(0), lane, 0, &failed, wlim, false,
                      true};
    RingSource ring = ring_source();
    Cursor<BS, FetchSource> cur_k;
    Cursor<BS, RingSource> cur_v;
    // the first window of the static first unit, requested together with its
    // context length
    const int first_win = p.stall_units ? 0 : unit_first_window(p, (int)blockIdx.x, lane);
    if (r == 0) cur_k.start(p, fetch); else cur_v.start(p, ring);
    // block-table entries in windows of 32 pages, the next window prefetched
    int win_base = 0, win_blk = 0, nxt_blk = 0;
    while (!failed && (r == 0 ? cur_k.valid() : cur_v.valid())) {
      const int cu_i = r == 0 ? cur_k.i : cur_v.i;
      const int cu_c = r == 0 ? cur_k.c : cur_v.c;
      const int cu_j = r == 0 ? cur_k.j : cur_v.j;
      const int cu_u = r == 0 ? cur_k.u : cur_v.u;
      const Unit& U = r == 0 ? cur_k.U : cur_v.U;
      const int32_t* table = p.block_table + (int64_t)U.b * p.max_blocks;
      if (cu_i == 0) {
        win_base = U.p0;
        if (cu_j == 0 && cu_u == (int)blockIdx.x) win_blk = first_win;
        else win_blk = (U.p0 + lane < U.p1) ? __ldg(table + U.p0 + lane) : 0;
        nxt_blk = (U.p0 + 32 + lane < U.p1) ? __ldg(table + U.p0 + 32 + lane) : 0;
        if (r == 0) {
          // this unit's G query rows -> Q operand buffer j & 1
          const int qb = cu_j & 1;
          bool ok = true;
          if (cu_j >= 2) ok = mbar_wait(q_empty(qb), ((cu_j - 2) >> 1) & 1, wlim);
          if (!__all_sync(kFull, ok)) {
            failed = true;
            break;
          }
          if (lane == 0) {
            const uint32_t fb = q_full(qb);
            mbar_arrive_expect_tx(fb, (uint32_t)G * NB * kRowBytes);
            const uint32_t qdst = base_u32 + kOffQ + qb * kOpBytes;
            const int row = U.b * p.Hq + U.h * G;
#pragma unroll
            for (int bx = 0; bx < NB; ++bx) tma_load_2d(qdst + bx * kOpHalf, &tmap_q, bx * 64, row, fb);
          }
          __syncwarp();
        }
      }
      const int c = cu_c;
      const int slot = c % kStages;
      if (c >= kStages) {
        const bool ok = mbar_wait(empty_bar(r, slot), ((c / kStages) - 1) & 1, wlim);
        if (!__all_sync(kFull, ok)) {
          failed = true;
          break;
        }
      }
      const int pg0 = U.p0 + cu_i * PPS;
      const int npg = min(PPS, U.p1 - pg0);
      if (pg0 + PPS > win_base + 32) {  // pg0 == win_base + 32: PPS divides 32
        win_base += 32;
        win_blk = nxt_blk;
        nxt_blk = (win_base + 32 + lane < U.p1) ? __ldg(table + win_base + 32 + lane) : 0;
      }
      {
        const uint32_t fb = full_bar(r, slot);
        // 16-bit K/V: D / 64 boxes of 64 dims per page; FP8: one box of D bytes
        constexpr int kBoxes = KV8 ? 1 : NB;
        constexpr int kBoxElems = KV8 ? D : 64;
        if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)npg * BS * kBoxes * kKVRow);
        __syncwarp();
        // lane i issues page i's boxes
        const int bl = __shfl_sync(kFull, win_blk, (pg0 + lane - win_base) & 31);
        if (lane < npg) {
          const uint32_t st = base_u32 + (r == 0 ? kOffK : kOffV) + slot * kSlotBytes;
          const uint32_t ro = (uint32_t)(lane * BS * kKVRow);
#pragma unroll
          for (int bx = 0; bx < kBoxes; ++bx)
            tma_load_2d(st + bx * kHalf + ro, map, U.h * D + bx * kBoxElems, bl * BS, fb);
        }
      }
      __syncwarp();
      if (r == 0) cur_k.advance(p, fetch); else cur_v.advance(p, ring);
    }
    if (r == 0) fetch.done();  // counted already unless a wait timed out
  } else if (kDual && (warp == kWarpProducerK || warp == kWarpProducerV ||
                        warp == kWarpProducerK2 || warp == kWarpProducerV2)) {
    // ------- producers: K ring (warps 4, 16), V ring (warps 5, 17) -------
    // With kDual each ring has two producer warps that take alternate
    // chunks: one thread issues a TMA box in ~80 cycles, so a single warp
    // per ring spent most of a half-byte chunk's time issuing its boxes.
    // Warp 4 also takes units from the counter and loads each unit's Q; the
    // others follow the unit ring.
    const int r = (warp == kWarpProducerV || warp == kWarpProducerV2) ? 1 : 0;
    const int par = (warp == kWarpProducerK2 || warp == kWarpProducerV2) ? 1 : 0;  // chunks c % 2 == par
    const bool fetcher = warp == kWarpProducerK;
    const CUtensorMap* map = r == 0 ? &tmap_k : &tmap_v;
    if (lane == 0) {
      prefetch_tensormap(map);
      if (fetcher) prefetch_tensormap(&tmap_q);
    }
    FetchSource fetch{&p, uring, uring_full(0), uring_empty(0), lane, 0, &failed, wlim, false,
                      true};
    RingSource ring = ring_source();
    Cursor<BS, FetchSource> cur_k;
    Cursor<BS, RingSource> cur_v;
    const int first_win = p.stall_units ? 0 : unit_first_window(p, (int)blockIdx.x, lane);
    if (fetcher) cur_k.start(p, fetch); else cur_v.start(p, ring);
    // block-table entries in windows of 32 pages, the next window prefetched
    int win_base = 0, win_blk = 0, nxt_blk = 0;
    while (!failed && (fetcher ? cur_k.valid() : cur_v.valid())) {
      const int cu_i = fetcher ? cur_k.i : cur_v.i;
      const int cu_c = fetcher ? cur_k.c : cur_v.c;
      const int cu_j = fetcher ? cur_k.j : cur_v.j;
      const int cu_u = fetcher ? cur_k.u : cur_v.u;
      const Unit& U = fetcher ? cur_k.U : cur_v.U;
      const int32_t* table = p.block_table + (int64_t)U.b * p.max_blocks;
      if (cu_i == 0) {
        win_base = U.p0;
        if (cu_j == 0 && cu_u == (int)blockIdx.x) win_blk = first_win;
        else win_blk = (U.p0 + lane < U.p1) ? __ldg(table + U.p0 + lane) : 0;
        nxt_blk = (U.p0 + 32 + lane < U.p1) ? __ldg(table + U.p0 + 32 + lane) : 0;
        if (fetcher) {
          // this unit's G query rows -> Q operand buffer j & 1
          const int qb = cu_j & 1;
          bool ok = true;
          if (cu_j >= 2) ok = mbar_wait(q_empty(qb), ((cu_j - 2) >> 1) & 1, wlim);
          if (!__all_sync(kFull, ok)) {
            failed = true;
            break;
          }
          if (lane == 0) {
            const uint32_t fb = q_full(qb);
            mbar_arrive_expect_tx(fb, (uint32_t)G * NB * kRowBytes);
            const uint32_t qdst = base_u32 + kOffQ + qb * kOpBytes;
            const int row = U.b * p.Hq + U.h * G;
#pragma unroll
            for (int bx = 0; bx < NB; ++bx) tma_load_2d(qdst + bx * kOpHalf, &tmap_q, bx * 64, row, fb);
          }
          __syncwarp();
        }
      }
      const int c = cu_c;
      const bool mine = !kDual || (c & 1) == par;  // this warp's chunk
      if (mine && c >= kStages) {
        const bool ok = mbar_wait(empty_bar(r, c % kStages), ((c / kStages) - 1) & 1, wlim);
        if (!__all_sync(kFull, ok)) {
          failed = true;
          break;
        }
      }
      const int pg0 = U.p0 + cu_i * PPS;
      const int npg = min(PPS, U.p1 - pg0);
      if (pg0 + PPS > win_base + 32) {  // pg0 == win_base + 32: PPS divides 32
        win_base += 32;
        win_blk = nxt_blk;
        nxt_blk = (win_base + 32 + lane < U.p1) ? __ldg(table + win_base + 32 + lane) : 0;
      }
      if (mine) {
        const int slot = c % kStages;
        {
          const uint32_t fb = full_bar(r, slot);
          // 16-bit K/V: D / 64 boxes of 64 dims per page; FP8: one box of D bytes
          constexpr int kBoxes = KV8 ? 1 : NB;
          constexpr int kBoxElems = KV8 ? D : 64;
          if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)npg * BS * kBoxes * kKVRow);
          __syncwarp();
          // lane i issues page i's boxes
          const int bl = __shfl_sync(kFull, win_blk, (pg0 + lane - win_base) & 31);
          if (lane < npg) {
            const uint32_t st = base_u32 + (r == 0 ? kOffK : kOffV) + slot * kSlotBytes;
            const uint32_t ro = (uint32_t)(lane * BS * kKVRow);
#pragma unroll
            for (int bx = 0; bx < kBoxes; ++bx)
              tma_load_2d(st + bx * kHalf + ro, map, U.h * D + bx * kBoxElems, bl * BS, fb);
          }
        }
        __syncwarp();
      }
      if (fetcher) cur_k.advance(p, fetch); else cur_v.advance(p, ring);
    }
    if (fetcher) fetch.done();  // counted already unless a wait timed out
  } else if (warp == kWarpMma || warp == kWarpMmaPV || (kDualPV && warp == kWarpMmaPV2)) {
    // ------------------------------ MMA issue -----------------------------
    // kind::f16: type fields 1 = bf16, 0 = f16; kind::f8f6f4: 0 = E4M3
    constexpr uint32_t idesc_qk = idesc_f16(128, kSCols, !FP16 && !KV8, false, false);
    // PV has M = D: at D 64 an M = 64 MMA, whose accumulator rows 16 q .. 16 q + 15
    // sit in TMEM lanes 32 q .. 32 q + 15
    constexpr uint32_t idesc_pv = idesc_f16(D, kOCols, !FP16 && !KV8, true, false);
    // S(c) = K(c) . Q^T into S[c & 1]; needs the K slot, the unit's Q and the
    // softmax's read of S(c-2)
    auto issue_qk = [&](const Cursor<BS, RingSource>& cur) {
      const int c = cur.c, slot = c % kStages, qb = cur.j & 1;
      bool ok = !failed;
      if (ok && cur.i == 0) ok = mbar_wait(q_full(qb), (cur.j >> 1) & 1, wlim);
      if (!__all_sync(kFull, ok)) failed = true;
      if (failed) return;
      if constexpr (KV8) {
        if (cur.i == 0) {
          // The unit's q rows (16-bit tile from TMA) become two fp8 terms,
          // q * sigma = hi + lo, with a power-of-two sigma per row that puts
          // the row's largest |q| in [128, 256): the fp8 QK^T then sees q
          // exactly except for elements below 2^-10 of the row maximum.
          // Done here, not in the K producer, so the TMA rings never wait for
          // a unit's Q.
          const uint8_t* qt = base + kOffQ + qb * kOpBytes;
          uint8_t* q8 = base + kOffQ8 + qb * kOpBytes;
          float* qs = reinterpret_cast<float*>(base + kOffQs) + qb * kGE;
          const int d0 = 4 * lane;  // lanes past D read the tile's zero half
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const uint2 w = *reinterpret_cast<const uint2*>(qt + op_offset(g, d0));
            float x[4];
            if constexpr (FP16) {
              const __half2 lo2 = *reinterpret_cast<const __half2*>(&w.x);
              const __half2 hi2 = *reinterpret_cast<const __half2*>(&w.y);
              x[0] = __low2float(lo2);
              x[1] = __high2float(lo2);
              x[2] = __low2float(hi2);
              x[3] = __high2float(hi2);
            } else {
              x[0] = __uint_as_float(w.x << 16);
              x[1] = __uint_as_float(w.x & 0xffff0000u);
              x[2] = __uint_as_float(w.y << 16);
              x[3] = __uint_as_float(w.y & 0xffff0000u);
            }
            float mx = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
            int e = 0;
            if (mx > 0.f) frexpf(mx, &e);
            const float sig = ldexpf(1.f, 8 - e);
            uint32_t hw = 0, lw = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float y = x[i] * sig;
              const uint8_t hb = to_e4m3(y);
              const uint8_t lb = to_e4m3(y - e4m3_to_float(hb));
              hw |= (uint32_t)hb << (8 * i);
              lw |= (uint32_t)lb << (8 * i);
            }
            if (d0 < D) {
              *reinterpret_cast<uint32_t*>(q8 + op8q_offset<D>(g, d0)) = hw;
              *reinterpret_cast<uint32_t*>(q8 + op8q_offset<D>(kN + g, d0)) = lw;
            }
            if (lane == 0) qs[g] = 1.f / sig;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(q8_full(qb));  // the row scales, for the softmax
        }
      }
      ok = mbar_wait(full_bar(0, slot), (c / kStages) & 1, wlim);
      if (ok && c >= 2) ok = mbar_wait(s_free(c & 1), ((c - 2) >> 1) & 1, wlim);
      if (!__all_sync(kFull, ok)) failed = true;
      if (failed) return;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t kb = base_u32 + kOffK + slot * kSlotBytes;
        if constexpr (KV8) {
          // S = K . [Q_hi; Q_lo]^T (N = 32: rows 16..31 of the operand are q_lo):
          // 32 fp8 dims (32 bytes) per step
          const uint32_t q8 = base_u32 + kOffQ8 + qb * kOpBytes;
#pragma unroll
          for (int k = 0; k < D / 32; ++k) {
            const uint64_t a = sdesc_rows<kKVRow>(kb + k * 32, 16);
            const uint64_t bq = sdesc_rows<kKVRow>(q8 + k * 32, 16);
            mma_f8_ss(tS(c & 1), a, bq, idesc_qk, k > 0 ? 1u : 0u);
          }
        } else {
          const uint32_t qa = base_u32 + kOffQ + qb * kOpBytes;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t a = sdesc_sw128(kb + (k >> 2) * kHalf + (k & 3) * 32, 16, 1024);
            const uint64_t bq = sdesc_sw128(qa + (k >> 2) * kOpHalf + (k & 3) * 32, 16, 1024);
            mma_f16_ss(tS(c & 1), a, bq, idesc_qk, k > 0 ? 1u : 0u);
          }
        }
        mma_commit(s_full(c & 1));
        mma_commit(empty_bar(0, slot));                          // K slot read
        if (cur.i == cur.U.n_chunks - 1) mma_commit(q_empty(qb));  // unit's Q read
      }
      __syncwarp();
    };
    // O(c) = V(c)^T . P(c)^T into O[c & 1]; needs the V slot, P(c) and the
    // fold of O(c-2)
    auto issue_pv = [&](int c) {
      const int slot = c % kStages;
      bool ok = !failed && mbar_wait(full_bar(1, slot), (c / kStages) & 1, wlim);
      if (ok) ok = mbar_wait(p_full(c & 1), (c >> 1) & 1, wlim);
      if (ok && c >= 2) ok = mbar_wait(o_free(c & 1), ((c - 2) >> 1) & 1, wlim);
      if (!__all_sync(kFull, ok)) failed = true;
      if (failed) return;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t vb = base_u32 + kOffV + slot * kSlotBytes;
        if constexpr (KV8) {
          // O = V^T . [P_0; P_1; P_2]^T (N = 48, one 16-row block per term): V^T
          // as an MN-major fp8 A operand (all 128 dims in one 128-byte row per
          // token), 32 tokens per step
          const uint32_t p8 = base_u32 + kOffP + (c & 1) * 3 * kOpHalf;
#pragma unroll
          for (int k = 0; k < kT / 32; ++k) {
            const uint64_t a = sdesc_rows<kKVRow>(vb + k * 32 * kKVRow, kSlotBytes);
            mma_f8_ss(tO(c & 1), a, sdesc_sw128(p8 + k * 32, 16, 1024), idesc_pv,
                      k > 0 ? 1u : 0u);
          }
        }
        // O = V^T . [P_hi; P_lo]^T (N = 32): V^T as an MN-major A operand with
        // 64-dim halves kHalf apart (LBO) and 8-token row groups 1 KiB apart
        // (SBO); P as a 32-row K-major operand (64-token halves 4 KiB apart);
        // 16 tokens per step
        const uint32_t pb16 = base_u32 + kOffP + (c & 1) * 2 * kOpBytes;
#pragma unroll
        for (int k = 0; k < (KV8 ? 0 : 8); ++k) {
          const uint64_t a = sdesc_sw128(vb + k * 2048, kHalf, 1024);
          const uint32_t po = (k >> 2) * (2 * kOpHalf) + (k & 3) * 32;
          mma_f16_ss(tO(c & 1), a, sdesc_sw128(pb16 + po, 16, 1024), idesc_pv, k > 0 ? 1u : 0u);
        }
        mma_commit(o_full(c & 1));
        mma_commit(empty_bar(1, slot));  // V slot read
      }
      __syncwarp();
    };
    // Each issuing warp walks the same chunk sequence: warp 6 issues QK^T,
    // warp 15 PV. Their MMAs overlap in the tensor pipe.
    // With two PV warps, warp 15 issues the even chunks' PV and the second
    // one the odd chunks' (separate O buffers, V slots and P buffers).
    const bool is_qk = warp == kWarpMma;
    const int pv_par = (kDualPV && warp == kWarpMmaPV2) ? 1 : 0;
    RingSource ring = ring_source();
    Cursor<BS, RingSource> cur;
    cur.start(p, ring);
    int last_c = -1;
    while (!failed && cur.valid()) {
      if (is_qk) issue_qk(cur);
      else if (!kDualPV || (cur.c & 1) == pv_par) issue_pv(cur.c);
      last_c = cur.c;
      cur.advance(p, ring);
    }
    // Drain the last slots' completion arrivals of this warp's ring so that
    // no MMA commit lands on this CTA's shared memory after it exits.
    const int r = is_qk ? 0 : 1;
    for (int c = last_c - kStages + 1 > 0 ? last_c - kStages + 1 : 0; c <= last_c && !failed; ++c) {
      const bool ok = mbar_wait(empty_bar(r, c % kStages), (c / kStages) & 1, wlim);
      if (!__all_sync(kFull, ok)) failed = true;
    }
    // The QK^T warp also committed the release of the last two units' Q
    // buffers (unit j: buffer j & 1, phase (j >> 1) & 1), which no producer
    // waits for; wait for those arrivals too.
    if (is_qk) {
      for (int j = cur.j - 2 > 0 ? cur.j - 2 : 0; j < cur.j && !failed; ++j) {
        const bool ok = mbar_wait(q_empty(j & 1), (j >> 1) & 1, wlim);
        if (!__all_sync(kFull, ok)) failed = true;
      }
    }
  } else if (warp < 4 || (warp >= kWarpSmxB0 && warp < kWarpSmxB0 + 4)) {
    // ------------------------------ softmax -------------------------------
    // Group 0 (warps 0-3) takes query-head columns [0, kGA), group 1 (warps
    // 11-14, when G >= 2) columns [kGA, G). Each group has the CTA-wide max,
    // P rows and O columns of its heads to itself, so the two run the same
    // chunk side by side; they meet only at unit boundaries.
    const int grp = warp >= kWarpSmxB0 ? 1 : 0;
    if (grp < kGroups) {
      const int wq = warp & 3;        // TMEM lane quadrant: warp w reads lanes 32 (w % 4) ..
      const int t = wq * 32 + lane;   // token row of S; output dim of O (D 128)
      // D 64 (M = 64 PV): lanes 0-15 of quadrant q hold output dims 16 q .. 16 q + 15
      const int od = D == 64 ? 16 * wq + lane : t;
      const bool od_ok = D != 64 || lane < 16;
      const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
      const int g0 = grp ? kGA : 0;   // first column of this group
      const int ng = grp ? G - kGA : kGA;
      const int bar = grp ? 3 : 1;    // the group's named barrier
      float* red = reinterpret_cast<float*>(base + kOffRed) + grp * 64;
      float* lred = reinterpret_cast<float*>(base + kOffLred) + grp * 32;
      float m_run[kGA], l_th[kGA], acc[kGA], alpha_prev[kGA];
      // A unit whose last chunk is not folded yet (u_pd >= 0): its state
      // waits until the next unit's first P is written, so the unit boundary
      // does not wait for the last PV to complete.
      float m_pd[kGA], l_pd[kGA], acc_pd[kGA], alpha_pd[kGA];
      int u_pd = -1, nsb_pd = 0;  // its index and its sequence's split count
      // kLd consecutive TMEM columns of this thread's lane
      auto tld = [&](uint32_t taddr, float (&v)[kLd]) {
        if constexpr (kLd == 8) tmem_ld_x8(taddr, v); else tmem_ld_x4(taddr, v);
      };
      // a = a * al + O(c), this group's columns
      auto fold = [&](int c, float (&a)[kGA], const float (&al)[kGA]) {
        bool ok = !failed && mbar_wait(o_full(c & 1), (c >> 1) & 1, wlim);
        if (!__all_sync(kFull, ok)) failed = true;
        tc_fence_after();
        // the stacked term columns of each head: g, 16 + g (, 32 + g)
        float o[kLd], o2[kLd], o3[kLd];
        tld(tO(c & 1) + lane_base + (uint32_t)g0, o);
        tld(tO(c & 1) + lane_base + (uint32_t)(kN + g0), o2);
        if constexpr (KV8) tld(tO(c & 1) + lane_base + (uint32_t)(2 * kN + g0), o3);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < kLd; ++j) o[j] += KV8 ? o2[j] + o3[j] : o2[j];
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free(c & 1));
#pragma unroll
        for (int j = 0; j < kGA; ++j) a[j] = a[j] * al[j] + o[j];
      };
      // Softmax warp 0 alone reads the unit ring and hands the index to the
      // other softmax warps, so all walk the same units through the same
      // named barriers (a late timeout in one warp cannot split them).
      RingSource ring = ring_source();
      volatile int* ubc = reinterpret_cast<volatile int*>(base + kOffUBcast);
      Unit U;
      auto next_unit = [&]() {
        int u = -1;
        if (warp == 0) u = ring.next(U);
        if (warp == 0 && lane == 0) unit_put(ubc, u, U);
        named_bar_sync(4, 128 * kGroups);
        u = unit_get(ubc, U);
        named_bar_sync(4, 128 * kGroups);  // before warp 0 overwrites it
        return u;
      };
      int c = 0, je = 0;  // je: units handed to the epilogue group
      int jq = 0;         // units with chunks (the Q buffer sequence)
      // Hands a finished unit's state (this group's columns) to the epilogue
      // group: the softmax denominators are the per-token partial sums added
      // over the group.
      auto finish = [&](int uf, int nsb, const float (&mf)[kGA], const float (&lf)[kGA],
                        const float (&af)[kGA]) {
#pragma unroll
        for (int j = 0; j < kGA; ++j) {
          float v = lf[j];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
          if (lane == 0) lred[wq * 8 + j] = v;
        }
        named_bar_sync(bar, 128);
        float Ls[kGA];
#pragma unroll
        for (int j = 0; j < kGA; ++j) Ls[j] = lred[j] + lred[8 + j] + lred[16 + j] + lred[24 + j];
        named_bar_sync(bar, 128);  // lred is rewritten by the next unit
        const int es = je % kEpiSlots;
        bool ok2 = !failed;
        if (ok2 && je >= kEpiSlots)
          ok2 = mbar_wait(ep_empty(es), ((je - kEpiSlots) / kEpiSlots) & 1, wlim);
        if (!__all_sync(kFull, ok2)) failed = true;
        float* st = reinterpret_cast<float*>(base + kOffEpi) + es * kEpiF;
#pragma unroll
        for (int j = 0; j < kGA; ++j)
          if (j < ng && od_ok) st[(g0 + j) * kHeadDim + od] = af[j];
        if (t == 0) {
#pragma unroll
          for (int j = 0; j < kGA; ++j) {
            if (j < ng) {
              st[kStMax + g0 + j] = mf[j];
              st[kStSum + g0 + j] = Ls[j];
            }
          }
          if (grp == 0) {
            reinterpret_cast<int*>(st)[kStU] = uf;
            reinterpret_cast<int*>(st)[kStU + 1] = nsb;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(ep_full(es));
        ++je;
      };
      for (int u = next_unit(); u >= 0; u = next_unit()) {
        const int hq0 = U.h * G;
        if (U.zero_fill && grp == 0) {
          for (int i = t; i < G * D; i += 128) {
            const int64_t o = ((int64_t)U.b * p.Hq + hq0) * D + i;
            if (p.out_f32) static_cast<float*>(p.out)[o] = 0.f;
            else static_cast<TNat*>(p.out)[o] = to_out<TNat>(0.f);
          }
        }
        if (U.n_chunks == 0) continue;
#pragma unroll
        for (int j = 0; j < kGA; ++j) {
          m_run[j] = -INFINITY;
          l_th[j] = 0.f;
          acc[j] = 0.f;
        }
        // logit scale per row: softmax scale (base 2) x K dequantisation
        // scale (x 1 / sigma of the row's fp8 q terms)
        const float ksc = p.k_scale ? __ldg(p.k_scale + (p.scale_per_head ? U.h : 0)) : 1.f;
        float qsc[kGA];
        if constexpr (KV8) {
          const bool okq = !failed && mbar_wait(q8_full(jq & 1), (jq >> 1) & 1, wlim);
          if (!__all_sync(kFull, okq)) failed = true;
          const float* qs = reinterpret_cast<const float*>(base + kOffQs) + (jq & 1) * kGE;
#pragma unroll
          for (int j = 0; j < kGA; ++j) qsc[j] = j < ng ? p.qscale * ksc * qs[g0 + j] : 0.f;
        } else {
#pragma unroll
          for (int j = 0; j < kGA; ++j) qsc[j] = p.qscale * ksc;
        }
        for (int i = 0; i < U.n_chunks; ++i, ++c) {
          const int slot = c % kStages;
          const int n_valid = min(kT, U.t1 - (U.t0 + i * kT));
          bool ok = !failed && mbar_wait(s_full(c & 1), (c >> 1) & 1, wlim);
          if (!__all_sync(kFull, ok)) failed = true;
          tc_fence_after();
          float s[kLd], s2[kLd];
          tld(tS(c & 1) + lane_base + (uint32_t)g0, s);
          if constexpr (KV8) tld(tS(c & 1) + lane_base + (uint32_t)(kN + g0), s2);
          tmem_ld_wait();
          if constexpr (KV8) {
#pragma unroll
            for (int j = 0; j < kLd; ++j) s[j] += s2[j];
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_free(c & 1));
#pragma unroll
          for (int j = 0; j < kGA; ++j) s[j] = (t < n_valid) ? s[j] * qsc[j] : -INFINITY;
          float* rb = red + (c & 1) * 32;
#pragma unroll
          for (int j = 0; j < kGA; ++j) {
            float mx = s[j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
            if (lane == 0) rb[wq * 8 + j] = mx;
          }
          named_bar_sync(bar, 128);
          // every softmax thread has read the row scales of this unit's Q buffer
          if (KV8 && i == 0 && t == 0) mbar_arrive(q_empty(jq & 1));
          float alpha[kGA], prs[kGA];
          uint8_t* pb = base + kOffP + (c & 1) * (KV8 ? 3 * kOpHalf : 2 * kOpBytes);
          // Every column's maxima are read before any P store: the byte and
          // 16-bit P stores may alias the float buffer as far as the compiler
          // knows, so interleaved they would serialise the columns.
#pragma unroll
          for (int j = 0; j < kGA; ++j) {
            const float mx = fmaxf(fmaxf(rb[j], rb[8 + j]), fmaxf(rb[16 + j], rb[24 + j]));
            const float mn = fmaxf(m_run[j], mx);  // finite: every chunk holds a valid token
            alpha[j] = exp2f(m_run[j] - mn);
            m_run[j] = mn;
            prs[j] = exp2f(s[j] - mn);
            l_th[j] = l_th[j] * alpha[j] + prs[j];
          }
#pragma unroll
          for (int j = 0; j < kGA; ++j) {
            const float pr = prs[j];
            if (j < ng) {  // rows of padding heads stay zero
              const int g = g0 + j;
              if constexpr (KV8) {
                // p * 256 = t0 + t1 + t2 in fp8 (about 12 significant bits)
                const float x = pr * kP8Scale;
                const uint8_t b0 = to_e4m3(x);
                const float r0 = x - e4m3_to_float(b0);
                const uint8_t b1 = to_e4m3(r0);
                const uint8_t b2 = to_e4m3(r0 - e4m3_to_float(b1));
                const uint32_t off = op8_offset(g, t);
                pb[off] = b0;
                pb[kOpHalf + off] = b1;
                pb[2 * kOpHalf + off] = b2;
              } else {
                const typename H::T hi = H::from(pr);
                const typename H::T lo = H::from(pr - H::to(hi));
                *reinterpret_cast<typename H::T*>(pb + op32_offset(g, t)) = hi;
                *reinterpret_cast<typename H::T*>(pb + op32_offset(kN + g, t)) = lo;
              }
            }
          }
          if (grp == 0 && n_valid < kT) {
            // keep stale or out-of-context V rows out of the MMA; the V tile
            // of this chunk must have landed first (its last page may be partial)
            ok = !failed && mbar_wait(full_bar(1, slot), (c / kStages) & 1, wlim);
            if (!__all_sync(kFull, ok)) failed = true;
            if (t >= n_valid) {
              uint8_t* vrow = base + kOffV + slot * kSlotBytes + t * kKVRow;
#pragma unroll
              for (int hh = 0; hh < (KV8 ? 1 : NB); ++hh)
#pragma unroll
                for (int q = 0; q < kKVRow / 16; ++q)
                  *reinterpret_cast<uint4*>(vrow + hh * kHalf + q * 16) = make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_full(c & 1));
          if (i > 0) {
            fold(c - 1, acc, alpha_prev);
          } else if (u_pd >= 0) {
            // the previous unit's last chunk
            fold(c - 1, acc_pd, alpha_pd);
            finish(u_pd, nsb_pd, m_pd, l_pd, acc_pd);
            u_pd = -1;
          }
#pragma unroll
          for (int j = 0; j < kGA; ++j) alpha_prev[j] = alpha[j];
        }
#pragma unroll
        for (int j = 0; j < kGA; ++j) {
          m_pd[j] = m_run[j];
          l_pd[j] = l_th[j];
          acc_pd[j] = acc[j];
          alpha_pd[j] = alpha_prev[j];
        }
        u_pd = u;
        nsb_pd = U.n_splits_b;
        ++jq;
      }
      if (u_pd >= 0) {
        fold(c - 1, acc_pd, alpha_pd);
        finish(u_pd, nsb_pd, m_pd, l_pd, acc_pd);
      }
      // end of work: an empty state tells the epilogue group to stop
      {
        const int es = je % kEpiSlots;
        bool ok2 = !failed;
        if (ok2 && je >= kEpiSlots)
          ok2 = mbar_wait(ep_empty(es), ((je - kEpiSlots) / kEpiSlots) & 1, wlim);
        if (!__all_sync(kFull, ok2)) failed = true;
        float* st = reinterpret_cast<float*>(base + kOffEpi) + es * kEpiF;
        if (grp == 0 && t == 0) reinterpret_cast<int*>(st)[kStU] = -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(ep_full(es));
      }
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const int t = threadIdx.x - kWarpEpi0 * 32;  // output dim
    volatile int* flag = reinterpret_cast<volatile int*>(base + kOffEpiFlag);
    for (int je = 0;; ++je) {
      const int es = je % kEpiSlots;
      const bool ok = !failed && mbar_wait(ep_full(es), (je / kEpiSlots) & 1, wlim);
      // the four warps agree on the outcome before acting on it
      if (t == 0) *flag = 0;
      named_bar_sync(2, kEpiThreads);
      if (!ok && lane == 0) *flag = 1;
      named_bar_sync(2, kEpiThreads);
      if (*flag) {
        failed = true;
        break;
      }
      float* st = reinterpret_cast<float*>(base + kOffEpi) + es * kEpiF;
      const int u = reinterpret_cast<volatile int*>(st)[kStU];
      if (u < 0) {
        // a cluster CTA whose split had nothing to merge still counts toward
        // the other CTAs' merge barriers
        if (p.cluster > 1 && je == 0 && t == 0) {
          const uint32_t me = cluster_ctarank();
          for (int q = 0; q < p.cluster; ++q)
            if (q != (int)me) mbar_arrive_remote(cluster_map(cl_bar, (uint32_t)q));
        }
        break;
      }
      // the unit from its index alone (no global load on this path): its
      // split, kv head and sequence, and the sequence's split count
      Unit U;
      U.split = u % p.num_splits;
      U.h = (u / p.num_splits) % p.Hkv;
      U.b = u / p.num_splits / p.Hkv;
      U.n_splits_b = reinterpret_cast<volatile int*>(st)[kStU + 1];
      const int hq0 = U.h * G;
      // V dequantisation scale (and the fp8 split factor of P)
      const float vsc = (p.v_scale ? __ldg(p.v_scale + (p.scale_per_head ? U.h : 0)) : 1.f) *
                        (KV8 ? 1.f / kP8Scale : 1.f);
      if (p.cluster > 1 && U.n_splits_b > 1) {
        // Cluster launch: this split's normalised partial and log-sum-exp stay
        // in this CTA's state slot; once every other CTA of the cluster has
        // signalled, each split with pages merges its share of the outputs,
        // reading the other splits' slots through distributed shared memory.
        if (t < D) {
#pragma unroll
          for (int g = 0; g < G; ++g) st[g * kHeadDim + t] = st[g * kHeadDim + t] / st[kStSum + g] * vsc;
        }
        if (t == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g)
            st[kStMax + g] = (st[kStMax + g] + log2f(st[kStSum + g])) * kLn2;
        }
        named_bar_sync(2, kEpiThreads);  // this CTA's slot holds its split's o and lse
        if (t == 0) {
          fence_acq_rel_cluster();
          for (int q = 0; q < p.cluster; ++q)
            if (q != U.split) mbar_arrive_remote(cluster_map(cl_bar, (uint32_t)q));
        }
        const bool okm = mbar_wait_cluster(cl_bar, 0, wlim);
        if (!__all_sync(kFull, okm)) failed = true;
        if (!failed) {
          // this split's share of the G x D outputs, each merged over the
          // sequence's splits with all their loads in flight together
          const int nsb = U.n_splits_b;
          const int per = (G * D + nsb - 1) / nsb;
          const int lo = U.split * per, hi = min(G * D, lo + per);
          const uint32_t st_u32 = smem_u32(st);
          for (int oi = lo + t; oi < hi; oi += kEpiThreads) {
            const int g = oi / D, d = oi - g * D;
            // groups of 8 splits, a running maximum across the groups
            float M = -INFINITY, wsum = 0.f, acc = 0.f;
            for (int s0 = 0; s0 < nsb; s0 += 8) {
              float l[8], v[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                if (s0 + k < nsb) {
                  const uint32_t rb = cluster_map(st_u32, (uint32_t)(s0 + k));
                  l[k] = ld_cluster_f32(rb + (uint32_t)(kStMax + g) * 4u);
                  v[k] = ld_cluster_f32(rb + (uint32_t)(g * kHeadDim + d) * 4u);
                }
              }
              float Mn = M;
#pragma unroll
              for (int k = 0; k < 8; ++k)
                if (s0 + k < nsb) Mn = fmaxf(Mn, l[k]);
              const float r = exp2f((M - Mn) * kLog2e);  // 0 on the first group
              wsum *= r;
              acc *= r;
              M = Mn;
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                if (s0 + k < nsb) {
                  const float w = exp2f((l[k] - M) * kLog2e);
                  wsum += w;
                  acc = fmaf(w, v[k], acc);
                }
              }
            }
            const int64_t row = (int64_t)U.b * p.Hq + hq0 + g;
            if (p.out_f32) static_cast<float*>(p.out)[row * D + d] = acc / wsum;
            else static_cast<TNat*>(p.out)[row * D + d] = to_out<TNat>(acc / wsum);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(ep_empty(es));
        continue;
      }
      if (t < D) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float Ls = st[kStSum + g];
          const float o = st[g * kHeadDim + t] / Ls * vsc;
          const int64_t row = (int64_t)U.b * p.Hq + hq0 + g;
          if (U.n_splits_b == 1) {
            if (p.out_f32) static_cast<float*>(p.out)[row * D + t] = o;
            else static_cast<TNat*>(p.out)[row * D + t] = to_out<TNat>(o);
          } else {
            const int64_t r = row * p.num_splits + U.split;
            p.ws_o[r * D + t] = o;
            if (t == 0) p.ws_lse[r] = (st[kStMax + g] + log2f(Ls)) * kLn2;
          }
        }
      }
      named_bar_sync(2, kEpiThreads);  // the state is read; the slot serves as merge scratch
      // the last split of this (sequence, kv head) merges all of them into `out`
      if (U.n_splits_b > 1) {
        // merge loads in flight per thread: fewer with the 576-thread launch,
        // whose register budget is smaller
        constexpr int kMergeChunk = kDual ? 4 : 8;
        if (p.out_f32) finish_split<G, D, float, kMergeChunk, kEpiThreads>(p, U.b, U.h, U.n_splits_b, t, st, 2);
        else finish_split<G, D, TNat, kMergeChunk, kEpiThreads>(p, U.b, U.h, U.n_splits_b, t, st, 2);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(ep_empty(es));
    }
  }

  if (failed && lane == 0 && atomicCAS(p.err, 0, kErrWaitTimeout) == 0) p.err[1] = blockIdx.x;
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // no CTA of a cluster leaves while another may still read its shared memory
  // or arrive on its barriers
  if (p.cluster > 1) cluster_sync_all();
}

template <int G, int D, int BS, bool FP16, bool KV8>
cudaError_t launch_one(const CUtensorMap* tk, const CUtensorMap* tv, const CUtensorMap* tq,
                       const PartialParams& p, cudaStream_t stream) {
  const int ctas = p.num_units < p.max_ctas ? p.num_units : p.max_ctas;
  if (ctas <= 0) return cudaSuccess;
  // Programmatic dependent launch (off with PDA_PDL=0): the CTAs may start
  // their set-up while the previous grid in the stream finishes; the kernel
  // waits for that grid before reading any input.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(tc_threads(G, D, KV8));
  cfg.dynamicSmemBytes = Layout<KV8, D, G>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n_attr = 0;
  if (pdl_enabled()) {
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
    ++n_attr;
  }
  if (p.cluster > 1) {
    // one CTA per unit, clusters of the p.cluster splits of one (sequence, kv head)
    if (p.num_units % p.cluster != 0) return cudaErrorInvalidValue;
    cfg.gridDim = dim3((unsigned)p.num_units);
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = (unsigned)p.cluster;
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr].val.clusterDim.z = 1;
    ++n_attr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n_attr;
  return cudaLaunchKernelEx(&cfg, paged_partial_tc_kernel<G, D, BS, FP16, KV8>, *tk, *tv, *tq, p);
}

template <int G, int D, int BS, bool FP16, bool KV8>
int max_clusters_one(int cluster) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cluster * 64u);
  cfg.blockDim = dim3(tc_threads(G, D, KV8));
  cfg.dynamicSmemBytes = Layout<KV8, D, G>::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, paged_partial_tc_kernel<G, D, BS, FP16, KV8>, &cfg) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int G, int D, int BS, bool FP16, bool KV8>
cudaError_t prepare_one() {
  cudaError_t e = cudaFuncSetAttribute(paged_partial_tc_kernel<G, D, BS, FP16, KV8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Layout<KV8, D, G>::kSmemBytes);
  // clusters of up to 16 CTAs (the splits of one sequence's kv head)
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(paged_partial_tc_kernel<G, D, BS, FP16, KV8>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

template <int G, int D, int BS, bool FP16, bool KV8>
int occupancy_one() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, paged_partial_tc_kernel<G, D, BS, FP16, KV8>, tc_threads(G, D, KV8),
          Layout<KV8, D, G>::kSmemBytes) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

// 16-bit K/V: G 3..16 (G 1 and 2 go to the CUDA-core kernel), D 64 or 128.
// FP8 K/V: any G up to 16, D 64 or 128, bf16 or fp16 queries.
__host__ __device__ constexpr bool geometry_supported(int G, int D, bool kv8 = false) {
  return kv8 ? (G >= 1 && G <= 16 && (D == 64 || D == 128))
             : (G >= 3 && G <= 16 && (D == 64 || D == 128));
}

// Dispatch over (G, block size 16 or 32, and 64 for G <= 8) for one head dim,
// input dtype and K/V type;
// each (head dim, dtype, K/V type) and G range GLo..GHi is instantiated in its
// own translation unit (G 1..8 and G 9..16 compile in parallel).
template <int D, bool FP16, bool KV8, int GLo = 1, int GHi = 8>
struct Dispatch {
  template <int G>
  static constexpr bool kBuilt = G >= GLo && G <= GHi && geometry_supported(G, D, KV8);
  template <int G>
  static cudaError_t launch_g(int BS, const CUtensorMap* tk, const CUtensorMap* tv,
                              const CUtensorMap* tq, const PartialParams& p, cudaStream_t s) {
    if constexpr (kBuilt<G>) {
      if (BS == 16) return launch_one<G, D, 16, FP16, KV8>(tk, tv, tq, p, s);
      if (BS == 32) return launch_one<G, D, 32, FP16, KV8>(tk, tv, tq, p, s);
      if constexpr (G <= 8)
        if (BS == 64) return launch_one<G, D, 64, FP16, KV8>(tk, tv, tq, p, s);
    }
    return cudaErrorInvalidValue;
  }
  template <int G>
  static cudaError_t prepare_g(int BS) {
    if constexpr (kBuilt<G>) {
      if (BS == 16) return prepare_one<G, D, 16, FP16, KV8>();
      if (BS == 32) return prepare_one<G, D, 32, FP16, KV8>();
      if constexpr (G <= 8)
        if (BS == 64) return prepare_one<G, D, 64, FP16, KV8>();
    }
    return cudaErrorInvalidValue;
  }
  template <int G>
  static int max_clusters_g(int BS, int cluster) {
    if constexpr (kBuilt<G>) {
      if (BS == 16) return max_clusters_one<G, D, 16, FP16, KV8>(cluster);
      if (BS == 32) return max_clusters_one<G, D, 32, FP16, KV8>(cluster);
      if constexpr (G <= 8)
        if (BS == 64) return max_clusters_one<G, D, 64, FP16, KV8>(cluster);
    }
    return 0;
  }
  template <int G>
  static int occupancy_g(int BS) {
    if constexpr (kBuilt<G>) {
      if (BS == 16) return occupancy_one<G, D, 16, FP16, KV8>();
      if (BS == 32) return occupancy_one<G, D, 32, FP16, KV8>();
      if constexpr (G <= 8)
        if (BS == 64) return occupancy_one<G, D, 64, FP16, KV8>();
    }
    return 1;
  }
  static cudaError_t launch(int G, int BS, const CUtensorMap* tk, const CUtensorMap* tv,
                            const CUtensorMap* tq, const PartialParams& p, cudaStream_t s) {
    switch (G) {
      case 1: return launch_g<1>(BS, tk, tv, tq, p, s);
      case 2: return launch_g<2>(BS, tk, tv, tq, p, s);
      case 3: return launch_g<3>(BS, tk, tv, tq, p, s);
      case 4: return launch_g<4>(BS, tk, tv, tq, p, s);
      case 5: return launch_g<5>(BS, tk, tv, tq, p, s);
      case 6: return launch_g<6>(BS, tk, tv, tq, p, s);
      case 7: return launch_g<7>(BS, tk, tv, tq, p, s);
      case 8: return launch_g<8>(BS, tk, tv, tq, p, s);
      case 9: return launch_g<9>(BS, tk, tv, tq, p, s);
      case 10: return launch_g<10>(BS, tk, tv, tq, p, s);
      case 11: return launch_g<11>(BS, tk, tv, tq, p, s);
      case 12: return launch_g<12>(BS, tk, tv, tq, p, s);
      case 13: return launch_g<13>(BS, tk, tv, tq, p, s);
      case 14: return launch_g<14>(BS, tk, tv, tq, p, s);
      case 15: return launch_g<15>(BS, tk, tv, tq, p, s);
      case 16: return launch_g<16>(BS, tk, tv, tq, p, s);
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
      case 9: return prepare_g<9>(BS);
      case 10: return prepare_g<10>(BS);
      case 11: return prepare_g<11>(BS);
      case 12: return prepare_g<12>(BS);
      case 13: return prepare_g<13>(BS);
      case 14: return prepare_g<14>(BS);
      case 15: return prepare_g<15>(BS);
      case 16: return prepare_g<16>(BS);
      default: return cudaErrorInvalidValue;
    }
  }
  static int max_clusters(int G, int BS, int cluster) {
    switch (G) {
      case 1: return max_clusters_g<1>(BS, cluster);
      case 2: return max_clusters_g<2>(BS, cluster);
      case 3: return max_clusters_g<3>(BS, cluster);
      case 4: return max_clusters_g<4>(BS, cluster);
      case 5: return max_clusters_g<5>(BS, cluster);
      case 6: return max_clusters_g<6>(BS, cluster);
      case 7: return max_clusters_g<7>(BS, cluster);
      case 8: return max_clusters_g<8>(BS, cluster);
      case 9: return max_clusters_g<9>(BS, cluster);
      case 10: return max_clusters_g<10>(BS, cluster);
      case 11: return max_clusters_g<11>(BS, cluster);
      case 12: return max_clusters_g<12>(BS, cluster);
      case 13: return max_clusters_g<13>(BS, cluster);
      case 14: return max_clusters_g<14>(BS, cluster);
      case 15: return max_clusters_g<15>(BS, cluster);
      case 16: return max_clusters_g<16>(BS, cluster);
      default: return 0;
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
      case 9: return occupancy_g<9>(BS);
      case 10: return occupancy_g<10>(BS);
      case 11: return occupancy_g<11>(BS);
      case 12: return occupancy_g<12>(BS);
      case 13: return occupancy_g<13>(BS);
      case 14: return occupancy_g<14>(BS);
      case 15: return occupancy_g<15>(BS);
      case 16: return occupancy_g<16>(BS);
      default: return 1;
    }
  }
};

}  // namespace tc
}  // namespace pda
