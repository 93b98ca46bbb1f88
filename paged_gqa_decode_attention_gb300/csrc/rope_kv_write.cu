// RoPE + paged-KV write (Loom Kernels landing page, "Supported now": "RoPE +
// paged-KV write - packed Q/K rotation + native cache write"): the step of a
// decode (or prefill) iteration that rotates the new tokens' query and key
// heads and stores the key and value heads into the paged cache the decode
// kernel reads, in one launch.
//
// For token t at position pos_t, table row cs = cos_sin[pos_t] (rot_dim
// floats: rot_dim/2 cosines, then rot_dim/2 sines) and rotated pair j:
//   (a, b) = (j, j + rot_dim/2)  rotate-halves      or  (2j, 2j + 1)  interleaved
//   y_a = x_a cos_j - x_b sin_j,   y_b = x_b cos_j + x_a sin_j,
// dims >= rot_dim unchanged. q heads go to q_out; rotated k heads and the
// unchanged v heads go to cache row slot_mapping[t] ([num_slots, Hkv, D],
// i.e. [num_blocks, block_size, Hkv, D] with slot = block * block_size + offset).
//
// Exactly rounded: every output is the storage-format rounding (to nearest,
// ties to even) of the double-precision value of the formula, the same result
// the FP64 definition gives. The fast path computes y in fp32 with one fused
// multiply-add and a proven error bound; if the rounding of the bound's two
// ends agrees, that is the answer, otherwise (about one element in 2^14) the
// pair is recomputed in double and rounded through a round-to-odd float
// (Boldo and Melquiond, "Emulation of FMA and correctly rounded sums: proved
// algorithms using rounding to odd", 2008), which avoids double rounding.
//
// Memory-bound: token rows move through shared memory by bulk asynchronous
// copies (no registers hold data in flight), so a ring of up to six ~16 KB
// tiles per CTA keeps enough bytes in flight to stream at HBM speed, and a
// dedicated mover warp lets the rotation of one tile overlap the copies of
// the others.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <string>

#include <mutex>

#include "paged_decode_attn.h"
#include "pda_internal.h"
#include "ptx.cuh"

namespace pda {
namespace {

constexpr int kRopeRotWarps = 8;                   // warps that rotate
constexpr int kRopeRotThreads = kRopeRotWarps * 32;
constexpr int kRopeThreads = kRopeRotThreads + 32;  // + the mover warp

struct RopeParams {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  int64_t q_stride;   // elements between consecutive tokens
  int64_t k_stride;
  int64_t v_stride;
  int64_t qo_stride;
  const int32_t* positions;  // [T]
  const int64_t* slots;      // [T]
  const float* cos_sin;      // [max_position, rot_dim]
  uint16_t* q_out;
  uint16_t* k_cache;         // [num_slots, Hkv, D]
  uint16_t* v_cache;
  int* err;                  // optional {code, detail}
  int64_t num_slots;
  int T, Hq, Hkv, D, rot_dim, max_position;
  int row_elems;    // (Hq + 2 Hkv) * D: one token's staged row
  int tile_tokens;  // tokens per tile (<= 32)
  int num_tiles;
  uint32_t div_tok_mul, div_tok_shift;  // x / per_token == (x * mul) >> shift
  uint32_t div_rot_mul, div_rot_shift;  // x / rot_items
  int stages;       // ring stages (<= kRopeMaxStages)
  int lag;          // a stage is refilled `lag` tiles after its stores were issued
  int fused;        // q, k, v are consecutive parts of one [T, row_elems] buffer
};

struct Bf16 {
  static __device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
  static __device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
  // (RN(x) in the low half, RN(y) in the high half)
  static __device__ __forceinline__ uint32_t pack2(float x, float y) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
};

struct Fp16 {
  static __device__ __forceinline__ float lo_f(uint32_t w) {
    return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
  }
  static __device__ __forceinline__ float hi_f(uint32_t w) {
    return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
  }
  static __device__ __forceinline__ uint32_t pack2(float x, float y) {
    const __half2 h = __floats2half2_rn(x, y);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
};

// Round-to-odd conversion double -> float: truncate, then set the last bit
// if anything was cut off. Rounding that float to a format with at least two
// fewer significant bits (bf16: 8, fp16: 11, float: 24) gives the correctly
// rounded result of the double.
__device__ __forceinline__ float round_to_odd_float(double d) {
  const float f = __double2float_rz(d);
  return ((double)f != d) ? __uint_as_float(__float_as_uint(f) | 1u) : f;
}

// Two outputs, packed: RN_fmt(a0*b0 + c0*d0) in the low half and
// RN_fmt(a1*b1 + c1*d1) in the high half, for storage-format values a, c and
// fp32 b, d; equal to rounding the double-precision value (a*b and c*d are
// exact in double, the sum is rounded once) to the format.
// Fast path: r = fma(a, b, fl(c*d)) is within 2^-24 (|fl(c*d)| + |r|)(1 + 2^-23)
// + 2^-149 of the exact value; m is twice that bound. If rounding r - m down
// and r + m up gives the same storage values, the exact values, inside
// [r - m, r + m], round to them too. Otherwise (about one output in 10^4)
// both are recomputed in double and rounded through a round-to-odd float.
// The bound is kept tight (per output) because a warp takes the slow path
// whenever one of its lanes does.
template <typename F>
__device__ __forceinline__ uint32_t rounded_dot2_x2(float a0, float b0, float c0, float d0,
                                                    float a1, float b1, float c1, float d1) {
  const float p0 = __fmul_rn(c0, d0), p1 = __fmul_rn(c1, d1);
  const float r0 = __fmaf_rn(a0, b0, p0), r1 = __fmaf_rn(a1, b1, p1);
  const float m0 = __fmaf_rn(fabsf(p0) + fabsf(r0), 0x1p-23f, 0x1p-147f);
  const float m1 = __fmaf_rn(fabsf(p1) + fabsf(r1), 0x1p-23f, 0x1p-147f);
  const uint32_t lo = F::pack2(__fsub_rd(r0, m0), __fsub_rd(r1, m1));
  const uint32_t hi = F::pack2(__fadd_ru(r0, m0), __fadd_ru(r1, m1));
  if (lo == hi) return lo;
  const double e0 = __dadd_rn(__dmul_rn((double)a0, (double)b0), __dmul_rn((double)c0, (double)d0));
  const double e1 = __dadd_rn(__dmul_rn((double)a1, (double)b1), __dmul_rn((double)c1, (double)d1));
  return F::pack2(round_to_odd_float(e0), round_to_odd_float(e1));
}

__device__ __forceinline__ int fast_div(int x, uint32_t mul, uint32_t shift) {
  return (int)(((uint64_t)(uint32_t)x * mul) >> shift);
}

__device__ __forceinline__ void record_error(int* err, int code, int detail) {
  if (err != nullptr && atomicCAS(err, 0, code) == 0) err[1] = detail;
}

constexpr int kRopeMaxStages = 6;
constexpr int kRopeDataOff = 128;           // 2 x kRopeMaxStages mbarriers first
constexpr int kRopeStageTarget = 16 * 1024;  // bytes of token rows per stage
constexpr int kRopeRingBytes = 192 * 1024;   // at most, for the whole ring
constexpr int kRopeMaxRowBytes = 48 * 1024;
constexpr int kRopeMaxTileTokens = 32;       // one lane of warp 0 per token

// Rotates the pairs of one 32-byte item in shared memory: angles j = 8u ..
// 8u + 7 of a head row, elements at offA and offB (16-byte vectors).
template <typename F, bool kNeox>
__device__ __forceinline__ void rotate_item(uint16_t* row, const float* cs_row, int half, int u) {
  const int offA = kNeox ? 8 * u : 16 * u;
  const int offB = kNeox ? half + 8 * u : 16 * u + 8;
  uint4* pa = reinterpret_cast<uint4*>(row + offA);
  uint4* pb = reinterpret_cast<uint4*>(row + offB);
  const uint4 A = *pa, B = *pb;
  const float* cs = cs_row + 8 * u;
  const float4 c0 = __ldg(reinterpret_cast<const float4*>(cs));
  const float4 c1 = __ldg(reinterpret_cast<const float4*>(cs + 4));
  const float4 s0 = __ldg(reinterpret_cast<const float4*>(cs + half));
  const float4 s1 = __ldg(reinterpret_cast<const float4*>(cs + half + 4));
  const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  const uint32_t wa[4] = {A.x, A.y, A.z, A.w};
  const uint32_t wb[4] = {B.x, B.y, B.z, B.w};
  uint32_t oa[4], ob[4];
  if constexpr (kNeox) {
    // pair i = (element i of A, element i of B); word w holds pairs 2w, 2w+1
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float a0 = F::lo_f(wa[w]), a1 = F::hi_f(wa[w]);
      const float b0 = F::lo_f(wb[w]), b1 = F::hi_f(wb[w]);
      const float cc0 = c[2 * w], cc1 = c[2 * w + 1], ss0 = s[2 * w], ss1 = s[2 * w + 1];
      oa[w] = rounded_dot2_x2<F>(a0, cc0, -b0, ss0, a1, cc1, -b1, ss1);
      ob[w] = rounded_dot2_x2<F>(b0, cc0, a0, ss0, b1, cc1, a1, ss1);
    }
  } else {
    // pair i = the two halves of word i of A (i < 4) or of B (i >= 4)
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float a = F::lo_f(wa[w]), b = F::hi_f(wa[w]);
      oa[w] = rounded_dot2_x2<F>(a, c[w], -b, s[w], b, c[w], a, s[w]);
      a = F::lo_f(wb[w]);
      b = F::hi_f(wb[w]);
      ob[w] = rounded_dot2_x2<F>(a, c[4 + w], -b, s[4 + w], b, c[4 + w], a, s[4 + w]);
    }
  }
  *pa = make_uint4(oa[0], oa[1], oa[2], oa[3]);
  *pb = make_uint4(ob[0], ob[1], ob[2], ob[3]);
}

// Persistent CTAs walk tiles of tile_tokens tokens (local tile i is tile
// blockIdx.x + i * gridDim.x), through a ring of p.stages shared-memory
// stages laid out [token][q heads | k heads | v heads][D].
//   warp 8 (mover): bulk-loads each tile's rows into its stage (one copy
//     when q, k, v are one contiguous fused buffer, else three per token);
//     once the rotating warps have released a stage, bulk-stores every
//     token's q row to q_out and its k and v rows to the cache slot (one
//     store group per lane), and refills a stage as soon as the stores of
//     the tile it held have read it.
//   warps 0-7 (rotators): wait for a stage, rotate its q and k pairs in
//     place, release it. They never wait for stores, so up to
//     stages - lag tiles of loads stay in flight ahead of the rotation.
// No block-wide barrier inside the loop; every wait is bounded.
template <typename F, bool kNeox>
__global__ void __launch_bounds__(kRopeThreads, 3) rope_kv_write_kernel(const RopeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* done = full + kRopeMaxStages;
  const int K = p.stages, lag = p.lag;
  uint16_t* data = reinterpret_cast<uint16_t*>(smem + kRopeDataOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_local = (p.num_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int64_t stage_elems = (int64_t)p.tile_tokens * p.row_elems;
  const uint32_t row_bytes = (uint32_t)p.row_elems * 2;
  const uint32_t q_bytes = (uint32_t)(p.Hq * p.D) * 2, kv_bytes = (uint32_t)(p.Hkv * p.D) * 2;

  if (tid == 0) {
    for (int s = 0; s < K; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&done[s]), kRopeRotWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  auto first_token = [&](int i) { return ((int)blockIdx.x + i * (int)gridDim.x) * p.tile_tokens; };
  auto tile_len = [&](int t0) { return min(p.tile_tokens, p.T - t0); };

  if (warp == kRopeRotWarps) {
    // ---------------- mover warp ----------------
    auto issue_load = [&](int i, int s) {
      const int t0 = first_token(i), nt = tile_len(t0);
      const uint32_t bar = smem_u32(&full[s]);
      const uint32_t dst0 = smem_u32(data + s * stage_elems);
      if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)nt * row_bytes);
      __syncwarp();
      if (p.fused) {
        if (lane == 0)
          bulk_load(dst0, p.q + (int64_t)t0 * p.q_stride, (uint32_t)nt * row_bytes, bar);
      } else if (lane < nt) {
        const int64_t t = t0 + lane;
        const uint32_t dst = dst0 + (uint32_t)lane * row_bytes;
        bulk_load(dst, p.q + t * p.q_stride, q_bytes, bar);
        bulk_load(dst + q_bytes, p.k + t * p.k_stride, kv_bytes, bar);
        bulk_load(dst + q_bytes + kv_bytes, p.v + t * p.v_stride, kv_bytes, bar);
      }
    };
    for (int s = 0; s < K && s < n_local; ++s) issue_load(s, s);
    for (int i = 0; i < n_local; ++i) {
      const int s = i % K;
      // refill the stage of tile i - lag once its stores have read it (the
      // stores of the lag - 1 tiles after it may still be reading)
      if (i >= lag && i - lag + K < n_local) {
        if (lag == 1) bulk_wait_read<0>();
        else bulk_wait_read<1>();
        __syncwarp();
        issue_load(i - lag + K, (i - lag) % K);
      }
      const int t0 = first_token(i), nt = tile_len(t0);
      const int64_t t = t0 + lane;
      int pos = 0;
      int64_t slot = -1;
      if (lane < nt) {  // in flight while the stage is being rotated
        pos = __ldg(p.positions + t);
        slot = __ldg(p.slots + t);
      }
      const bool ok = mbar_wait_sleep(smem_u32(&done[s]), (uint32_t)(i / K) & 1u);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) record_error(p.err, kErrWaitTimeout, t0);
        break;
      }
      if (lane < nt) {
        const uint32_t src = smem_u32(data + s * stage_elems + (int64_t)lane * p.row_elems);
        if (pos < 0 || pos >= p.max_position) {
          record_error(p.err, kErrPosition, (int)t);
        } else {
          bulk_store(p.q_out + t * p.qo_stride, src, q_bytes);
          if (slot >= p.num_slots) {
            record_error(p.err, kErrSlot, (int)t);
          } else if (slot >= 0) {
            bulk_store(p.k_cache + slot * p.Hkv * p.D, src + q_bytes, kv_bytes);
            bulk_store(p.v_cache + slot * p.Hkv * p.D, src + q_bytes + kv_bytes, kv_bytes);
          }
        }
      }
      bulk_commit();
    }
    bulk_wait<0>();
    return;
  }

  // ---------------- rotating warps ----------------
  const int rot_items = p.rot_dim >> 4, half = p.rot_dim >> 1;
  const int per_token = (p.Hq + p.Hkv) * rot_items;
  for (int i = 0; i < n_local; ++i) {
    const int s = i % K;
    const int t0 = first_token(i), nt = tile_len(t0);
    const bool ok = mbar_wait_sleep(smem_u32(&full[s]), (uint32_t)(i / K) & 1u);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) record_error(p.err, kErrWaitTimeout, t0);
      break;
    }
    uint16_t* st = data + s * stage_elems;
    // item it = (token j, rem); j and rem advance without dividing, and the
    // token's position and table row are looked up once per token
    int j = fast_div(tid, p.div_tok_mul, p.div_tok_shift);
    int rem = tid - j * per_token;
    int cur_j = -1;
    bool valid = false;
    const float* cs_row = p.cos_sin;
    for (int it = tid; it < nt * per_token; it += kRopeRotThreads) {
      if (j != cur_j) {
        cur_j = j;
        const int pos = __ldg(p.positions + t0 + j);
        valid = pos >= 0 && pos < p.max_position;
        cs_row = p.cos_sin + (int64_t)(valid ? pos : 0) * p.rot_dim;
      }
      if (valid) {
        const int r = fast_div(rem, p.div_rot_mul, p.div_rot_shift);
        rotate_item<F, kNeox>(st + (int64_t)j * p.row_elems + r * p.D, cs_row, half,
                              rem - r * rot_items);
      }
      rem += kRopeRotThreads;
      while (rem >= per_token) {
        rem -= per_token;
        ++j;
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&done[s]));
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A set of equally spaced byte ranges: rows [base + i*stride, + len), i < n.
struct Rows {
  int64_t base, stride, len, n;
};

// Whether two row sets share a byte. Exact for a single range against
// anything and for two sets with the same stride (the views of one fused
// projection buffer); otherwise conservative (whole extents).
bool overlaps(Rows a, Rows b) {
  if (a.len <= 0 || b.len <= 0 || a.n <= 0 || b.n <= 0) return false;
  if (a.n == 1 && b.n > 1) std::swap(a, b);
  auto fdiv = [](int64_t x, int64_t y) { return x / y - ((x % y != 0) && ((x < 0) != (y < 0))); };
  if (b.n == 1) {
    if (a.n == 1 || a.stride <= 0) {
      const int64_t a1 = a.base + (a.n - 1) * a.stride + a.len;
      return a.base < b.base + b.len && b.base < a1;
    }
    // rows i with a.base + i*stride in (b.base - a.len, b.base + b.len)
    const int64_t lo = fdiv(b.base - a.len - a.base, a.stride) + 1;
    const int64_t hi = -fdiv(-(b.base + b.len - a.base), a.stride) - 1;
    return std::max<int64_t>(lo, 0) <= std::min<int64_t>(hi, a.n - 1);
  }
  if (a.stride == b.stride && a.stride > 0) {
    // rows i of a and k of b meet iff d - a.len < (i - k) * stride < d + b.len
    const int64_t d = b.base - a.base, S = a.stride;
    const int64_t lo = fdiv(d - a.len, S) + 1;
    const int64_t hi = -fdiv(-(d + b.len), S) - 1;
    return std::max<int64_t>(lo, -(b.n - 1)) <= std::min<int64_t>(hi, a.n - 1);
  }
  const int64_t a1 = a.base + (a.n - 1) * a.stride + a.len;
  const int64_t b1 = b.base + (b.n - 1) * b.stride + b.len;
  return a.base < b1 && b.base < a1;
}

int fail(int code, const std::string& msg) { return set_last_error(code, msg.c_str()); }

// Division by a fixed d >= 1 as one wide multiply and a shift, exact for
// every x < 2^31 (Granlund and Montgomery, "Division by invariant integers
// using multiplication", 1994): with l = ceil(log2 d), mul = ceil(2^(31+l) / d)
// fits in 32 bits and x / d = (x * mul) >> (31 + l).
void magic_div(uint32_t d, uint32_t* mul, uint32_t* shift) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  *mul = (uint32_t)(((1ull << (31 + l)) + d - 1) / d);
  *shift = 31 + l;
}

struct DeviceInfo {
  int num_sms = 0;
  bool prepared = false;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[64];

template <typename F, bool kNeox>
cudaError_t prepare_one(int smem_max) {
  return cudaFuncSetAttribute(rope_kv_write_kernel<F, kNeox>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
}

// SM count of `device`, and the kernels' shared-memory limit set once.
cudaError_t device_info(int device, int* num_sms) {
  if (device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[device];
  if (!d.prepared) {
    cudaError_t e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, device);
    const int smem_max = kRopeDataOff + kRopeRingBytes;
    if (e == cudaSuccess) e = prepare_one<Bf16, true>(smem_max);
    if (e == cudaSuccess) e = prepare_one<Bf16, false>(smem_max);
    if (e == cudaSuccess) e = prepare_one<Fp16, true>(smem_max);
    if (e == cudaSuccess) e = prepare_one<Fp16, false>(smem_max);
    if (e != cudaSuccess) return e;
    d.prepared = true;
  }
  *num_sms = d.num_sms;
  return cudaSuccess;
}

}  // namespace
}  // namespace pda

extern "C" int paged_decode_attn_rope_kv_write(
    const void* q, int64_t q_token_stride, const void* k, int64_t k_token_stride, const void* v,
    int64_t v_token_stride, const int32_t* positions, const int64_t* slot_mapping,
    const float* cos_sin_cache, int max_position, int rot_dim, int neox_style, int num_tokens,
    int num_q_heads, int num_kv_heads, int head_dim, int dtype, void* q_out,
    int64_t q_out_token_stride, void* k_cache, void* v_cache, int64_t num_slots, int* err,
    int device, void* stream) {
  using pda::fail;
  using pda::Rows;
  if (num_tokens < 0) return fail(PDA_EINVAL, "num_tokens < 0");
  if (num_q_heads < 1 || num_kv_heads < 1) return fail(PDA_EINVAL, "head counts must be >= 1");
  if (head_dim < 16 || head_dim > 1024 || head_dim % 16 != 0)
    return fail(PDA_EINVAL, "head_dim must be a multiple of 16 in [16, 1024]");
  if (rot_dim < 0 || rot_dim > head_dim || rot_dim % 16 != 0)
    return fail(PDA_EINVAL, "rot_dim must be a multiple of 16 in [0, head_dim]");
  if (dtype != PDA_BF16 && dtype != PDA_FP16) return fail(PDA_EINVAL, "dtype must be bf16 or fp16");
  if (num_slots < 0) return fail(PDA_EINVAL, "num_slots < 0");
  if (max_position < 0) return fail(PDA_EINVAL, "max_position < 0");
  if (device < 0) return fail(PDA_EINVAL, "device must be >= 0");
  const int64_t hq_d = (int64_t)num_q_heads * head_dim, hkv_d = (int64_t)num_kv_heads * head_dim;
  const int64_t row_elems = hq_d + 2 * hkv_d;
  if (row_elems * 2 > pda::kRopeMaxRowBytes)
    return fail(PDA_EUNSUPPORTED, "(num_q_heads + 2 num_kv_heads) * head_dim * 2 exceeds 48 KiB");
  if (q_token_stride == 0) q_token_stride = hq_d;
  if (k_token_stride == 0) k_token_stride = hkv_d;
  if (v_token_stride == 0) v_token_stride = hkv_d;
  if (q_out_token_stride == 0) q_out_token_stride = hq_d;
  if (q_token_stride < hq_d || q_out_token_stride < hq_d || k_token_stride < hkv_d ||
      v_token_stride < hkv_d)
    return fail(PDA_EINVAL, "a token stride is smaller than its row of heads");
  if ((q_token_stride | k_token_stride | v_token_stride | q_out_token_stride) % 8 != 0)
    return fail(PDA_EINVAL, "token strides must be multiples of 8 elements (16 bytes)");
  if (num_tokens == 0) return PDA_OK;
  if (!q || !k || !v || !positions || !slot_mapping || !q_out || !k_cache || !v_cache ||
      (rot_dim > 0 && !cos_sin_cache))
    return fail(PDA_EINVAL, "a required pointer is NULL");
  if (!pda::aligned16(q) || !pda::aligned16(k) || !pda::aligned16(v) || !pda::aligned16(q_out) ||
      !pda::aligned16(k_cache) || !pda::aligned16(v_cache) ||
      (cos_sin_cache && !pda::aligned16(cos_sin_cache)) || (err && (uintptr_t)err % 4))
    return fail(PDA_EINVAL, "tensors must be 16-byte aligned");
  // aliasing: outputs against inputs and each other, row sets in bytes
  const int64_t T = num_tokens;
  auto rows = [T](const void* p, int64_t stride, int64_t len) {
    return Rows{(int64_t)reinterpret_cast<uintptr_t>(p), stride * 2, len * 2, T};
  };
  auto span = [](const void* p, int64_t bytes) {
    return Rows{(int64_t)reinterpret_cast<uintptr_t>(p), bytes, bytes, 1};
  };
  const Rows rq = rows(q, q_token_stride, hq_d), rk = rows(k, k_token_stride, hkv_d);
  const Rows rv = rows(v, v_token_stride, hkv_d), rqo = rows(q_out, q_out_token_stride, hq_d);
  const Rows rkc = span(k_cache, num_slots * hkv_d * 2), rvc = span(v_cache, num_slots * hkv_d * 2);
  const Rows rpos = span(positions, T * 4), rslot = span(slot_mapping, T * 8);
  const Rows rcs = span(cos_sin_cache, cos_sin_cache ? (int64_t)max_position * rot_dim * 4 : 0);
  const Rows rerr = span(err, err ? 8 : 0);
  const bool q_in_place = (q == q_out && q_token_stride == q_out_token_stride);
  if (!q_in_place && pda::overlaps(rqo, rq))
    return fail(PDA_EALIAS, "q_out overlaps q (only the exact in-place form is allowed)");
  const Rows ins[6] = {rk, rv, rpos, rslot, rcs, rerr};
  const Rows outs[3] = {rqo, rkc, rvc};
  for (int o = 0; o < 3; ++o) {
    for (const Rows& in : ins)
      if (pda::overlaps(outs[o], in)) return fail(PDA_EALIAS, "an output overlaps an input");
    for (int j = o + 1; j < 3; ++j)
      if (pda::overlaps(outs[o], outs[j]))
        return fail(PDA_EALIAS, "q_out, k_cache and v_cache must not overlap");
    if (o > 0 && pda::overlaps(outs[o], rq)) return fail(PDA_EALIAS, "a cache overlaps q");
  }
  int prev = -1;
  cudaError_t e = cudaGetDevice(&prev);
  if (e == cudaSuccess && prev != device) e = cudaSetDevice(device);
  if (e != cudaSuccess)
    return fail(PDA_ECUDA, std::string("cudaSetDevice: ") + cudaGetErrorString(e));
  int num_sms = 0;
  e = pda::device_info(device, &num_sms);
  if (e != cudaSuccess) {
    if (prev >= 0 && prev != device) cudaSetDevice(prev);
    return fail(PDA_ECUDA, std::string("rope_kv_write set-up: ") + cudaGetErrorString(e));
  }
  // Tiles: up to ~16 KB of token rows (<= 32 tokens); fewer tokens per tile
  // when that still gives every SM two tiles, so short calls spread out.
  const int64_t row_bytes = row_elems * 2;
  int n_max = (int)std::min<int64_t>(pda::kRopeMaxTileTokens,
                                     std::max<int64_t>(1, pda::kRopeStageTarget / row_bytes));
  int n = (int)std::min<int64_t>(n_max, std::max<int64_t>(1, (T + 2 * num_sms - 1) / (2 * num_sms)));
  const int64_t num_tiles = (T + n - 1) / n;
  const uint32_t per_token_items =
      std::max<uint32_t>(1, (uint32_t)(num_q_heads + num_kv_heads) * (uint32_t)(rot_dim / 16));
  const int stage_bytes = n * (int)row_bytes;
  const int stages = std::min(pda::kRopeMaxStages, pda::kRopeRingBytes / stage_bytes);
  const int lag = stages >= 5 ? 2 : 1;
  const int smem = pda::kRopeDataOff + stages * stage_bytes;
  const int per_sm = std::max(1, std::min(3, 233472 / (smem + 1024)));  // 3 by registers
  const int64_t grid = std::min<int64_t>(num_tiles, (int64_t)num_sms * per_sm);
  pda::RopeParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.q_stride = q_token_stride;
  p.k_stride = k_token_stride;
  p.v_stride = v_token_stride;
  p.qo_stride = q_out_token_stride;
  p.positions = positions;
  p.slots = slot_mapping;
  p.cos_sin = cos_sin_cache;
  p.q_out = static_cast<uint16_t*>(q_out);
  p.k_cache = static_cast<uint16_t*>(k_cache);
  p.v_cache = static_cast<uint16_t*>(v_cache);
  p.err = err;
  p.num_slots = num_slots;
  p.T = num_tokens;
  p.Hq = num_q_heads;
  p.Hkv = num_kv_heads;
  p.D = head_dim;
  p.rot_dim = rot_dim;
  p.max_position = max_position;
  p.row_elems = (int)row_elems;
  p.tile_tokens = n;
  p.num_tiles = (int)num_tiles;
  pda::magic_div(per_token_items, &p.div_tok_mul, &p.div_tok_shift);
  pda::magic_div(rot_dim >= 16 ? rot_dim / 16 : 1, &p.div_rot_mul, &p.div_rot_shift);
  p.stages = stages;
  p.lag = lag;
  p.fused = (k == p.q + hq_d && v == p.q + hq_d + hkv_d && q_token_stride == row_elems &&
             k_token_stride == row_elems && v_token_stride == row_elems);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool neox = neox_style != 0;
  const dim3 g((unsigned)grid), b(pda::kRopeThreads);
  if (dtype == PDA_BF16) {
    if (neox) pda::rope_kv_write_kernel<pda::Bf16, true><<<g, b, smem, s>>>(p);
    else pda::rope_kv_write_kernel<pda::Bf16, false><<<g, b, smem, s>>>(p);
  } else {
    if (neox) pda::rope_kv_write_kernel<pda::Fp16, true><<<g, b, smem, s>>>(p);
    else pda::rope_kv_write_kernel<pda::Fp16, false><<<g, b, smem, s>>>(p);
  }
  e = cudaGetLastError();
  if (prev >= 0 && prev != device) cudaSetDevice(prev);
  if (e != cudaSuccess)
    return fail(PDA_ECUDA, std::string("rope_kv_write launch: ") + cudaGetErrorString(e));
  return PDA_OK;
}
