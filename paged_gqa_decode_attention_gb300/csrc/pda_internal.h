// Private launch boundary between the C ABI (api.cpp) and the CUDA kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace pda {

constexpr int kHeadDim = 128;  // the tensor-core kernel's head dim
constexpr int kMaxSplits = 64;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

// Device error word layout: err[0] = code (0 = none), err[1] = detail.
enum DeviceError : int {
  kErrNone = 0,
  kErrContextLen = 1,
  kErrBlockId = 2,
  kErrWaitTimeout = 3,
  kErrPosition = 4,  // RoPE + KV write: position outside the cos/sin table
  kErrSlot = 5,      // RoPE + KV write: slot beyond the cache
};

struct PartialParams {
  const void* q;               // [B, Hq, D]
  const int32_t* block_table;  // [B, max_blocks]
  const int32_t* context_lens; // [B]
  void* out;                   // [B, Hq, D]
  float* ws_o;                 // [B, Hq, num_splits, D]
  float* ws_lse;               // [B, Hq, num_splits]
  int* err;                    // device error word
  int* counters;               // [B, Hkv] split tickets for the fused merge; zero between calls
  int* sched;                  // [2] work counter and done counter of the persistent kernel;
                               // zero between calls
  int Hq;
  int Hkv;
  int max_blocks;
  int chunk_pages;  // pages per split
  int num_splits;   // S (grid.x); row stride of the workspace
  float qscale;     // scale * log2(e): logits are kept in base-2 units
  int num_units;    // S * Hkv * B work units (persistent tensor-core kernel)
  int max_ctas;     // resident CTAs the persistent kernel launches at most
  int out_f32;      // out is fp32 (else the input dtype)
  const float* k_scale;  // K/V dequantisation scales: [Hkv] (scale_per_head) or [1];
  const float* v_scale;  // NULL = 1
  int scale_per_head;
  // Fault injection for the timeout tests (tensor-core kernel): stall_units
  // makes the unit-fetching warp publish no unit, so every other role's
  // first wait runs out with nothing issued or in flight; wait_ns (0 = the
  // default kWaitLimitNs) shortens every pipeline wait.
  int stall_units = 0;
  unsigned long long wait_ns = 0;
  // Tensor-core kernel: > 1 when the launch is made of thread-block clusters
  // of this many CTAs, one per split of a (sequence, kv head), every CTA one
  // unit; the splits then merge through distributed shared memory instead
  // of the workspace and the split tickets.
  int cluster = 0;
};

struct MergeParams {
  const float* o;               // [rows, num_splits, head_dim]
  const float* lse;             // [rows, num_splits], natural log
  const int32_t* context_lens;  // decode path: per-sequence split counts; null = all splits
  void* out;                    // [rows, head_dim]
  int rows;
  int num_splits;
  int head_dim;
  int Hq;           // decode path: rows = b * Hq + hq
  int block_size;   // decode path
  int max_blocks;   // decode path
  int chunk_pages;  // decode path
};

// The two implementations of the split-K partial kernel.
enum PartialKernel : int {
  kPartialCudaCore = 0,    // QK/PV on the FMA pipe (partial_kernel.cuh): G 1..8 at D 64 and
                           // 128, G 1..4 at D 256
  kPartialTensorCore = 1,  // QK/PV with tcgen05 MMAs into TMEM (partial_tc_kernel.cuh):
                           // G 3..16, D 64 and 128 (FP8 K/V: G 1..16)
};

// The kernel a geometry uses unless overridden (PDA_PARTIAL_KERNEL): the
// faster one as measured on GB300. With G = 4 or 8 query heads per kv head
// the packed tile is a real contraction and the tensor-core kernel wins (B=4,
// L=32768 at G=4: 0.0974 vs 0.1000 ms; the 128-sequence serving mix at G=8:
// 0.114 vs 0.255 ms); otherwise the CUDA-core kernel is used.
constexpr int default_partial_kernel(int group, int head_dim, bool kv_fp8 = false) {
  return (kv_fp8 || (group >= 3 && group <= 16 && (head_dim == 64 || head_dim == 128)))
             ? kPartialTensorCore
             : kPartialCudaCore;
}

// CTAs per SM each kernel is built for (its launch bounds and shared memory);
// the planner's figure when no GPU is queried.
constexpr int partial_ctas_per_sm_hint(int kernel, int group, int head_dim) {
  return kernel == kPartialTensorCore ? 1
                                      : ((group * head_dim > 512 || head_dim >= 256) ? 1 : 2);
}

// Work slots per wave the split planner counts on. Measured on GB300
// (split-count sweeps of the B=4 L=32768, B=1 L=32768 and B=1 / B=4 L=8192
// steps): a few long streams per SM do best when one wave covers the whole
// step, and the tensor-core kernel with 16-bit K/V saturates HBM with about
// 27/32 of the SMs (128 of 152). So it plans for 128 units of one wave (B=4
// L=32768: 0.932-0.945 of peak, against 0.912-0.925 with two units on each
// of 152 CTAs). The launch still uses every SM, so steps of many short units
// balance over all of them. FP8 K/V is limited per SM and plans for every
// SM, as does the CUDA-core kernel. PDA_PLAN_SLOTS overrides (experiments).
int planning_slots(int kernel, bool kv_fp8, int num_sms, int ctas_per_sm);

// kv_fp8: K/V caches hold FP8 E4M3 (tensor-core kernel, D 64 or 128, bf16 or fp16 q).
bool partial_supported(int group, int head_dim, int block_size, int dtype, bool kv_fp8);
bool partial_kernel_supported(int kernel, int group, int head_dim, bool kv_fp8);
cudaError_t partial_prepare(int kernel, int group, int head_dim, int block_size, int dtype,
                            bool kv_fp8);
int partial_ctas_per_sm(int kernel, int group, int head_dim, int block_size, int dtype,
                        bool kv_fp8);
// How many clusters of `cluster` CTAs of the tensor-core kernel can be
// resident at once (0 if none, or if that cluster size is not allowed).
int partial_max_clusters(int group, int head_dim, int block_size, int dtype, bool kv_fp8,
                         int cluster);

// tmap_q (a [B * Hq, D] view of q, boxes of 64 dims x G rows) is read by
// the tensor-core kernel only; both kernels take the output type from
// p.out_f32.
cudaError_t launch_partial(int kernel, int group, int head_dim, int block_size, int dtype,
                           bool kv_fp8, const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                           const CUtensorMap* tmap_q, const PartialParams& p, int batch,
                           cudaStream_t stream);

// out_dtype: 0 bf16, 1 fp16, 2 f32
cudaError_t launch_merge(const MergeParams& p, int out_dtype, cudaStream_t stream);

cudaError_t launch_validate(const int32_t* block_table, const int32_t* context_lens, int batch,
                            int max_blocks, int block_size, int64_t num_blocks, int* err,
                            cudaStream_t stream);

// Whether kernels are launched with programmatic dependent launch (default
// on; the environment variable PDA_PDL=0 turns it off, read once).
bool pdl_enabled();

// Records `msg` as this thread's last error (paged_decode_attn_last_error)
// and returns `code`.
int set_last_error(int code, const char* msg);

}  // namespace pda
