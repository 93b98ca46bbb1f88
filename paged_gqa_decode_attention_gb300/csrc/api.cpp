// C ABI of the paged decode-attention library: argument checks, the split
// planner, the per-handle workspace and TMA descriptor cache, and the launch
// of the partial kernel (which also merges the splits). Nothing here throws
// across the ABI.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdlib>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "paged_decode_attn.h"
#include "pda_internal.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int cuda_fail(const char* what, cudaError_t e) {
  return fail(PDA_ECUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" +
                             cudaGetErrorString(e) + ")");
}

// Planner cost constants, in token-equivalents of one CTA's streaming time:
// the fixed cost of a work unit (q and first-page latency, the unit's state
// hand-off, partial write and merge ticket) and of merging split partials.
// Chosen from split-count sweeps on GB300 (B=1 and B=4 at L=8192 and
// L=32768, FP8 B=8 L=32768, the 128-sequence serving mix, 28/4-head B=16
// L=8192): a unit of the persistent tensor-core kernel costs about 512
// tokens, a CTA of the CUDA-core kernel about 256; with these (and the
// planning slots below) the planner's pick is the fastest measured split
// count or within 2% of it on every one of those cases.
constexpr int kOverheadTokensCudaCore = 256;
constexpr int kOverheadTokensTensorCore = 512;
constexpr int kMergeTokens = 96;

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Shape checks shared by create and plan; returns PDA_OK or an error.
int check_config(const pda_config* c) {
  if (!c) return fail(PDA_EINVAL, "config is NULL");
  if (c->num_q_heads <= 0 || c->num_kv_heads <= 0)
    return fail(PDA_EINVAL, "num_q_heads and num_kv_heads must be positive");
  if (c->num_q_heads % c->num_kv_heads != 0)
    return fail(PDA_EINVAL, "num_q_heads must be a multiple of num_kv_heads");
  if (c->num_kv_heads > 65535) return fail(PDA_EINVAL, "num_kv_heads > 65535");
  const int G = c->num_q_heads / c->num_kv_heads;
  if (c->head_dim <= 0 || c->block_size <= 0)
    return fail(PDA_EINVAL, "head_dim and block_size must be positive");
  if (c->dtype != PDA_BF16 && c->dtype != PDA_FP16)
    return fail(PDA_EINVAL, "dtype must be PDA_BF16 or PDA_FP16");
  if (c->max_batch < 1 || c->max_batch > 65535)
    return fail(PDA_EINVAL, "max_batch must be in [1, 65535]");
  if (c->max_blocks_per_seq < 1) return fail(PDA_EINVAL, "max_blocks_per_seq must be >= 1");
  if ((int64_t)c->max_blocks_per_seq * c->block_size > INT_MAX)
    return fail(PDA_EINVAL, "max_blocks_per_seq * block_size overflows int32");
  if (c->max_splits < 1 || c->max_splits > pda::kMaxSplits)
    return fail(PDA_EINVAL, "max_splits must be in [1, 64]");
  if (c->device < 0) return fail(PDA_EINVAL, "device must be >= 0");
  if (c->kv_fp8 != 0 && c->kv_fp8 != 1) return fail(PDA_EINVAL, "kv_fp8 must be 0 or 1");
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256)
    return fail(PDA_EUNSUPPORTED, "head_dim must be 64, 128 or 256");
  if (c->kv_fp8 && !pda::partial_supported(G, c->head_dim, c->block_size, c->dtype, true))
    return fail(PDA_EUNSUPPORTED,
                "FP8 K/V caches need head_dim 64 or 128, group size 1..16, dtype PDA_BF16 "
                "or PDA_FP16 and block_size 16 or 32 (or 64 at group size <= 8)");
  if (!pda::partial_supported(G, c->head_dim, c->block_size, c->dtype, c->kv_fp8 != 0))
    return fail(PDA_EUNSUPPORTED,
                "unsupported geometry: group size must be 1..16 (1..4 at head_dim 256) and "
                "block_size 16 or 32 (or 64 at group size <= 8)");
  return PDA_OK;
}

// A small call runs on the CUDA-core kernel even where the tensor-core kernel
// is the default (16-bit K/V, a geometry both support): with few short units
// the step is mostly fixed cost, and the CUDA-core kernel's (no TMEM, no
// persistent scheduling, 160-thread CTAs, two per SM) is the smaller.
// Measured on GB300 at 32/8 heads, back to back / cold, CUDA-core against
// tensor-core: 32 sequences of 16-64 tokens 4.6 / 10.2 us against 9.5 / 16.7;
// 32 x 256 tokens (34 MB) 9.3 / 16.4 against 10.3 / 20.5; 8 x 512 (17 MB)
// 8.8 / 14.8 against 9.8 / 21.1; 2 x 1024 8.2 / 14.3 against 9.6 / 18.4. The
// tensor cores win back to back from 34 MB at 1024-2048 tokens (8 x 1024:
// 11.8 against 11.2) and at 67 MB of 256-token contexts (64 x 256: 18.0
// against 16.6). So: contexts up to 256 tokens and 48 MiB of K/V, or up to
// 1024 tokens and 20 MiB (the call's bytes bounded from its table width).
constexpr int kShortContextTokens = 256;
constexpr int64_t kShortStepKvBytes = int64_t(48) << 20;
constexpr int kMidContextTokens = 1024;
constexpr int64_t kMidStepKvBytes = int64_t(20) << 20;

// The kernel one call runs: the default for the geometry, or the CUDA-core
// kernel for a small call (max_len: the call's longest context, its table
// width times the block size or the hint when smaller; batch x Hkv x max_len
// x D x 4 bytes bounds its 16-bit K/V bytes).
constexpr int call_partial_kernel(int group, int head_dim, bool kv_fp8, int64_t max_len,
                                  int64_t batch, int num_kv_heads) {
  const int64_t bytes = batch * num_kv_heads * max_len * head_dim * 4;
  return (pda::default_partial_kernel(group, head_dim, kv_fp8) == pda::kPartialTensorCore &&
          !kv_fp8 && group <= 8 && (head_dim == 64 || head_dim == 128) &&
          ((max_len <= kShortContextTokens && bytes <= kShortStepKvBytes) ||
           (max_len <= kMidContextTokens && bytes <= kMidStepKvBytes)))
             ? pda::kPartialCudaCore
             : pda::default_partial_kernel(group, head_dim, kv_fp8);
}

void plan_splits(const pda_config& c, int kernel, int num_sms, int ctas_per_sm, int batch,
                 int max_blocks, int hint, int forced, int* S_out, int* chunk_out) {
  const int overhead = kernel == pda::kPartialTensorCore ? kOverheadTokensTensorCore
                                                         : kOverheadTokensCudaCore;
  const int bs = c.block_size;
  int64_t max_len = (int64_t)max_blocks * bs;
  if (hint > 0 && hint < max_len) max_len = hint;
  const int max_pages = max_len > 0 ? ceil_div(max_len, bs) : 1;
  const int cap = c.max_splits < max_pages ? c.max_splits : max_pages;
  int S = 1;
  if (forced > 0) {
    S = forced < cap ? forced : cap;
  } else {
    const int64_t base = (int64_t)(batch > 0 ? batch : 1) * c.num_kv_heads;
    const int64_t slots = pda::planning_slots(kernel, c.kv_fp8 != 0, num_sms, ctas_per_sm);
    double best = INFINITY;
    for (int s = 1; s <= cap; ++s) {
      const int chunk = ceil_div(max_pages, s);
      const int s_eff = ceil_div(max_pages, chunk);
      if (s_eff != s) continue;  // identical to a smaller split count
      const int64_t waves = (base * s_eff + slots - 1) / slots;
      const double cost = (double)waves * ((double)chunk * bs + overhead) +
                          (s_eff > 1 ? kMergeTokens : 0);
      if (cost < best * (1.0 - 1e-9)) {
        best = cost;
        S = s_eff;
      }
    }
  }
  const int chunk = ceil_div(max_pages, S);
  *S_out = ceil_div(max_pages, chunk);
  *chunk_out = chunk;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A [num_blocks * block_size, Hkv * D] view of a cache, loaded as boxes of
// 128 bytes (64 16-bit dims or 128 fp8 dims) x block_size rows with 128-byte
// swizzle; FP8 at head dim 64: 64-byte boxes with 64-byte swizzle.
int encode_cache_map(CUtensorMap* m, const void* base, int Hkv, int D, int bs,
                     int64_t num_blocks, bool fp8 = false) {
  auto fn = tensor_map_encoder();
  if (!fn) return fail(PDA_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const int esz = fp8 ? 1 : 2;
  const int box_bytes = (fp8 && D == 64) ? 64 : 128;
  cuuint64_t dims[2] = {(cuuint64_t)Hkv * D, (cuuint64_t)num_blocks * bs};
  cuuint64_t strides[1] = {(cuuint64_t)Hkv * D * esz};
  cuuint32_t box[2] = {(cuuint32_t)(box_bytes / esz), (cuuint32_t)bs};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(PDA_ECUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(r));
  return PDA_OK;
}

// A [B * Hq, D] view of q, loaded as boxes of 64 dims x G rows (the G
// query heads of one kv head) with 128-byte swizzle.
int encode_q_map(CUtensorMap* m, const void* q, int64_t rows, int D, int group) {
  auto fn = tensor_map_encoder();
  if (!fn) return fail(PDA_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)group};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(q), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(PDA_ECUDA, "cuTensorMapEncodeTiled (q) failed with CUresult " + std::to_string(r));
  return PDA_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return na && nb && a0 < b0 + nb && b0 < a0 + na;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Makes `dev` current for the scope and restores the caller's device.
struct DeviceGuard {
  int prev = -1;
  cudaError_t err = cudaSuccess;
  explicit DeviceGuard(int dev) {
    err = cudaGetDevice(&prev);
    if (err == cudaSuccess && prev != dev) err = cudaSetDevice(dev);
    else if (err == cudaSuccess) prev = -1;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

}  // namespace

int pda::set_last_error(int code, const char* msg) { return fail(code, msg); }

int pda::planning_slots(int kernel, bool kv_fp8, int num_sms, int ctas_per_sm) {
  static const int forced = [] {
    const char* e = std::getenv("PDA_PLAN_SLOTS");
    return e ? std::atoi(e) : 0;
  }();
  const int slots = (num_sms > 0 ? num_sms : 1) * (ctas_per_sm > 0 ? ctas_per_sm : 1);
  int n = slots;
  if (kernel == kPartialTensorCore && !kv_fp8) n = (slots * 27) / 32;
  if (forced > 0) n = forced;
  return n < 1 ? 1 : (n > slots ? slots : n);
}

bool pda::pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("PDA_PDL");
    return !(e && std::strcmp(e, "0") == 0);
  }();
  return on;
}

struct pda_handle_s {
  pda_config cfg;
  int group = 1;
  int kernel = 0;  // pda::PartialKernel
  int num_sms = 1;
  int ctas_per_sm = 1;
  // Calls of short contexts run on the CUDA-core kernel where the tensor-core
  // kernel is the default (call_partial_kernel); off when
  // PDA_PARTIAL_KERNEL pins the kernel.
  bool small_cc = false;
  int cc_ctas_per_sm = 1;
  void* ws = nullptr;
  float* ws_o = nullptr;
  float* ws_lse = nullptr;
  int* err = nullptr;
  int* counters = nullptr;  // [max_batch, Hkv] split tickets
  size_t counter_bytes = 0;
  int test_stall_runs = 0;  // timeout tests: this many first runs publish no unit
  // Tensor-core kernel: clusters of c CTAs (c = 2..16) that can be resident
  // at once, so a step of groups <= max_clusters[S] (sequence, kv head) pairs
  // runs as clusters that merge their splits in distributed shared memory;
  // 0 = that cluster size is not available. PDA_CLUSTER_MERGE=0 turns the
  // cluster launch off for this handle (A/B runs, tests of the other path).
  int max_clusters[17] = {};
  // TMA descriptors for the last (k_cache, v_cache, num_blocks) seen
  const void* tm_k = nullptr;
  const void* tm_v = nullptr;
  int64_t tm_nb = -1;
  alignas(64) CUtensorMap tmap_k;
  alignas(64) CUtensorMap tmap_v;
};

namespace {

struct LaunchShape {
  int splits, chunk_pages, ctas, cluster;
  int64_t units;
  int kernel, ctas_per_sm;  // the kernel this call runs and its CTAs per SM
};

// The longest context a call can have: its table width in tokens, or the
// hint when that is smaller.
int64_t call_max_len(const pda_config& c, int max_blocks, int hint) {
  const int64_t len = (int64_t)max_blocks * c.block_size;
  return hint > 0 && hint < len ? hint : len;
}

// How a run of this handle is launched: the split plan, the work units, the
// CTAs and, for the tensor-core kernel, whether the launch is one wave of
// clusters (one per (sequence, kv head), the splits merging through
// distributed shared memory) when every pair fits.
LaunchShape launch_shape(const pda_handle_s* h, int batch, int max_blocks, int hint, int forced) {
  const pda_config& c = h->cfg;
  LaunchShape r{1, 1, 0, 0, 0, h->kernel, h->ctas_per_sm};
  if (h->small_cc &&
      call_partial_kernel(h->group, c.head_dim, false, call_max_len(c, max_blocks, hint),
                               batch, c.num_kv_heads) == pda::kPartialCudaCore) {
    r.kernel = pda::kPartialCudaCore;
    r.ctas_per_sm = h->cc_ctas_per_sm;
  }
  plan_splits(c, r.kernel, h->num_sms, r.ctas_per_sm, batch, max_blocks, hint, forced,
              &r.splits, &r.chunk_pages);
  r.units = (int64_t)r.splits * c.num_kv_heads * batch;
  if (r.kernel == pda::kPartialTensorCore) {
    const int64_t max_ctas = (int64_t)h->num_sms * r.ctas_per_sm;
    r.ctas = (int)(r.units < max_ctas ? r.units : max_ctas);
    if (r.splits >= 2 && r.splits <= 16 &&
        (int64_t)batch * c.num_kv_heads <= h->max_clusters[r.splits]) {
      r.cluster = r.splits;
      r.ctas = (int)r.units;
    }
  } else {
    r.ctas = (int)(r.units < INT_MAX ? r.units : INT_MAX);
  }
  return r;
}

}  // namespace

extern "C" {

int paged_decode_attn_abi_version(void) { return PDA_ABI_VERSION; }

const char* paged_decode_attn_last_error(void) { return g_last_error.c_str(); }

int paged_decode_attn_create(const pda_config* cfg, pda_handle* out_handle) {
  if (!out_handle) return fail(PDA_EINVAL, "out_handle is NULL");
  *out_handle = nullptr;
  int st = check_config(cfg);
  if (st != PDA_OK) return st;
  DeviceGuard guard(cfg->device);
  if (guard.err != cudaSuccess) return cuda_fail("cudaSetDevice", guard.err);
  pda_handle h = new (std::nothrow) pda_handle_s();
  if (!h) return fail(PDA_ENOMEM, "host allocation of the handle failed");
  h->cfg = *cfg;
  h->group = cfg->num_q_heads / cfg->num_kv_heads;
  cudaError_t e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, cfg->device);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail("cudaDeviceGetAttribute", e);
  }
  // The partial kernel: PDA_PARTIAL_KERNEL=tensor_core (groups of 4 or 8
  // query heads) or cuda_core overrides the default; read here, once per
  // handle (A/B measurements and tests).
  const bool kv8 = cfg->kv_fp8 != 0;
  h->kernel = pda::default_partial_kernel(h->group, cfg->head_dim, kv8);
  const char* kernel_env = std::getenv("PDA_PARTIAL_KERNEL");
  h->small_cc = !kernel_env &&
                call_partial_kernel(h->group, cfg->head_dim, kv8, 1, 1, 1) ==
                    pda::kPartialCudaCore &&
                h->kernel == pda::kPartialTensorCore;
  if (const char* env = kernel_env) {
    if (std::strcmp(env, "cuda_core") == 0 &&
        pda::partial_kernel_supported(pda::kPartialCudaCore, h->group, cfg->head_dim, kv8))
      h->kernel = pda::kPartialCudaCore;
    else if (std::strcmp(env, "tensor_core") == 0 &&
             pda::partial_kernel_supported(pda::kPartialTensorCore, h->group, cfg->head_dim, kv8))
      h->kernel = pda::kPartialTensorCore;
  }
  // Timeout tests (tensor-core kernel only): PDA_TEST_STALL_RUNS=n makes the
  // first n runs of this handle publish no work unit with a 1 ms wait limit,
  // so every pipeline wait runs out while nothing is in flight; the run
  // records error code 3 and the next run must be exact.
  if (const char* env = std::getenv("PDA_TEST_STALL_RUNS"))
    if (h->kernel == pda::kPartialTensorCore) h->test_stall_runs = std::atoi(env);
  e = pda::partial_prepare(h->kernel, h->group, cfg->head_dim, cfg->block_size, cfg->dtype, kv8);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail("cudaFuncSetAttribute", e);
  }
  const char* cl_env = std::getenv("PDA_CLUSTER_MERGE");
  if (h->kernel == pda::kPartialTensorCore && !(cl_env && std::strcmp(cl_env, "0") == 0))
    for (int c = 2; c <= 16 && c <= cfg->max_splits; ++c)
      h->max_clusters[c] = pda::partial_max_clusters(h->group, cfg->head_dim, cfg->block_size,
                                                     cfg->dtype, kv8, c);
  // Plan with the residency the kernel is built for, so paged_decode_attn_plan
  // (no GPU) and run agree; fall back to the measured figure if it is lower.
  const int occ =
      pda::partial_ctas_per_sm(h->kernel, h->group, cfg->head_dim, cfg->block_size, cfg->dtype,
                               kv8);
  const int hint = pda::partial_ctas_per_sm_hint(h->kernel, h->group, cfg->head_dim);
  h->ctas_per_sm = occ < hint ? occ : hint;
  if (h->small_cc) {
    e = pda::partial_prepare(pda::kPartialCudaCore, h->group, cfg->head_dim, cfg->block_size,
                             cfg->dtype, false);
    if (e != cudaSuccess) {
      delete h;
      return cuda_fail("cudaFuncSetAttribute", e);
    }
    const int occ_cc = pda::partial_ctas_per_sm(pda::kPartialCudaCore, h->group, cfg->head_dim,
                                                cfg->block_size, cfg->dtype, false);
    const int hint_cc =
        pda::partial_ctas_per_sm_hint(pda::kPartialCudaCore, h->group, cfg->head_dim);
    h->cc_ctas_per_sm = occ_cc < hint_cc ? occ_cc : hint_cc;
  }
  const size_t rows = (size_t)cfg->max_batch * cfg->num_q_heads * cfg->max_splits;
  const size_t o_bytes = rows * cfg->head_dim * sizeof(float);
  const size_t lse_bytes = ((rows * sizeof(float)) + 255) & ~size_t(255);
  const size_t err_bytes = 256;
  // split tickets [max_batch, Hkv], then the persistent kernel's 2 counters
  h->counter_bytes = ((size_t)cfg->max_batch * cfg->num_kv_heads + 2) * sizeof(int);
  e = cudaMalloc(&h->ws, o_bytes + lse_bytes + err_bytes + h->counter_bytes);
  if (e != cudaSuccess) {
    delete h;
    cudaGetLastError();
    return fail(PDA_ENOMEM, std::string("workspace cudaMalloc failed: ") + cudaGetErrorString(e));
  }
  h->ws_o = static_cast<float*>(h->ws);
  h->ws_lse = reinterpret_cast<float*>(static_cast<char*>(h->ws) + o_bytes);
  h->err = reinterpret_cast<int*>(static_cast<char*>(h->ws) + o_bytes + lse_bytes);
  h->counters = reinterpret_cast<int*>(static_cast<char*>(h->ws) + o_bytes + lse_bytes + err_bytes);
  e = cudaMemset(h->err, 0, err_bytes + h->counter_bytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(h->ws);
    delete h;
    return cuda_fail("cudaMemset", e);
  }
  *out_handle = h;
  return PDA_OK;
}

void paged_decode_attn_destroy(pda_handle h) {
  if (!h) return;
  if (h->ws) {
    DeviceGuard guard(h->cfg.device);
    cudaFree(h->ws);
  }
  delete h;
}

int paged_decode_attn_plan(const pda_config* cfg, int num_sms, int batch, int max_blocks,
                           int max_context_len_hint, int* num_splits, int* chunk_pages) {
  int st = check_config(cfg);
  if (st != PDA_OK) return st;
  if (!num_splits || !chunk_pages) return fail(PDA_EINVAL, "output pointer is NULL");
  if (num_sms < 1) return fail(PDA_EINVAL, "num_sms must be >= 1");
  if (batch < 0 || batch > cfg->max_batch) return fail(PDA_EINVAL, "batch out of range");
  if (max_blocks < 1 || max_blocks > cfg->max_blocks_per_seq)
    return fail(PDA_EINVAL, "max_blocks out of range");
  if (max_context_len_hint < 0) return fail(PDA_EINVAL, "max_context_len_hint < 0");
  const int G = cfg->num_q_heads / cfg->num_kv_heads;
  const int kernel = call_partial_kernel(G, cfg->head_dim, cfg->kv_fp8 != 0,
                                              call_max_len(*cfg, max_blocks, max_context_len_hint),
                                              batch, cfg->num_kv_heads);
  plan_splits(*cfg, kernel, num_sms, pda::partial_ctas_per_sm_hint(kernel, G, cfg->head_dim),
              batch, max_blocks, max_context_len_hint, 0, num_splits, chunk_pages);
  return PDA_OK;
}

int paged_decode_attn_run_ex(pda_handle h, const void* q, const void* k_cache,
                             const void* v_cache, const int32_t* block_table,
                             const int32_t* context_lens, int batch, int max_blocks,
                             int64_t num_blocks, float scale, void* out, void* stream,
                             int num_splits, int max_context_len_hint, int out_dtype) {
  return paged_decode_attn_run_scaled(h, q, k_cache, v_cache, block_table, context_lens, batch,
                                      max_blocks, num_blocks, scale, nullptr, nullptr, 0, out,
                                      stream, num_splits, max_context_len_hint, out_dtype);
}

int paged_decode_attn_run_scaled(pda_handle h, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_table,
                                 const int32_t* context_lens, int batch, int max_blocks,
                                 int64_t num_blocks, float scale, const float* k_scale,
                                 const float* v_scale, int scale_per_head, void* out,
                                 void* stream, int num_splits, int max_context_len_hint,
                                 int out_dtype) {
  if (!h) return fail(PDA_EINVAL, "handle is NULL");
  const pda_config& c = h->cfg;
  if (batch < 0 || batch > c.max_batch) return fail(PDA_EINVAL, "batch out of [0, max_batch]");
  if (batch == 0) return PDA_OK;
  if (!q || !k_cache || !v_cache || !block_table || !context_lens || !out)
    return fail(PDA_EINVAL, "a tensor pointer is NULL");
  if (max_blocks < 1 || max_blocks > c.max_blocks_per_seq)
    return fail(PDA_EINVAL, "max_blocks out of [1, max_blocks_per_seq]");
  if (num_blocks < 1 || num_blocks * c.block_size > (int64_t)INT_MAX)
    return fail(PDA_EINVAL, "num_blocks * block_size must be in [1, 2^31)");
  if (!std::isfinite(scale)) return fail(PDA_EINVAL, "scale is not finite");
  if (num_splits < 0 || num_splits > c.max_splits)
    return fail(PDA_EINVAL, "num_splits out of [0, max_splits]");
  if (max_context_len_hint < 0) return fail(PDA_EINVAL, "max_context_len_hint < 0");
  if (out_dtype == -1) out_dtype = c.dtype;
  if (out_dtype != c.dtype && out_dtype != PDA_F32)
    return fail(PDA_EINVAL, "out_dtype must be -1, the input dtype or PDA_F32");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return fail(PDA_EINVAL, "q, k_cache, v_cache and out must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_table) | reinterpret_cast<uintptr_t>(context_lens)) & 3u)
    return fail(PDA_EINVAL, "block_table and context_lens must be 4-byte aligned");

  if (scale_per_head != 0 && scale_per_head != 1)
    return fail(PDA_EINVAL, "scale_per_head must be 0 or 1");
  if ((reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale)) & 3u)
    return fail(PDA_EINVAL, "k_scale and v_scale must be 4-byte aligned");
  const size_t esz = 2;
  const size_t kv_esz = c.kv_fp8 ? 1 : 2;
  const size_t out_esz = out_dtype == PDA_F32 ? 4 : 2;
  const size_t n_q = (size_t)batch * c.num_q_heads * c.head_dim;
  const size_t cache_bytes =
      (size_t)num_blocks * c.block_size * c.num_kv_heads * c.head_dim * kv_esz;
  const size_t scale_bytes = (scale_per_head ? (size_t)c.num_kv_heads : 1) * 4;
  const size_t out_bytes = n_q * out_esz;
  if (overlaps(out, out_bytes, q, n_q * esz) || overlaps(out, out_bytes, k_cache, cache_bytes) ||
      overlaps(out, out_bytes, v_cache, cache_bytes) ||
      overlaps(out, out_bytes, block_table, (size_t)batch * max_blocks * 4) ||
      overlaps(out, out_bytes, context_lens, (size_t)batch * 4) ||
      overlaps(out, out_bytes, k_scale, k_scale ? scale_bytes : 0) ||
      overlaps(out, out_bytes, v_scale, v_scale ? scale_bytes : 0))
    return fail(PDA_EALIAS, "out overlaps an input");

  DeviceGuard guard(c.device);
  if (guard.err != cudaSuccess) return cuda_fail("cudaSetDevice", guard.err);

  if (h->tm_k != k_cache || h->tm_v != v_cache || h->tm_nb != num_blocks) {
    int st = encode_cache_map(&h->tmap_k, k_cache, c.num_kv_heads, c.head_dim, c.block_size,
                              num_blocks, c.kv_fp8 != 0);
    if (st == PDA_OK)
      st = encode_cache_map(&h->tmap_v, v_cache, c.num_kv_heads, c.head_dim, c.block_size,
                            num_blocks, c.kv_fp8 != 0);
    if (st != PDA_OK) {
      h->tm_k = h->tm_v = nullptr;
      h->tm_nb = -1;
      return st;
    }
    h->tm_k = k_cache;
    h->tm_v = v_cache;
    h->tm_nb = num_blocks;
  }

  const LaunchShape shape =
      launch_shape(h, batch, max_blocks, max_context_len_hint, num_splits);
  const int S = shape.splits, chunk = shape.chunk_pages;
  const int64_t units = shape.units;
  if (units > INT_MAX) return fail(PDA_EINVAL, "splits * num_kv_heads * batch exceeds 2^31");
  alignas(64) CUtensorMap tmap_q;
  if (shape.kernel == pda::kPartialTensorCore) {
    int st = encode_q_map(&tmap_q, q, (int64_t)batch * c.num_q_heads, c.head_dim, h->group);
    if (st != PDA_OK) return st;
  } else {
    std::memset(&tmap_q, 0, sizeof tmap_q);
  }

  pda::PartialParams p;
  p.q = q;
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.out = out;
  p.ws_o = h->ws_o;
  p.ws_lse = h->ws_lse;
  p.err = h->err;
  p.counters = h->counters;
  p.sched = h->counters + (size_t)c.max_batch * c.num_kv_heads;
  p.Hq = c.num_q_heads;
  p.Hkv = c.num_kv_heads;
  p.max_blocks = max_blocks;
  p.chunk_pages = chunk;
  p.num_splits = S;
  p.qscale = scale * pda::kLog2e;
  p.num_units = (int)units;
  p.max_ctas = h->num_sms * shape.ctas_per_sm;
  p.out_f32 = out_dtype == PDA_F32;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.scale_per_head = scale_per_head;
  p.cluster = shape.cluster;
  if (h->test_stall_runs > 0 && shape.kernel == pda::kPartialTensorCore) {
    --h->test_stall_runs;
    p.stall_units = 1;
    p.wait_ns = 1000ull * 1000ull;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = pda::launch_partial(shape.kernel, h->group, c.head_dim, c.block_size, c.dtype,
                                      c.kv_fp8 != 0, &h->tmap_k, &h->tmap_v, &tmap_q, p, batch,
                                      s);
  if (e != cudaSuccess) return cuda_fail("partial kernel launch", e);
  return PDA_OK;
}

int paged_decode_attn_run(pda_handle h, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_table, const int32_t* context_lens, int batch,
                          int max_blocks, int64_t num_blocks, float scale, void* out,
                          void* stream) {
  return paged_decode_attn_run_ex(h, q, k_cache, v_cache, block_table, context_lens, batch,
                                  max_blocks, num_blocks, scale, out, stream, 0, 0, -1);
}

int paged_decode_attn_launch_shape(pda_handle h, int batch, int max_blocks,
                                   int max_context_len_hint, int num_splits, int* splits,
                                   int* chunk_pages, int* ctas, int* cluster) {
  if (!h) return fail(PDA_EINVAL, "handle is NULL");
  if (!splits || !chunk_pages || !ctas || !cluster) return fail(PDA_EINVAL, "output pointer is NULL");
  const pda_config& c = h->cfg;
  if (batch < 1 || batch > c.max_batch) return fail(PDA_EINVAL, "batch out of [1, max_batch]");
  if (max_blocks < 1 || max_blocks > c.max_blocks_per_seq)
    return fail(PDA_EINVAL, "max_blocks out of [1, max_blocks_per_seq]");
  if (num_splits < 0 || num_splits > c.max_splits)
    return fail(PDA_EINVAL, "num_splits out of [0, max_splits]");
  if (max_context_len_hint < 0) return fail(PDA_EINVAL, "max_context_len_hint < 0");
  const LaunchShape r = launch_shape(h, batch, max_blocks, max_context_len_hint, num_splits);
  *splits = r.splits;
  *chunk_pages = r.chunk_pages;
  *ctas = r.ctas;
  *cluster = r.cluster > 1 ? r.cluster : 1;
  return PDA_OK;
}

int paged_decode_attn_merge(const float* partial_o, const float* partial_lse, int rows,
                            int num_splits, int head_dim, void* out, int out_dtype, int device,
                            void* stream) {
  if (rows < 0) return fail(PDA_EINVAL, "rows < 0");
  if (num_splits < 1 || num_splits > pda::kMaxSplits)
    return fail(PDA_EINVAL, "num_splits must be in [1, 64]");
  if (head_dim < 4 || head_dim > 512 || head_dim % 4 != 0)
    return fail(PDA_EINVAL, "head_dim must be a multiple of 4 in [4, 512]");
  if (out_dtype != PDA_BF16 && out_dtype != PDA_FP16 && out_dtype != PDA_F32)
    return fail(PDA_EINVAL, "out_dtype must be PDA_BF16, PDA_FP16 or PDA_F32");
  if (device < 0) return fail(PDA_EINVAL, "device < 0");
  if (rows == 0) return PDA_OK;
  if (!partial_o || !partial_lse || !out) return fail(PDA_EINVAL, "a pointer is NULL");
  if (!aligned16(partial_o) || !aligned16(out) || (reinterpret_cast<uintptr_t>(partial_lse) & 3u))
    return fail(PDA_EINVAL, "partial_o and out must be 16-byte aligned, partial_lse 4-byte");
  const size_t out_bytes = (size_t)rows * head_dim * (out_dtype == PDA_F32 ? 4 : 2);
  if (overlaps(out, out_bytes, partial_o, (size_t)rows * num_splits * head_dim * 4) ||
      overlaps(out, out_bytes, partial_lse, (size_t)rows * num_splits * 4))
    return fail(PDA_EALIAS, "out overlaps an input");
  DeviceGuard guard(device);
  if (guard.err != cudaSuccess) return cuda_fail("cudaSetDevice", guard.err);
  pda::MergeParams m;
  m.o = partial_o;
  m.lse = partial_lse;
  m.context_lens = nullptr;
  m.out = out;
  m.rows = rows;
  m.num_splits = num_splits;
  m.head_dim = head_dim;
  m.Hq = 1;
  m.block_size = 1;
  m.max_blocks = 1;
  m.chunk_pages = 1;
  cudaError_t e = pda::launch_merge(m, out_dtype, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("merge kernel launch", e);
  return PDA_OK;
}

int paged_decode_attn_validate(pda_handle h, const int32_t* block_table,
                               const int32_t* context_lens, int batch, int max_blocks,
                               int64_t num_blocks, void* stream) {
  if (!h) return fail(PDA_EINVAL, "handle is NULL");
  if (batch < 0 || batch > h->cfg.max_batch) return fail(PDA_EINVAL, "batch out of range");
  if (batch == 0) return PDA_OK;
  if (!block_table || !context_lens) return fail(PDA_EINVAL, "a pointer is NULL");
  if (max_blocks < 1 || max_blocks > h->cfg.max_blocks_per_seq)
    return fail(PDA_EINVAL, "max_blocks out of range");
  if (num_blocks < 1) return fail(PDA_EINVAL, "num_blocks < 1");
  DeviceGuard guard(h->cfg.device);
  if (guard.err != cudaSuccess) return cuda_fail("cudaSetDevice", guard.err);
  cudaError_t e = pda::launch_validate(block_table, context_lens, batch, max_blocks,
                                       h->cfg.block_size, num_blocks, h->err,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("validate kernel launch", e);
  return PDA_OK;
}

int paged_decode_attn_check_device_error(pda_handle h, int* code, int* detail, void* stream) {
  if (!h || !code || !detail) return fail(PDA_EINVAL, "a pointer is NULL");
  DeviceGuard guard(h->cfg.device);
  if (guard.err != cudaSuccess) return cuda_fail("cudaSetDevice", guard.err);
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
  int host[2] = {0, 0};
  e = cudaMemcpy(host, h->err, sizeof host, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->err, 0, sizeof host);
  // a kernel that gave up may have left split tickets behind
  if (e == cudaSuccess && host[0] == pda::kErrWaitTimeout)
    e = cudaMemset(h->counters, 0, h->counter_bytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail("reading the device error word", e);
  *code = host[0];
  *detail = host[1];
  return PDA_OK;
}

}  // extern "C"
