// paged_decode_attn_run_noalloc: the decode-attention call for callers that
// must not allocate device memory (see the header for who they are).
//
// It launches the same split-K partial kernel as paged_decode_attn_run_ex,
// but its scratch (split partials, split LSEs, split tickets and the error
// word) is a fixed array compiled into this library
// instead of a handle's cudaMalloc'd workspace. Nothing here allocates:
// no cudaMalloc/cudaFree, no allocating library routine.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <set>
#include <tuple>

#include "paged_decode_attn.h"
#include "pda_internal.h"

namespace {

// Scratch capacity: 2^21 floats (8 MiB) of split partial outputs, 2^16 floats
// (256 KiB) of split LSEs, 64 ints for the kernels' error word, 2^16 ints
// (256 KiB) of split tickets, one per (sequence, kv head), and the 2 work
// counters of the persistent kernel.
constexpr size_t kPartialFloats = size_t(1) << 21;
constexpr size_t kLseFloats = size_t(1) << 16;
constexpr size_t kErrInts = 64;
constexpr size_t kCounterInts = size_t(1) << 16;  // split tickets
constexpr size_t kSchedInts = 2;                  // persistent kernel's work counters
constexpr size_t kScratchBytes =
    (kPartialFloats + kLseFloats) * 4 + (kErrInts + kCounterInts + kSchedInts) * 4;

// One copy per GPU that loads the library, alive until the process exits.
// In host code this name is only a stand-in for the symbol; the device
// address comes from cudaGetSymbolAddress at set-up.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};  // device address of the array, per device
int g_num_sms[kMaxDevices] = {};
std::set<std::tuple<int, int, int, int>> g_prepared;  // (device, group * 1024 + head_dim, block_size, dtype)

int fail(int code, const char* msg) { return pda::set_last_error(code, msg); }

int cuda_fail(const char* what, cudaError_t e) {
  char buf[256];
  snprintf(buf, sizeof buf, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  return fail(PDA_ECUDA, buf);
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return na && nb && a0 < b0 + nb && b0 < a0 + na;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

// Same descriptor as the handle path: [num_blocks * block_size, Hkv * D]
// view, 64 x block_size boxes, 128-byte swizzle. Fills a host struct only.
bool encode(CUtensorMap* m, const void* base, int Hkv, int D, int bs, int64_t num_blocks) {
  auto fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)Hkv * D, (cuuint64_t)num_blocks * bs};
  cuuint64_t strides[1] = {(cuuint64_t)Hkv * D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)bs};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B * Hq, D] view of q, boxes of 64 dims x G rows (tensor-core kernel).
bool encode_q(CUtensorMap* m, const void* q, int64_t rows, int D, int group) {
  auto fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)group};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Once per device (with `dev` current): the scratch array's device address,
// the SM count, and the kernels' shared-memory limit for this geometry.
int setup_device(int dev, int group, int head_dim, int bs, int dtype, void** scratch,
                 int* num_sms) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_fail("cudaGetSymbolAddress(scratch)", e);
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail("cudaDeviceGetAttribute", e);
    g_num_sms[dev] = sms;
    g_scratch_addr[dev] = p;
  }
  const auto key = std::make_tuple(dev, group * 1024 + head_dim, bs, dtype);
  if (!g_prepared.count(key)) {
    cudaError_t e = pda::partial_prepare(pda::default_partial_kernel(group, head_dim), group,
                                         head_dim, bs, dtype, false);
    if (e != cudaSuccess) return cuda_fail("cudaFuncSetAttribute", e);
    g_prepared.insert(key);
  }
  *scratch = g_scratch_addr[dev];
  *num_sms = g_num_sms[dev];
  return PDA_OK;
}

}  // namespace

extern "C" int paged_decode_attn_run_noalloc(const void* q, const void* k_cache,
                                             const void* v_cache, const int32_t* block_table,
                                             const int32_t* context_lens, int batch,
                                             int num_q_heads, int num_kv_heads, int head_dim,
                                             int block_size, int dtype, int max_blocks,
                                             int64_t num_blocks, float scale, void* out,
                                             int num_splits, int device, void* stream) {
  if (batch < 0 || batch > 65535) return fail(PDA_EINVAL, "batch must be in [0, 65535]");
  if (max_blocks < 1) return fail(PDA_EINVAL, "max_blocks must be >= 1");
  if (device < 0 || device >= kMaxDevices) return fail(PDA_EINVAL, "device out of range");
  pda_config cfg = {num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                    batch > 0 ? batch : 1, max_blocks, 64, device};
  int S = 1, chunk = 1;
  // shape validation (host only): the same checks as create
  int st = paged_decode_attn_plan(&cfg, 1, batch, max_blocks, 0, &S, &chunk);
  if (st != PDA_OK) return st;
  if (batch == 0) return PDA_OK;
  if (!q || !k_cache || !v_cache || !block_table || !context_lens || !out)
    return fail(PDA_EINVAL, "a tensor pointer is NULL");
  if (num_blocks < 1 || num_blocks * block_size > (int64_t)INT_MAX)
    return fail(PDA_EINVAL, "num_blocks * block_size must be in [1, 2^31)");
  if (!std::isfinite(scale)) return fail(PDA_EINVAL, "scale is not finite");
  if (num_splits < 0 || num_splits > pda::kMaxSplits)
    return fail(PDA_EINVAL, "num_splits out of [0, 64]");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return fail(PDA_EINVAL, "q, k_cache, v_cache and out must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_table) | reinterpret_cast<uintptr_t>(context_lens)) & 3u)
    return fail(PDA_EINVAL, "block_table and context_lens must be 4-byte aligned");
  const size_t n_q = (size_t)batch * num_q_heads * head_dim;
  const size_t cache_bytes = (size_t)num_blocks * block_size * num_kv_heads * head_dim * 2;
  if (overlaps(out, n_q * 2, q, n_q * 2) || overlaps(out, n_q * 2, k_cache, cache_bytes) ||
      overlaps(out, n_q * 2, v_cache, cache_bytes) ||
      overlaps(out, n_q * 2, block_table, (size_t)batch * max_blocks * 4) ||
      overlaps(out, n_q * 2, context_lens, (size_t)batch * 4))
    return fail(PDA_EALIAS, "out overlaps an input");

  // Split count that fits the scratch: rows * S * D partial floats, rows * S LSEs.
  const size_t rows = (size_t)batch * num_q_heads;
  size_t fit = kPartialFloats / (rows * head_dim);
  if (kLseFloats / rows < fit) fit = kLseFloats / rows;
  if ((size_t)batch * num_kv_heads > kCounterInts) fit = 1;  // no room for split tickets
  // An explicit request runs as S = ceil(max_blocks / chunk) splits of chunk
  // pages (the handle path's rule); only that S has to fit.
  if (num_splits > 0) {
    const int cap = num_splits < max_blocks ? num_splits : max_blocks;
    chunk = (max_blocks + cap - 1) / cap;
    S = (max_blocks + chunk - 1) / chunk;
    if (S > 1 && (size_t)S > fit) {
      char buf[320];
      snprintf(buf, sizeof buf,
               "num_splits %d runs as %d splits, which need %zu bytes of split partials; the "
               "built-in scratch holds %zu (at most %zu splits for this batch)",
               num_splits, S, rows * (size_t)S * (head_dim + 1) * 4,
               (kPartialFloats + kLseFloats) * 4, fit);
      return fail(PDA_EINVAL, buf);
    }
  }

  int prev = -1;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  if (prev != device && (e = cudaSetDevice(device)) != cudaSuccess)
    return cuda_fail("cudaSetDevice", e);
  struct Restore {
    int prev, dev;
    ~Restore() {
      if (prev != dev) cudaSetDevice(prev);
    }
  } restore{prev, device};

  const int group = num_q_heads / num_kv_heads;
  void* scratch = nullptr;
  int num_sms = 1;
  st = setup_device(device, group, head_dim, block_size, dtype, &scratch, &num_sms);
  if (st != PDA_OK) return st;

  if (num_splits == 0) {
    cfg.max_splits = fit < 1 ? 1 : (fit > (size_t)pda::kMaxSplits ? pda::kMaxSplits : (int)fit);
    st = paged_decode_attn_plan(&cfg, num_sms, batch, max_blocks, 0, &S, &chunk);
    if (st != PDA_OK) return st;
  }

  const int kernel = pda::default_partial_kernel(group, head_dim);
  const int64_t units = (int64_t)S * num_kv_heads * batch;
  if (units > INT_MAX) return fail(PDA_EINVAL, "splits * num_kv_heads * batch exceeds 2^31");
  alignas(64) CUtensorMap tk, tv, tq;
  std::memset(&tq, 0, sizeof tq);
  if (!encode(&tk, k_cache, num_kv_heads, head_dim, block_size, num_blocks) ||
      !encode(&tv, v_cache, num_kv_heads, head_dim, block_size, num_blocks) ||
      (kernel == pda::kPartialTensorCore &&
       !encode_q(&tq, q, (int64_t)batch * num_q_heads, head_dim, group)))
    return fail(PDA_ECUDA, "cuTensorMapEncodeTiled failed");

  float* ws_o = static_cast<float*>(scratch);
  float* ws_lse = ws_o + kPartialFloats;
  int* err = reinterpret_cast<int*>(ws_lse + kLseFloats);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* counters = err + kErrInts;
  // the error word and the split tickets must start at zero; the partials are
  // fully written before use
  int* sched = counters + kCounterInts;
  e = cudaMemsetAsync(err, 0, 2 * sizeof(int), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(sched, 0, kSchedInts * sizeof(int), s);
  if (e == cudaSuccess && S > 1)
    e = cudaMemsetAsync(counters, 0, (size_t)batch * num_kv_heads * sizeof(int), s);
  if (e != cudaSuccess) return cuda_fail("cudaMemsetAsync(scratch)", e);

  pda::PartialParams p;
  p.q = q;
  p.block_table = block_table;
  p.context_lens = context_lens;
  p.out = out;
  p.ws_o = ws_o;
  p.ws_lse = ws_lse;
  p.err = err;
  p.counters = counters;
  p.sched = sched;
  p.Hq = num_q_heads;
  p.Hkv = num_kv_heads;
  p.max_blocks = max_blocks;
  p.chunk_pages = chunk;
  p.num_splits = S;
  p.qscale = scale * pda::kLog2e;
  p.num_units = (int)units;
  p.max_ctas = num_sms * pda::partial_ctas_per_sm_hint(kernel, group, head_dim);
  p.out_f32 = 0;
  p.k_scale = nullptr;
  p.v_scale = nullptr;
  p.scale_per_head = 0;
  e = pda::launch_partial(kernel, group, head_dim, block_size, dtype, false, &tk, &tv, &tq, p,
                          batch, s);
  if (e != cudaSuccess) return cuda_fail("partial kernel launch", e);
  return PDA_OK;
}
