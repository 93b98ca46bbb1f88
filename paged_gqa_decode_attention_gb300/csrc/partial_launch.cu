// Host-side entry points of the partial kernels: support checks, shared-memory
// attributes, occupancy, and dispatch over (kernel, head dim, input dtype).
#include "partial_kernel.cuh"
#include "partial_tc_kernel.cuh"

namespace pda {

#define PDA_DECLARE_CC(dt, D)                                                                  \
  cudaError_t launch_partial_cc_##dt##_d##D(int, int, const CUtensorMap*, const CUtensorMap*,  \
                                            const PartialParams&, int, cudaStream_t);          \
  cudaError_t prepare_partial_cc_##dt##_d##D(int, int);                                        \
  int occupancy_partial_cc_##dt##_d##D(int, int);
PDA_DECLARE_CC(bf16, 64)
PDA_DECLARE_CC(bf16, 128)
PDA_DECLARE_CC(bf16, 256)
PDA_DECLARE_CC(fp16, 64)
PDA_DECLARE_CC(fp16, 128)
PDA_DECLARE_CC(fp16, 256)
#undef PDA_DECLARE_CC

#define PDA_DECLARE_TC(dt, D)                                                                  \
  cudaError_t launch_partial_tc_##dt##_d##D(int, int, const CUtensorMap*, const CUtensorMap*,  \
                                            const CUtensorMap*, const PartialParams&,          \
                                            cudaStream_t);                                     \
  cudaError_t prepare_partial_tc_##dt##_d##D(int, int);                                        \
  int occupancy_partial_tc_##dt##_d##D(int, int);                                             \
  int max_clusters_partial_tc_##dt##_d##D(int, int, int);
PDA_DECLARE_TC(bf16, 64)
PDA_DECLARE_TC(bf16, 128)
PDA_DECLARE_TC(fp16, 64)
PDA_DECLARE_TC(fp16, 128)
PDA_DECLARE_TC(kv8_bf16, 64)
PDA_DECLARE_TC(kv8_bf16, 128)
PDA_DECLARE_TC(kv8_fp16, 64)
PDA_DECLARE_TC(kv8_fp16, 128)
// group sizes 9..16
PDA_DECLARE_TC(bf16, 64_g16)
PDA_DECLARE_TC(bf16, 128_g16)
PDA_DECLARE_TC(fp16, 64_g16)
PDA_DECLARE_TC(fp16, 128_g16)
PDA_DECLARE_TC(kv8_bf16, 64_g16)
PDA_DECLARE_TC(kv8_bf16, 128_g16)
PDA_DECLARE_TC(kv8_fp16, 64_g16)
PDA_DECLARE_TC(kv8_fp16, 128_g16)
#undef PDA_DECLARE_TC

namespace {

// Calls the CUDA-core function for (dtype, head dim): `f` receives the
// matching launch, prepare and occupancy entry points.
template <typename F>
auto with_cc(int dtype, int head_dim, F f) {
#define PDA_CC_CASE(dt, D)                                                             \
  return f(launch_partial_cc_##dt##_d##D, prepare_partial_cc_##dt##_d##D,              \
           occupancy_partial_cc_##dt##_d##D)
  if (dtype == 1) {
    if (head_dim == 64) PDA_CC_CASE(fp16, 64);
    if (head_dim == 256) PDA_CC_CASE(fp16, 256);
    PDA_CC_CASE(fp16, 128);
  }
  if (head_dim == 64) PDA_CC_CASE(bf16, 64);
  if (head_dim == 256) PDA_CC_CASE(bf16, 256);
  PDA_CC_CASE(bf16, 128);
#undef PDA_CC_CASE
}

// Same for the tensor-core kernel (head dims 64 and 128, 16-bit or FP8 K/V, bf16 or
// fp16 queries; group sizes 9..16 in their own units).
template <typename F>
auto with_tc(int dtype, int head_dim, bool kv_fp8, int group, F f) {
#define PDA_TC_CASE(dt, D)                                                             \
  return f(launch_partial_tc_##dt##_d##D, prepare_partial_tc_##dt##_d##D,              \
           occupancy_partial_tc_##dt##_d##D, max_clusters_partial_tc_##dt##_d##D)
  if (group > 8) {
    if (kv_fp8) {
      if (dtype == 1) {
        if (head_dim == 64) PDA_TC_CASE(kv8_fp16, 64_g16);
        PDA_TC_CASE(kv8_fp16, 128_g16);
      }
      if (head_dim == 64) PDA_TC_CASE(kv8_bf16, 64_g16);
      PDA_TC_CASE(kv8_bf16, 128_g16);
    }
    if (dtype == 1) {
      if (head_dim == 64) PDA_TC_CASE(fp16, 64_g16);
      PDA_TC_CASE(fp16, 128_g16);
    }
    if (head_dim == 64) PDA_TC_CASE(bf16, 64_g16);
    PDA_TC_CASE(bf16, 128_g16);
  }
  if (kv_fp8) {
    if (dtype == 1) {
      if (head_dim == 64) PDA_TC_CASE(kv8_fp16, 64);
      PDA_TC_CASE(kv8_fp16, 128);
    }
    if (head_dim == 64) PDA_TC_CASE(kv8_bf16, 64);
    PDA_TC_CASE(kv8_bf16, 128);
  }
  if (dtype == 1) {
    if (head_dim == 64) PDA_TC_CASE(fp16, 64);
    PDA_TC_CASE(fp16, 128);
  }
  if (head_dim == 64) PDA_TC_CASE(bf16, 64);
  PDA_TC_CASE(bf16, 128);
#undef PDA_TC_CASE
}

}  // namespace

bool partial_supported(int group, int head_dim, int block_size, int dtype, bool kv_fp8) {
  const bool bs_ok = block_size == 16 || block_size == 32 || (block_size == 64 && group <= 8);
  if (kv_fp8)
    return tc::geometry_supported(group, head_dim, true) && bs_ok && (dtype == 0 || dtype == 1);
  return (partial::geometry_supported(group, head_dim) ||
          tc::geometry_supported(group, head_dim, false)) &&
         bs_ok && (dtype == 0 || dtype == 1);
}

bool partial_kernel_supported(int kernel, int group, int head_dim, bool kv_fp8) {
  if (kernel == kPartialTensorCore) return tc::geometry_supported(group, head_dim, kv_fp8);
  return kernel == kPartialCudaCore && !kv_fp8 && partial::geometry_supported(group, head_dim);
}

cudaError_t partial_prepare(int kernel, int group, int head_dim, int block_size, int dtype,
                            bool kv_fp8) {
  if (kernel == kPartialTensorCore)
    return with_tc(dtype, head_dim, kv_fp8, group, [&](auto, auto prepare, auto, auto) {
      return prepare(group, block_size);
    });
  return with_cc(dtype, head_dim, [&](auto, auto prepare, auto) {
    return prepare(group, block_size);
  });
}

int partial_ctas_per_sm(int kernel, int group, int head_dim, int block_size, int dtype,
                        bool kv_fp8) {
  if (kernel == kPartialTensorCore)
    return with_tc(dtype, head_dim, kv_fp8, group, [&](auto, auto, auto occupancy, auto) {
      return occupancy(group, block_size);
    });
  return with_cc(dtype, head_dim, [&](auto, auto, auto occupancy) {
    return occupancy(group, block_size);
  });
}

int partial_max_clusters(int group, int head_dim, int block_size, int dtype, bool kv_fp8,
                         int cluster) {
  if (!tc::geometry_supported(group, head_dim, kv_fp8) || cluster < 2 || cluster > 16) return 0;
  return with_tc(dtype, head_dim, kv_fp8, group, [&](auto, auto, auto, auto max_clusters) {
    return max_clusters(group, block_size, cluster);
  });
}

cudaError_t launch_partial(int kernel, int group, int head_dim, int block_size, int dtype,
                           bool kv_fp8, const CUtensorMap* tk, const CUtensorMap* tv,
                           const CUtensorMap* tq, const PartialParams& p, int batch,
                           cudaStream_t stream) {
  if (kernel == kPartialTensorCore)
    return with_tc(dtype, head_dim, kv_fp8, group, [&](auto launch, auto, auto, auto) {
      return launch(group, block_size, tk, tv, tq, p, stream);
    });
  return with_cc(dtype, head_dim, [&](auto launch, auto, auto) {
    return launch(group, block_size, tk, tv, p, batch, stream);
  });
}

}  // namespace pda
