// Host-side entry points of the partial kernels: support checks, shared-memory
// attributes, occupancy, and dispatch over (kernel, input dtype).
#include "partial_kernel.cuh"

namespace pda {

cudaError_t launch_partial_bf16(int, int, bool, const CUtensorMap*, const CUtensorMap*,
                               const PartialParams&, int, cudaStream_t);
cudaError_t launch_partial_fp16(int, int, bool, const CUtensorMap*, const CUtensorMap*,
                               const PartialParams&, int, cudaStream_t);
cudaError_t launch_partial_tc_bf16(int, int, bool, const CUtensorMap*, const CUtensorMap*,
                                  const CUtensorMap*, const PartialParams&, cudaStream_t);
cudaError_t launch_partial_tc_fp16(int, int, bool, const CUtensorMap*, const CUtensorMap*,
                                  const CUtensorMap*, const PartialParams&, cudaStream_t);
cudaError_t prepare_partial_bf16(int, int);
cudaError_t prepare_partial_fp16(int, int);
cudaError_t prepare_partial_tc_bf16(int, int);
cudaError_t prepare_partial_tc_fp16(int, int);
int occupancy_partial_bf16(int, int);
int occupancy_partial_fp16(int, int);
int occupancy_partial_tc_bf16(int, int);
int occupancy_partial_tc_fp16(int, int);

bool partial_supported(int group, int block_size, int dtype) {
  const bool g_ok = group == 1 || group == 2 || group == 4 || group == 8;
  const bool bs_ok = block_size == 16 || block_size == 32;
  return g_ok && bs_ok && (dtype == 0 || dtype == 1);
}

bool partial_kernel_supported(int kernel, int group) {
  if (kernel == kPartialTensorCore) return group == 4 || group == 8;
  return kernel == kPartialCudaCore;
}

cudaError_t partial_prepare(int kernel, int group, int block_size, int dtype) {
  if (kernel == kPartialTensorCore)
    return dtype == 1 ? prepare_partial_tc_fp16(group, block_size)
                      : prepare_partial_tc_bf16(group, block_size);
  return dtype == 1 ? prepare_partial_fp16(group, block_size)
                    : prepare_partial_bf16(group, block_size);
}

int partial_ctas_per_sm(int kernel, int group, int block_size, int dtype) {
  if (kernel == kPartialTensorCore)
    return dtype == 1 ? occupancy_partial_tc_fp16(group, block_size)
                      : occupancy_partial_tc_bf16(group, block_size);
  return dtype == 1 ? occupancy_partial_fp16(group, block_size)
                    : occupancy_partial_bf16(group, block_size);
}

cudaError_t launch_partial(int kernel, int group, int block_size, int dtype, bool out_f32,
                           const CUtensorMap* tk, const CUtensorMap* tv, const CUtensorMap* tq,
                           const PartialParams& p, int batch, cudaStream_t stream) {
  if (kernel == kPartialTensorCore)
    return dtype == 1 ? launch_partial_tc_fp16(group, block_size, out_f32, tk, tv, tq, p, stream)
                      : launch_partial_tc_bf16(group, block_size, out_f32, tk, tv, tq, p, stream);
  return dtype == 1 ? launch_partial_fp16(group, block_size, out_f32, tk, tv, p, batch, stream)
                    : launch_partial_bf16(group, block_size, out_f32, tk, tv, p, batch, stream);
}

}  // namespace pda
