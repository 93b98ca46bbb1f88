// Host-side entry points of the partial kernel: geometry facts for the
// planner and dtype dispatch.
#include "partial_kernel.cuh"

namespace pda {

cudaError_t launch_partial_bf16(int, int, bool, const CUtensorMap*, const CUtensorMap*,
                               const PartialParams&, int, cudaStream_t);
cudaError_t launch_partial_fp16(int, int, bool, const CUtensorMap*, const CUtensorMap*,
                               const PartialParams&, int, cudaStream_t);
cudaError_t prepare_partial_bf16(int, int);
cudaError_t prepare_partial_fp16(int, int);
int occupancy_partial_bf16(int, int);
int occupancy_partial_fp16(int, int);

int partial_threads() { return partial::kThreads; }

size_t partial_smem_bytes(int) { return partial::kSmemBytes; }

bool partial_supported(int group, int block_size, int dtype) {
  const bool g_ok = group == 1 || group == 2 || group == 4 || group == 8;
  const bool bs_ok = block_size == 16 || block_size == 32;
  return g_ok && bs_ok && (dtype == 0 || dtype == 1);
}

cudaError_t partial_prepare(int group, int block_size, int dtype) {
  return dtype == 1 ? prepare_partial_fp16(group, block_size)
                    : prepare_partial_bf16(group, block_size);
}

int partial_ctas_per_sm(int group, int block_size, int dtype) {
  return dtype == 1 ? occupancy_partial_fp16(group, block_size)
                    : occupancy_partial_bf16(group, block_size);
}

cudaError_t launch_partial(int group, int block_size, int dtype, bool out_f32,
                           const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                           const PartialParams& p, int batch, cudaStream_t stream) {
  return dtype == 1
             ? launch_partial_fp16(group, block_size, out_f32, tmap_k, tmap_v, p, batch, stream)
             : launch_partial_bf16(group, block_size, out_f32, tmap_k, tmap_v, p, batch, stream);
}

}  // namespace pda
