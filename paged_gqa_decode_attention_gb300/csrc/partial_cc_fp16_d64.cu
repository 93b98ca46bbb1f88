// Instantiations of the CUDA-core split-K partial kernel for fp16 inputs and
// head dim 64 (one translation unit per (dtype, head dim) so they compile in
// parallel).
#include "partial_kernel.cuh"

namespace pda {

cudaError_t launch_partial_cc_fp16_d64(int G, int BS, const CUtensorMap* tk,
                                         const CUtensorMap* tv, const PartialParams& p, int batch,
                                         cudaStream_t s) {
  return partial::Dispatch<64, true>::launch(G, BS, tk, tv, p, batch, s);
}

cudaError_t prepare_partial_cc_fp16_d64(int G, int BS) {
  return partial::Dispatch<64, true>::prepare(G, BS);
}

int occupancy_partial_cc_fp16_d64(int G, int BS) {
  return partial::Dispatch<64, true>::occupancy(G, BS);
}

}  // namespace pda
