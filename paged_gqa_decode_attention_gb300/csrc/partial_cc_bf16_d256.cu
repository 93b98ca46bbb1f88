// Instantiations of the CUDA-core split-K partial kernel for bf16 inputs and
// head dim 256 (one translation unit per (dtype, head dim) so they compile in
// parallel).
#include "partial_kernel.cuh"

namespace pda {

cudaError_t launch_partial_cc_bf16_d256(int G, int BS, const CUtensorMap* tk,
                                         const CUtensorMap* tv, const PartialParams& p, int batch,
                                         cudaStream_t s) {
  return partial::Dispatch<256, false>::launch(G, BS, tk, tv, p, batch, s);
}

cudaError_t prepare_partial_cc_bf16_d256(int G, int BS) {
  return partial::Dispatch<256, false>::prepare(G, BS);
}

int occupancy_partial_cc_bf16_d256(int G, int BS) {
  return partial::Dispatch<256, false>::occupancy(G, BS);
}

}  // namespace pda
