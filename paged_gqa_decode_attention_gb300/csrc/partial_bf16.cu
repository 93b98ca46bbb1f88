// Instantiations of the split-K partial kernel for bf16 inputs (one
// translation unit per input dtype so the two compile in parallel).
#include "partial_kernel.cuh"

namespace pda {

cudaError_t launch_partial_bf16(int G, int BS, bool f32, const CUtensorMap* tk,
                               const CUtensorMap* tv, const PartialParams& p, int batch,
                               cudaStream_t s) {
  return partial::Dispatch<false>::launch(G, BS, f32, tk, tv, p, batch, s);
}

cudaError_t prepare_partial_bf16(int G, int BS) { return partial::Dispatch<false>::prepare(G, BS); }

int occupancy_partial_bf16(int G, int BS) { return partial::Dispatch<false>::occupancy(G, BS); }

}  // namespace pda
