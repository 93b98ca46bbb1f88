// Instantiations of the tensor-core split-K partial kernel for bf16 inputs.
#include "partial_tc_kernel.cuh"

namespace pda {

cudaError_t launch_partial_tc_bf16(int G, int BS, bool f32, const CUtensorMap* tk,
                                  const CUtensorMap* tv, const CUtensorMap* tq,
                                  const PartialParams& p, cudaStream_t s) {
  return tc::Dispatch<false>::launch(G, BS, f32, tk, tv, tq, p, s);
}

cudaError_t prepare_partial_tc_bf16(int G, int BS) { return tc::Dispatch<false>::prepare(G, BS); }

int occupancy_partial_tc_bf16(int G, int BS) { return tc::Dispatch<false>::occupancy(G, BS); }

}  // namespace pda
