// Instantiations of the tensor-core split-K partial kernel for fp16 inputs.
#include "partial_tc_kernel.cuh"

namespace pda {

cudaError_t launch_partial_tc_fp16(int G, int BS, bool f32, const CUtensorMap* tk,
                                  const CUtensorMap* tv, const CUtensorMap* tq,
                                  const PartialParams& p, cudaStream_t s) {
  return tc::Dispatch<true>::launch(G, BS, f32, tk, tv, tq, p, s);
}

cudaError_t prepare_partial_tc_fp16(int G, int BS) { return tc::Dispatch<true>::prepare(G, BS); }

int occupancy_partial_tc_fp16(int G, int BS) { return tc::Dispatch<true>::occupancy(G, BS); }

}  // namespace pda
