// Instantiations of the tensor-core split-K partial kernel for fp16 inputs
// and head dim 64.
#include "partial_tc_kernel.cuh"

namespace pda {

cudaError_t launch_partial_tc_fp16_d64(int G, int BS, const CUtensorMap* tk,
                                         const CUtensorMap* tv, const CUtensorMap* tq,
                                         const PartialParams& p, cudaStream_t s) {
  return tc::Dispatch<64, true, false>::launch(G, BS, tk, tv, tq, p, s);
}

cudaError_t prepare_partial_tc_fp16_d64(int G, int BS) {
  return tc::Dispatch<64, true, false>::prepare(G, BS);
}

int occupancy_partial_tc_fp16_d64(int G, int BS) {
  return tc::Dispatch<64, true, false>::occupancy(G, BS);
}

int max_clusters_partial_tc_fp16_d64(int G, int BS, int cluster) {
  return tc::Dispatch<64, true, false>::max_clusters(G, BS, cluster);
}

}  // namespace pda
