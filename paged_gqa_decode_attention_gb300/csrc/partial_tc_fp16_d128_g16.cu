// Instantiations of the tensor-core split-K partial kernel for fp16 inputs,
// head dim 128 and group sizes 9..16.
#include "partial_tc_kernel.cuh"

namespace pda {

cudaError_t launch_partial_tc_fp16_d128_g16(int G, int BS, const CUtensorMap* tk,
                                            const CUtensorMap* tv, const CUtensorMap* tq,
                                            const PartialParams& p, cudaStream_t s) {
  return tc::Dispatch<128, true, false, 9, 16>::launch(G, BS, tk, tv, tq, p, s);
}

cudaError_t prepare_partial_tc_fp16_d128_g16(int G, int BS) {
  return tc::Dispatch<128, true, false, 9, 16>::prepare(G, BS);
}

int occupancy_partial_tc_fp16_d128_g16(int G, int BS) {
  return tc::Dispatch<128, true, false, 9, 16>::occupancy(G, BS);
}

int max_clusters_partial_tc_fp16_d128_g16(int G, int BS, int cluster) {
  return tc::Dispatch<128, true, false, 9, 16>::max_clusters(G, BS, cluster);
}

}  // namespace pda
