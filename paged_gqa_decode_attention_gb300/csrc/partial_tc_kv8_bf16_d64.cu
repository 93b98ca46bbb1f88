// Instantiations of the tensor-core split-K partial kernel for FP8 (E4M3)
// K/V caches with bf16 queries and head dim 64.
#include "partial_tc_kernel.cuh"

namespace pda {

cudaError_t launch_partial_tc_kv8_bf16_d64(int G, int BS, const CUtensorMap* tk,
                                            const CUtensorMap* tv, const CUtensorMap* tq,
                                            const PartialParams& p, cudaStream_t s) {
  return tc::Dispatch<64, false, true>::launch(G, BS, tk, tv, tq, p, s);
}

cudaError_t prepare_partial_tc_kv8_bf16_d64(int G, int BS) {
  return tc::Dispatch<64, false, true>::prepare(G, BS);
}

int occupancy_partial_tc_kv8_bf16_d64(int G, int BS) {
  return tc::Dispatch<64, false, true>::occupancy(G, BS);
}

int max_clusters_partial_tc_kv8_bf16_d64(int G, int BS, int cluster) {
  return tc::Dispatch<64, false, true>::max_clusters(G, BS, cluster);
}

}  // namespace pda
