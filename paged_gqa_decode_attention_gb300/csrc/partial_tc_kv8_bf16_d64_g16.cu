// Instantiations of the tensor-core split-K partial kernel for FP8 (E4M3)
// K/V caches with bf16 queries,
// head dim 64 and group sizes 9..16.
#include "partial_tc_kernel.cuh"

namespace pda {

cudaError_t launch_partial_tc_kv8_bf16_d64_g16(int G, int BS, const CUtensorMap* tk,
                                            const CUtensorMap* tv, const CUtensorMap* tq,
                                            const PartialParams& p, cudaStream_t s) {
  return tc::Dispatch<64, false, true, 9, 16>::launch(G, BS, tk, tv, tq, p, s);
}

cudaError_t prepare_partial_tc_kv8_bf16_d64_g16(int G, int BS) {
  return tc::Dispatch<64, false, true, 9, 16>::prepare(G, BS);
}

int occupancy_partial_tc_kv8_bf16_d64_g16(int G, int BS) {
  return tc::Dispatch<64, false, true, 9, 16>::occupancy(G, BS);
}

int max_clusters_partial_tc_kv8_bf16_d64_g16(int G, int BS, int cluster) {
  return tc::Dispatch<64, false, true, 9, 16>::max_clusters(G, BS, cluster);
}

}  // namespace pda
