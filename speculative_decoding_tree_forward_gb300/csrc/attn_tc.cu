// tcgen05 / TMEM tree attention for 128 packed query rows per KV head.
// (Not yet implemented: the automatic path uses the warp-MMA kernel.)
#include "attn_common.cuh"

namespace ts {

bool attn_tc_available() { return false; }
int attn_tc_occupancy(int, int) { return 0; }
size_t attn_tc_smem_bytes(int, int) { return 0; }
int attn_tc_threads() { return 0; }
cudaError_t launch_attn_tc(const AttnParams&, const CUtensorMap&, const CUtensorMap&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace ts
