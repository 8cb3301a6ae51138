// Instantiation: attention forward, bf16_d64.
#include "attn_kernel.cuh"
#include "launchers.h"

namespace gb300 {

cudaError_t launch_attn_bf16_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& o, const AttnParams& p, int grid, cudaStream_t stream) {
  return launch_attn<64, false>(q, k, v, o, p, grid, stream);
}

int status_attn_bf16_d64(bool clear) { return read_tu_status(clear); }

}  // namespace gb300
