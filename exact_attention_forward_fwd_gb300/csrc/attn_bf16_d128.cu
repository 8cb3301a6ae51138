// Instantiation: attention forward, bf16_d128.
#include "attn_kernel.cuh"
#include "launchers.h"

namespace gb300 {

cudaError_t launch_attn_bf16_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& o, const AttnParams& p, int grid, cudaStream_t stream) {
  return launch_attn<128, false>(q, k, v, o, p, grid, stream);
}

int status_attn_bf16_d128(bool clear) { return read_tu_status(clear); }

}  // namespace gb300
