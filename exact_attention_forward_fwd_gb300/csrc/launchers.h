// Entry points of the per-configuration kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace gb300 {

struct AttnParams;

cudaError_t launch_attn_bf16_d64(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                 const AttnParams&, int grid, cudaStream_t);
cudaError_t launch_attn_bf16_d128(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                  const AttnParams&, int grid, cudaStream_t);
cudaError_t launch_attn_fp8_d128(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                 const AttnParams&, int grid, cudaStream_t);
int status_attn_bf16_d64(bool clear);
int status_attn_bf16_d128(bool clear);
int status_attn_fp8_d128(bool clear);

// FP8 operand preparation: x bf16 [BH][N][128] -> e4m3 (row layout, or
// transposed [BH][128][Npad]) plus per-128-row-block scales; persistent grid of
// three CTAs per SM (sms = the device's SM count).
cudaError_t launch_fp8_prep(const void* x, void* x8, float* scales, const signed char* signs,
                            int BH, int H, int N, int transpose_out, int sms, cudaStream_t stream);
int status_fp8_prep(bool clear);

// Split-KV merge of `splits` partial results ([splits][BH][N][D] fp32 O,
// [splits][BH][N] lse) into O bf16 [BH][N][D] and lse [BH][N] (lse may be null).
cudaError_t launch_splitkv_merge(const float* o_part, const float* lse_part, void* o, float* lse,
                                 int splits, int BH, int N, int D, cudaStream_t stream);

// Attention backward: prep (D, scaled lse), dK/dV kernel, dQ kernel, in
// order on `stream`.  lp, dd: [BH][Npad] f32 scratch.
struct BwdParams;
cudaError_t launch_attn_bwd(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dO, const BwdParams& p, const void* o,
                            const void* dO_ptr, const float* lse, float* lp, float* dd, int sms,
                            cudaStream_t stream);
int status_attn_bwd(bool clear);

}  // namespace gb300
