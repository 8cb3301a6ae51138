// FP8 E4M3 operand preparation (memory-bound): optional incoherent-processing
// rotation of each row by H_128 diag(signs) (fast Walsh-Hadamard transform),
// then per block of 128 rows: s = amax / 448 (1 for an all-zero block) and
// codes = E4M3_rn_satfinite(x / s).
//
// Sources: "4.3 FlashAttention 2 & 3: Work Partitioning, Warp Specialization &
// FP8", section "Incoherent processing: rotate away the outliers" (M = H D
// applied as x M, orthonormal Sylvester H, O(d log d) fast transform, s =
// amax / 448); "FlashAttention-3: How Warp Specialization, Asynchronous TMA
// Tiling, and FP8 Hardware Acceleration Scale Attention on Hopper GPUs",
// section 4 (one scale per block of each operand).
//
// One CTA per (batch*head, 128-row block), 8 warps x 16 rows; each lane owns
// 4 consecutive columns of a 128-column row.  Butterfly stages of half-width
// 1 and 2 stay inside a lane; stages 4..64 exchange with lane ^ (h / 4).
#include <cuda_runtime.h>

#include <cstdint>

#include "launchers.h"
#include "ptx.cuh"

namespace gb300 {

namespace {

constexpr int kRows = 128;
constexpr int kD = 128;
constexpr float kInvSqrtD = 0.08838834764831845f;   // 1 / sqrt(128)

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

template <bool ROTATE, bool TRANSPOSE>
__global__ void __launch_bounds__(256) fp8_prep_kernel(const uint16_t* __restrict__ x,
                                                       uint8_t* __restrict__ x8,
                                                       float* __restrict__ scales,
                                                       const int8_t* __restrict__ signs, int H,
                                                       int N, int nblk, int Npad) {
  __shared__ float warp_max[8];
  const int blk = blockIdx.x % nblk;
  const int bh = blockIdx.x / nblk;
  const int h = bh % H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  float sg[4] = {1.f, 1.f, 1.f, 1.f};
  if (ROTATE) {
    const uint32_t s4 = *reinterpret_cast<const uint32_t*>(signs + (size_t)h * kD + 4 * lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) sg[e] = static_cast<float>(static_cast<int8_t>((s4 >> (8 * e)) & 0xFF)) * kInvSqrtD;
  }

  float v[16][4];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int r = blk * kRows + warp * 16 + i;
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < N) {
      const uint2 raw = *reinterpret_cast<const uint2*>(x + ((size_t)bh * N + r) * kD + 4 * lane);
      a[0] = bf16_to_f32(raw.x & 0xFFFF);
      a[1] = bf16_to_f32(raw.x >> 16);
      a[2] = bf16_to_f32(raw.y & 0xFFFF);
      a[3] = bf16_to_f32(raw.y >> 16);
    }
    if (ROTATE) {
      // half-width 1: (0,1), (2,3)
      float b0 = a[0] + a[1], b1 = a[0] - a[1], b2 = a[2] + a[3], b3 = a[2] - a[3];
      // half-width 2: (0,2), (1,3)
      a[0] = b0 + b2;
      a[1] = b1 + b3;
      a[2] = b0 - b2;
      a[3] = b1 - b3;
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {   // half-width 4m across lanes
        // lower lane: a + o; upper lane: o - a (one FMA with the lane's sign)
        const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float o = __shfl_xor_sync(0xffffffffu, a[e], m);
          a[e] = fmaf(a[e], sgn, o);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) a[e] *= sg[e];
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[i][e] = a[e];
      amax = fmaxf(amax, fabsf(a[e]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) warp_max[warp] = amax;
  __syncthreads();
  float bmax = warp_max[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) bmax = fmaxf(bmax, warp_max[w]);
  const float s = (bmax > 0.f) ? __fdiv_rn(bmax, 448.0f) : 1.0f;
  if (threadIdx.x == 0) scales[(size_t)bh * nblk + blk] = s;
  // x / s correctly rounded without a division per element: q = RN(x r) with r
  // the correctly rounded reciprocal, then one correction q + RN(x - q s) r
  // (the residual is exact by FMA) -- Markstein's final step, which yields the
  // correctly rounded binary32 quotient when r = RN(1 / s).  The sign is taken
  // from q so that x = -0 gives -0 (the correction would add +0).  A block
  // whose scale is subnormal (amax below 448 * 2^-126) divides instead: 1 / s
  // may then exceed the f32 range.  The branch is uniform over the block.
  const bool tiny = s < 1.17549435e-38f;   // 2^-126, the smallest normal f32
  const float rcp = tiny ? 0.0f : __frcp_rn(s);
  auto div_s = [&](float xv) {
    if (tiny) return __fdiv_rn(xv, s);
    const float q = xv * rcp;
    const float res = fmaf(-q, s, xv);
    return copysignf(fmaf(res, rcp, q), q);
  };

  uint32_t cw[16];   // codes of this lane's 4 columns, one word per row
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int r = blk * kRows + warp * 16 + i;
    cw[i] = pack_e4m3x4(div_s(v[i][0]), div_s(v[i][1]), div_s(v[i][2]), div_s(v[i][3]));
    if (!TRANSPOSE && r < N)
      *reinterpret_cast<uint32_t*>(x8 + ((size_t)bh * N + r) * kD + 4 * lane) = cw[i];
  }
  if (TRANSPOSE) {
    // Output row c (a head-dim column) holds the block's 128 keys, contiguous.
    // Each 4 x 4 byte block (4 rows x this lane's 4 columns) is transposed in
    // registers with byte permutes, so the lane owns 16 consecutive keys of
    // each of its columns: one 16-byte store per column.  Rows past N hold
    // code 0, the padding.
    uint32_t col[4][4];   // [column e][group g of 4 rows]
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t t0 = __byte_perm(cw[4 * g], cw[4 * g + 1], 0x5140);
      const uint32_t t1 = __byte_perm(cw[4 * g], cw[4 * g + 1], 0x7362);
      const uint32_t t2 = __byte_perm(cw[4 * g + 2], cw[4 * g + 3], 0x5140);
      const uint32_t t3 = __byte_perm(cw[4 * g + 2], cw[4 * g + 3], 0x7362);
      col[0][g] = __byte_perm(t0, t2, 0x5410);
      col[1][g] = __byte_perm(t0, t2, 0x7632);
      col[2][g] = __byte_perm(t1, t3, 0x5410);
      col[3][g] = __byte_perm(t1, t3, 0x7632);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint4* dst = reinterpret_cast<uint4*>(x8 + ((size_t)bh * kD + 4 * lane + e) * Npad +
                                            (size_t)blk * kRows + warp * 16);
      *dst = make_uint4(col[e][0], col[e][1], col[e][2], col[e][3]);
    }
  }
}

}  // namespace

cudaError_t launch_fp8_prep(const void* x, void* x8, float* scales, const signed char* signs,
                            int BH, int H, int N, int transpose_out, cudaStream_t stream) {
  const int nblk = (N + kRows - 1) / kRows;
  const int Npad = nblk * kRows;
  const dim3 grid(static_cast<unsigned>(BH) * nblk), block(256);
  const auto* xs = static_cast<const uint16_t*>(x);
  auto* xo = static_cast<uint8_t*>(x8);
  const auto* sg = reinterpret_cast<const int8_t*>(signs);
  if (signs && transpose_out)
    fp8_prep_kernel<true, true><<<grid, block, 0, stream>>>(xs, xo, scales, sg, H, N, nblk, Npad);
  else if (signs)
    fp8_prep_kernel<true, false><<<grid, block, 0, stream>>>(xs, xo, scales, sg, H, N, nblk, Npad);
  else if (transpose_out)
    fp8_prep_kernel<false, true><<<grid, block, 0, stream>>>(xs, xo, scales, sg, H, N, nblk, Npad);
  else
    fp8_prep_kernel<false, false><<<grid, block, 0, stream>>>(xs, xo, scales, sg, H, N, nblk, Npad);
  return cudaGetLastError();
}

}  // namespace gb300
