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
// Layout of the work: persistent CTAs (three per SM) walk the (batch*head,
// 128-row block) tiles.  A tile (128 rows x 128 bf16 = 32 KB) arrives by TMA
// into one of two shared-memory buffers per CTA, refilled as soon as its
// values are in registers, so the loads overlap the arithmetic and the stores.
// (Measured on the FP8 workload: three CTAs with two buffers beat two CTAs
// with three buffers, and 512-thread CTAs with four threads per row; the
// register cap of three CTAs costs a few spilled words.)
// Two threads share a row, 64 columns each: the butterfly stages of half-width
// 1..32 stay in registers (on packed f32 pairs), the stage of half-width 64
// exchanges with the partner lane.  The codes go straight from registers to
// memory: row-major [BH][N][128], or transposed [BH][128][Npad] for V (keys
// contiguous; rows past N are code 0, the padding), where 4 x 4 byte blocks
// transpose in registers and each warp store writes 128 consecutive keys.
// Every wait is bounded: a copy that never lands sets the status word and the
// CTA returns.
#include <cuda_runtime.h>

#include <cstdint>

#include "launchers.h"
#include "ptx.cuh"
#include "tmap.h"

namespace gb300 {

namespace {

constexpr int kRows = 128;
constexpr int kD = 128;
constexpr float kInvSqrtD = 0.08838834764831845f;   // 1 / sqrt(128)
constexpr int kThreads = 256;
constexpr int kTileBytes = kRows * kD * 2;           // bf16 input tile
constexpr int kStages = 2;                           // input buffers per CTA
constexpr int kSmemBytes = kStages * kTileBytes + 1024;
constexpr int kCtasPerSm = 3;
constexpr int kStatusTimeout = -5;
constexpr unsigned long long kTimeoutNs = 1000000000ull;   // 1 s per wait

// Status word of this translation unit (read back by attn_device_status).
__device__ int g_prep_status;

// Bounded wait on an mbarrier phase; false after kTimeoutNs (status set).
__device__ __forceinline__ bool prep_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kTimeoutNs) {
      atomicCAS(&g_prep_status, 0, kStatusTimeout);
      return false;
    }
  }
}

// Packed f32 pairs (the sm_100 family's f32x2 operations; add and fma in ptx.cuh).
__device__ __forceinline__ uint64_t f32x2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <bool ROTATE, bool TRANSPOSE>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    fp8_prep_kernel(const __grid_constant__ CUtensorMap tmX, uint8_t* __restrict__ x8,
                    float* __restrict__ scales, const int8_t* __restrict__ signs, int H, int N,
                    int nblk, int Npad, int ntiles) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kStages];
  __shared__ float warp_max[2][8];   // per iteration parity: a fast warp may write the next
  // 128-byte swizzled tiles need 1024-byte alignment.
  const uint32_t sIn = (smem_addr(smem_raw) + 1023u) & ~1023u;   // kStages 32 KB input tiles
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid >> 1;                          // row of the tile
  const int h = tid & 1;                           // column half: [64h, 64h + 64)

  if (tid == 0) {
    for (int b = 0; b < kStages; ++b) mbar_init(smem_addr(&full[b]), 1);
    fence_mbarrier_init();
  }
  __syncthreads();

  auto load_tile = [&](int t, int b) {
    const uint32_t bar = smem_addr(&full[b]);
    mbar_arrive_expect_tx(bar, kTileBytes);
    const int bh = t / nblk, blk = t - bh * nblk;
    tma_load_3d(sIn + b * kTileBytes, &tmX, bar, 0, blk * kRows, bh);
    tma_load_3d(sIn + b * kTileBytes + kTileBytes / 2, &tmX, bar, 64, blk * kRows, bh);
  };
  // This CTA's tiles are blockIdx.x + i * gridDim.x; the first kStages load at once.
  int issued = 0;   // tiles whose load this CTA has issued (thread 0)
  if (tid == 0)
    for (int k = 0; k < kStages && (int)blockIdx.x + k * (int)gridDim.x < ntiles; ++k, ++issued)
      load_tile(blockIdx.x + k * gridDim.x, k);

  int i = 0;
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
    const int b = i % kStages;
    const int bh = t / nblk, blk = t - bh * nblk;
    if (!__syncthreads_and(prep_wait(smem_addr(&full[b]), (i / kStages) & 1))) break;

    const uint32_t tile = sIn + b * kTileBytes;
    // Thread layouts.  Row-major output or a rotation: two threads per row r,
    // columns [64h, 64h + 64), held as 32 packed pairs.  Transposed output
    // without rotation (V): lane q holds keys 4q..4q+3 and warp w columns
    // [16w, 16w + 16), so that 4 x 4 blocks of codes transpose in registers.
    constexpr bool kRowMap = !TRANSPOSE || ROTATE;
    uint64_t p[32];
    if (kRowMap) {
      // Slab h of the tile; 16-byte chunk c of row r at position c ^ (r & 7).
      const uint32_t rowa = tile + h * (kTileBytes / 2) + r * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int4 w = ld_shared_v4_s32(rowa + ((c ^ (r & 7)) << 4));
        const uint32_t u[4] = {(uint32_t)w.x, (uint32_t)w.y, (uint32_t)w.z, (uint32_t)w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float x = bf16_lo(u[k]), y = bf16_hi(u[k]);
          // Rotation: the butterfly of half-width 1 on the word's two columns.
          p[4 * c + k] = ROTATE ? f32x2_pack(x + y, x - y) : f32x2_pack(x, y);
        }
      }
    } else {
      const int q = lane, wc = warp;   // keys 4q + k, columns 16 wc + j
      const uint32_t slab = tile + (wc >> 2) * (kTileBytes / 2);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int rr = 4 * q + k;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int c = 2 * (wc & 3) + c2;
          const int4 w = ld_shared_v4_s32(slab + rr * 128 + ((c ^ (rr & 7)) << 4));
          const uint32_t u[4] = {(uint32_t)w.x, (uint32_t)w.y, (uint32_t)w.z, (uint32_t)w.w};
#pragma unroll
          for (int m = 0; m < 4; ++m) p[8 * k + 4 * c2 + m] = f32x2_pack(bf16_lo(u[m]), bf16_hi(u[m]));
        }
      }
    }
    if (ROTATE) {
      // Butterflies of half-width 2..32 on packed column pairs (pair k holds
      // columns 2k, 2k + 1 of this thread's 64).
#pragma unroll
      for (int hp = 1; hp < 32; hp <<= 1) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          if (k & hp) continue;
          const uint64_t x = p[k], y = p[k + hp];
          p[k] = f32x2_add(x, y);
          p[k + hp] = f32x2_sub(x, y);
        }
      }
      // Half-width 64 across the partner lane (the lower half takes a + o, the
      // upper half o - a), then 1 / sqrt(128).  The column signs are applied
      // to the codes below: rounding and saturation are symmetric in sign.
      const uint64_t sgn2 = h ? f32x2_pack(-1.0f, -1.0f) : f32x2_pack(1.0f, 1.0f);
      const uint64_t c2 = f32x2_pack(kInvSqrtD, kInvSqrtD);
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        float x0, x1;
        f32x2_unpack(p[k], x0, x1);
        const float o0 = __shfl_xor_sync(0xffffffffu, x0, 1);
        const float o1 = __shfl_xor_sync(0xffffffffu, x1, 1);
        p[k] = f32x2_mul(f32x2_fma(p[k], sgn2, f32x2_pack(o0, o1)), c2);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      float x0, x1;
      f32x2_unpack(p[k], x0, x1);
      amax = fmaxf(amax, fmaxf(fabsf(x0), fabsf(x1)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) warp_max[i & 1][warp] = amax;
    __syncthreads();
    // Every thread has its values in registers: buffer b takes the tile
    // kStages ahead.
    if (tid == 0 && t + kStages * (int)gridDim.x < ntiles) {
      load_tile(t + kStages * gridDim.x, b);
      ++issued;
    }
    float bmax = warp_max[i & 1][0];
#pragma unroll
    for (int w = 1; w < 8; ++w) bmax = fmaxf(bmax, warp_max[i & 1][w]);
    const float s = (bmax > 0.f) ? __fdiv_rn(bmax, 448.0f) : 1.0f;
    if (tid == 0) scales[(size_t)bh * nblk + blk] = s;
    // x / s correctly rounded without a division per element: q = RN(x r) with
    // r the correctly rounded reciprocal, then one correction q + RN(x - q s) r
    // (the residual is exact by FMA) -- Markstein's final step, which yields
    // the correctly rounded binary32 quotient when r = RN(1 / s).  The sign is
    // taken from q so that x = -0 gives -0 (the correction would add +0).  A
    // block whose scale is subnormal (amax below 448 * 2^-126) divides
    // instead: 1 / s may then exceed the f32 range.  The branch is uniform.
    const bool tiny = s < 1.17549435e-38f;   // 2^-126, the smallest normal f32
    const float rcp = tiny ? 0.0f : __frcp_rn(s);
    const uint64_t rcp2 = f32x2_pack(rcp, rcp), ns2 = f32x2_pack(-s, -s);
    uint32_t cw[16];   // codes: pairs 2j, 2j + 1 (four consecutive columns) per word
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float y[4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint64_t x = p[2 * j + e];
        float x0, x1, q0, q1, r0, r1;
        f32x2_unpack(x, x0, x1);
        if (tiny) {
          r0 = __fdiv_rn(x0, s);
          r1 = __fdiv_rn(x1, s);
        } else {
          const uint64_t q = f32x2_mul(x, rcp2);
          const uint64_t res = f32x2_fma(q, ns2, x);
          f32x2_unpack(f32x2_fma(res, rcp2, q), r0, r1);
          f32x2_unpack(q, q0, q1);
          r0 = copysignf(r0, q0);
          r1 = copysignf(r1, q1);
        }
        y[2 * e] = r0;
        y[2 * e + 1] = r1;
      }
      cw[j] = pack_e4m3x4(y[0], y[1], y[2], y[3]);
    }
    if (ROTATE) {
      // Column signs (-1 has its top bit set) flip the codes' sign bits.
      // (4-byte loads: the signs are only required to be 4-byte aligned.)
      const uint32_t* sp = reinterpret_cast<const uint32_t*>(signs + (size_t)(bh % H) * kD + 64 * h);
#pragma unroll
      for (int j = 0; j < 16; ++j) cw[j] ^= __ldg(sp + j) & 0x80808080u;
    }
    if (!TRANSPOSE) {
      // Row r: bytes [64h, 64h + 64) of its 128 (rows past N are not written).
      const int row = blk * kRows + r;
      if (row < N) {
        uint4* dst = reinterpret_cast<uint4*>(x8 + ((size_t)bh * N + row) * kD + 64 * h);
#pragma unroll
        for (int m = 0; m < 4; ++m) dst[m] = make_uint4(cw[4 * m], cw[4 * m + 1], cw[4 * m + 2], cw[4 * m + 3]);
      }
    } else if (ROTATE) {
      // Transposed, row layout: output row d = 64h + j holds the tile's keys;
      // this thread writes key r of its 64 rows.  Rows past N are the padding:
      // code 0 (a rotated zero may carry a sign).
      const bool pad = blk * kRows + r >= N;
      uint8_t* dst = x8 + ((size_t)bh * kD + 64 * h) * Npad + (size_t)blk * kRows + r;
#pragma unroll
      for (int j = 0; j < 64; ++j)
        dst[(size_t)j * Npad] = pad ? 0 : static_cast<uint8_t>((cw[j >> 2] >> (8 * (j & 3))) & 0xFF);
    } else {
      // Transposed (V): cw[4k + w] holds key 4q + k, columns 16 wc + 4w .. + 3.
      // Each 4 x 4 byte block (4 keys x 4 columns) is transposed with byte
      // permutes into 4 words, one per column, bytes = the 4 keys; the warp's
      // 32 lanes then write 128 consecutive keys of output row d per store.
      // Keys past N are the padding: code 0.
      const int q = lane, wc = warp;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (blk * kRows + 4 * q + k >= N) {
#pragma unroll
          for (int w = 0; w < 4; ++w) cw[4 * k + w] = 0u;
        }
      uint32_t* dst = reinterpret_cast<uint32_t*>(x8 + ((size_t)bh * kD + 16 * wc) * Npad +
                                                  (size_t)blk * kRows + 4 * q);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t t0 = __byte_perm(cw[w], cw[4 + w], 0x5140);
        const uint32_t t1 = __byte_perm(cw[w], cw[4 + w], 0x7362);
        const uint32_t t2 = __byte_perm(cw[8 + w], cw[12 + w], 0x5140);
        const uint32_t t3 = __byte_perm(cw[8 + w], cw[12 + w], 0x7362);
        const uint32_t col[4] = {__byte_perm(t0, t2, 0x5410), __byte_perm(t0, t2, 0x7632),
                                 __byte_perm(t1, t3, 0x5410), __byte_perm(t1, t3, 0x7632)};
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[(size_t)(4 * w + e) * (Npad / 4)] = col[e];
      }
    }
  }
  // Every load this CTA started must have landed before it exits (only after
  // a wait gave up are any left: each issued tile's barrier phase, bounded).
  if (tid == 0)
    for (int k = i; k < issued; ++k) prep_wait(smem_addr(&full[k % kStages]), (k / kStages) & 1);
}

}  // namespace

int status_fp8_prep(bool clear) {
  int s = 0;
  if (cudaMemcpyFromSymbol(&s, g_prep_status, sizeof(int)) != cudaSuccess) return -4;
  if (clear && s != 0) {
    int z = 0;
    if (cudaMemcpyToSymbol(g_prep_status, &z, sizeof(int)) != cudaSuccess) return -4;
  }
  return s;
}

template <bool R, bool T>
static cudaError_t launch_one(const CUtensorMap& mx, uint8_t* x8, float* scales, const int8_t* signs,
                              int H, int N, int nblk, int Npad, int ntiles, int grid,
                              cudaStream_t stream) {
  auto kern = fp8_prep_kernel<R, T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, kSmemBytes, stream>>>(mx, x8, scales, signs, H, N, nblk, Npad, ntiles);
  return cudaGetLastError();
}

cudaError_t launch_fp8_prep(const void* x, void* x8, float* scales, const signed char* signs,
                            int BH, int H, int N, int transpose_out, int sms, cudaStream_t stream) {
  const int nblk = (N + kRows - 1) / kRows;
  const int Npad = nblk * kRows;
  const int ntiles = BH * nblk;
  CUtensorMap mx;
  if (!encode_map_3d(&mx, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, N, BH, 64, kRows))
    return cudaErrorInvalidValue;
  const int grid = ntiles < kCtasPerSm * sms ? ntiles : kCtasPerSm * sms;
  auto* xo = static_cast<uint8_t*>(x8);
  const auto* sg = reinterpret_cast<const int8_t*>(signs);
  if (signs && transpose_out)
    return launch_one<true, true>(mx, xo, scales, sg, H, N, nblk, Npad, ntiles, grid, stream);
  if (signs) return launch_one<true, false>(mx, xo, scales, sg, H, N, nblk, Npad, ntiles, grid, stream);
  if (transpose_out)
    return launch_one<false, true>(mx, xo, scales, sg, H, N, nblk, Npad, ntiles, grid, stream);
  return launch_one<false, false>(mx, xo, scales, sg, H, N, nblk, Npad, ntiles, grid, stream);
}

}  // namespace gb300
