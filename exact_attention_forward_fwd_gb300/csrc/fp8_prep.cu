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
// Layout of the work: persistent CTAs (two per SM) walk the (batch*head,
// 128-row block) tiles.  A tile (128 rows x 128 bf16 = 32 KB) arrives by TMA
// into one of two shared-memory buffers while the previous tile is worked on,
// so the loads of one tile overlap the arithmetic and the stores of the other.
// Two threads share a row, 64 columns each: the butterfly stages of half-width
// 1..32 stay in registers, the stage of half-width 64 exchanges with the
// partner lane.  The codes go out through a 16 KB shared-memory tile and a
// TMA store: row-major [BH][N][128] (rows past N clipped by the copy), or
// transposed [BH][128][Npad] for V (keys contiguous; rows past N are code 0,
// the padding).  Every wait is bounded: a copy that never lands sets the
// status word and the CTA returns.
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
constexpr int kOutBytes = kRows * kD;                // E4M3 output tile
constexpr int kSmemBytes = 2 * kTileBytes + kOutBytes + 1024;
constexpr int kCtasPerSm = 2;
constexpr int kStatusTimeout = -5;
constexpr unsigned long long kTimeoutNs = 1000000000ull;   // 1 s per wait

// Status word of this translation unit (read back by attn_device_status).
__device__ int g_prep_status;

__device__ __forceinline__ void st_shared_u8(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u8 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

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

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <bool ROTATE, bool TRANSPOSE>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    fp8_prep_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmOut,
                    float* __restrict__ scales, const int8_t* __restrict__ signs, int H, int N,
                    int nblk, int ntiles) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[2];
  __shared__ float warp_max[8];
  // 128-byte swizzled tiles need 1024-byte alignment.
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t sIn = base;                       // two 32 KB input tiles (two 16 KB slabs each)
  const uint32_t sOut = base + 2 * kTileBytes;     // 16 KB output tile
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid >> 1;                          // row of the tile
  const int h = tid & 1;                           // column half: [64h, 64h + 64)

  if (tid == 0) {
    mbar_init(smem_addr(&full[0]), 1);
    mbar_init(smem_addr(&full[1]), 1);
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
  int issued = 0;   // tiles whose load this CTA has issued (thread 0)
  if (tid == 0 && (int)blockIdx.x < ntiles) {
    load_tile(blockIdx.x, 0);
    issued = 1;
  }

  int i = 0;
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
    const int b = i & 1;
    const int bh = t / nblk, blk = t - bh * nblk;
    // The next tile into the other buffer: every thread finished reading it in
    // the previous iteration (the barrier before its store).
    if (tid == 0 && t + (int)gridDim.x < ntiles) {
      load_tile(t + gridDim.x, b ^ 1);
      ++issued;
    }
    if (!__syncthreads_and(prep_wait(smem_addr(&full[b]), (i >> 1) & 1))) break;

    // This thread's 64 values of row r (slab h of the tile; 16-byte chunk c of
    // a row at position c ^ (r & 7) in the 128-byte swizzle).
    float a[64];
    const uint32_t row = sIn + b * kTileBytes + h * (kTileBytes / 2) + r * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const int4 w = ld_shared_v4_s32(row + ((c ^ (r & 7)) << 4));
      const uint32_t u[4] = {(uint32_t)w.x, (uint32_t)w.y, (uint32_t)w.z, (uint32_t)w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        a[8 * c + 2 * k] = bf16_lo(u[k]);
        a[8 * c + 2 * k + 1] = bf16_hi(u[k]);
      }
    }
    if (ROTATE) {
      // Butterflies of half-width 1..32 within the 64 columns held here.
#pragma unroll
      for (int hw = 1; hw < 64; hw <<= 1) {
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          if (j & hw) continue;
          const float x = a[j], y = a[j + hw];
          a[j] = x + y;
          a[j + hw] = x - y;
        }
      }
      // Half-width 64 across the partner lane: the lower half takes a + o,
      // the upper half o - a (one FMA with the half's sign).
      const float sgn = h ? -1.0f : 1.0f;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const float o = __shfl_xor_sync(0xffffffffu, a[j], 1);
        a[j] = fmaf(a[j], sgn, o);
      }
      // Column signs of the head, times 1 / sqrt(128).
      // (4-byte loads: the signs are only required to be 4-byte aligned.)
      const int head = bh % H;
      const uint32_t* sp = reinterpret_cast<const uint32_t*>(signs + (size_t)head * kD + 64 * h);
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const uint32_t u = __ldg(sp + q);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          a[4 * q + k] *= static_cast<float>(static_cast<int8_t>((u >> (8 * k)) & 0xFF)) * kInvSqrtD;
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 64; ++j) amax = fmaxf(amax, fabsf(a[j]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) warp_max[warp] = amax;
    // The output tile is written again below: the previous tile's store must
    // have read it.
    if (tid == 0) bulk_wait_read_all();
    __syncthreads();
    float bmax = warp_max[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) bmax = fmaxf(bmax, warp_max[w]);
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
    auto div_s = [&](float xv) {
      if (tiny) return __fdiv_rn(xv, s);
      const float q = xv * rcp;
      const float res = fmaf(-q, s, xv);
      return copysignf(fmaf(res, rcp, q), q);
    };
    uint32_t cw[16];   // codes of columns 64h + 4j .. 64h + 4j + 3
    // Rows past N are the transposed output's padding: code 0 (their rotated
    // zeros may carry a sign, which would encode as -0).
    const bool pad = TRANSPOSE && blk * kRows + r >= N;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      cw[j] = pad ? 0u
                  : pack_e4m3x4(div_s(a[4 * j]), div_s(a[4 * j + 1]), div_s(a[4 * j + 2]), div_s(a[4 * j + 3]));
    if (!TRANSPOSE) {
      // Row r of the output tile, bytes [64h, 64h + 64), in the 128-byte swizzle.
#pragma unroll
      for (int m = 0; m < 4; ++m)
        st_shared_v4(sOut + r * 128 + (((4 * h + m) ^ (r & 7)) << 4), cw[4 * m], cw[4 * m + 1],
                     cw[4 * m + 2], cw[4 * m + 3]);
    } else {
      // Transposed: output row d = 64h + j holds the tile's 128 keys; key r is
      // byte r & 15 of 16-byte chunk r >> 4, at position (r >> 4) ^ (d & 7).
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int d = 64 * h + j;
        st_shared_u8(sOut + d * 128 + ((((r >> 4) ^ (d & 7))) << 4) + (r & 15),
                     (cw[j >> 2] >> (8 * (j & 3))) & 0xFF);
      }
    }
    fence_proxy_async_smem();   // generic-proxy writes -> the tensor store's reads
    __syncthreads();
    if (tid == 0) {
      if (TRANSPOSE)
        tma_store_3d(&tmOut, sOut, blk * kRows, 0, bh);
      else
        tma_store_3d(&tmOut, sOut, 0, blk * kRows, bh);
      bulk_commit();
    }
  }
  // Every copy this CTA started must be complete before it exits: the loads
  // (each issued tile's barrier phase) and the stores.
  if (tid == 0) {
    for (int k = i; k < issued; ++k) prep_wait(smem_addr(&full[k & 1]), (k >> 1) & 1);
    bulk_wait_all();
  }
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
static cudaError_t launch_one(const CUtensorMap& mx, const CUtensorMap& mo, float* scales,
                              const int8_t* signs, int H, int N, int nblk, int ntiles, int grid,
                              cudaStream_t stream) {
  auto kern = fp8_prep_kernel<R, T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, kSmemBytes, stream>>>(mx, mo, scales, signs, H, N, nblk, ntiles);
  return cudaGetLastError();
}

cudaError_t launch_fp8_prep(const void* x, void* x8, float* scales, const signed char* signs,
                            int BH, int H, int N, int transpose_out, int sms, cudaStream_t stream) {
  const int nblk = (N + kRows - 1) / kRows;
  const int Npad = nblk * kRows;
  const int ntiles = BH * nblk;
  CUtensorMap mx, mo;
  if (!encode_map_3d(&mx, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, N, BH, 64, kRows))
    return cudaErrorInvalidValue;
  const bool ok = transpose_out
                      ? encode_map_3d(&mo, x8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Npad, kD, BH, kRows, kD)
                      : encode_map_3d(&mo, x8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kD, N, BH, kD, kRows);
  if (!ok) return cudaErrorInvalidValue;
  const int grid = ntiles < kCtasPerSm * sms ? ntiles : kCtasPerSm * sms;
  const auto* sg = reinterpret_cast<const int8_t*>(signs);
  if (signs && transpose_out) return launch_one<true, true>(mx, mo, scales, sg, H, N, nblk, ntiles, grid, stream);
  if (signs) return launch_one<true, false>(mx, mo, scales, sg, H, N, nblk, ntiles, grid, stream);
  if (transpose_out) return launch_one<false, true>(mx, mo, scales, sg, H, N, nblk, ntiles, grid, stream);
  return launch_one<false, false>(mx, mo, scales, sg, H, N, nblk, ntiles, grid, stream);
}

}  // namespace gb300
