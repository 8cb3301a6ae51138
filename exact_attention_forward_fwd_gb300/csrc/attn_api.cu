// C-ABI boundary: argument validation, TMA descriptor encoding, persistent
// grid sizing and launch.  No allocation, no host synchronisation except in
// attn_device_status().
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <algorithm>
#include <functional>
#include <queue>
#include <vector>

#include "attn.h"
#include "attn_bwd.cuh"
#include "attn_kernel.cuh"
#include "launchers.h"
#include "tmap.h"

using namespace gb300;

namespace {

constexpr unsigned long long kDefaultTimeoutNs = 1000000000ull;   // 1 s per wait

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int units_for(int BH, int N) { return BH * ((N + 255) / 256); }

// sm_103 (GB300) only: the library carries sm_103a code and nothing else.
int device_check(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;
  *num_sms = sms;
  return ATTN_OK;
}

int check_shape(int B, int H, int N, float scale, int causal) {
  if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  // Unit index (BH * pairs) and the flat output offsets stay in range.
  if (static_cast<long long>(B) * H * ((N + 255) / 256) > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// The kernels' form of the caller's scale: a positive multiplier of the
// scores in base 2, |scale| * log2(e), plus two flags.  scale < 0: the score
// product negates its K operand (exact), so scale * q.k = |scale| * (q.(-k)).
// scale = 0: every visible score is replaced by 0 (the multiplier is then
// log2(e), which 0 leaves 0), while masked keys stay -inf.
void set_scale(float scale, float* scale_log2, int* neg, int* zero) {
  const double a = scale < 0.0f ? -static_cast<double>(scale) : static_cast<double>(scale);
  *neg = scale < 0.0f ? 1 : 0;
  *zero = scale == 0.0f ? 1 : 0;
  *scale_log2 = static_cast<float>((scale == 0.0f ? 1.0 : a) * 1.4426950408889634);
}

AttnParams base_params(void* o, float* lse, int B, int H, int H_kv, int N, float scale,
                       int causal, int window) {
  AttnParams p{};
  const int BH = B * H;
  p.o = o;
  p.lse = lse;
  p.N = N;
  p.BH = BH;
  p.H = H;
  p.group = H / H_kv;
  p.window = window;
  p.nkb = (N + 127) / 128;
  p.npairs = (N + 255) / 256;
  p.num_units = BH * p.npairs;
  p.causal = causal;
  set_scale(scale, &p.scale_log2, &p.neg_scale, &p.zero_scale);
  p.timeout_ns = kDefaultTimeoutNs;
  p.splits = 1;
  // Causal order: groups of heads whose K and V (bf16, head dim <= 128) take at
  // most 48 MiB, well inside the 129 MB L2 next to the Q and O streams.
  {
    const long long kv_bytes = 4LL * N * 128;
    long long hg = (48LL << 20) / (kv_bytes > 0 ? kv_bytes : 1);
    if (hg < 1) hg = 1;
    if (hg > BH) hg = BH;
    p.hgroup = static_cast<int>(hg);
  }
  return p;
}

constexpr int kMaxSplits = 64;
constexpr long long kUnitOverheadBlocks = 4;   // split-KV time model (measured)
constexpr double kBytesPerKeyBlock = 8.8e6;     // HBM bytes moved in one key block's time

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Bytes of the split-KV workspace: partial O, then partial lse (each 256-aligned).
size_t splitkv_bytes(int B, int H, int N, int d, int splits, size_t* lse_offset) {
  const size_t rows = static_cast<size_t>(splits) * static_cast<size_t>(B) * H * N;
  const size_t o_bytes = round256(rows * d * sizeof(float));
  if (lse_offset) *lse_offset = o_bytes;
  return o_bytes + round256(rows * sizeof(float));
}

// Split-KV arguments of run_bf16 (splits == 0: the plain path).
struct SplitArgs {
  int splits = 0;
  void* workspace = nullptr;
  size_t workspace_bytes = 0;
};

// Scratch of attn_fwd_splitkv_static: a file-scope device array (no allocation
// call anywhere).  In host code g_splitkv_scratch names a host-side shadow, not
// device memory, so the device address is looked up with cudaGetSymbolAddress,
// with the calling device current, and that address is what the kernels get.
// The lookup is repeated on every call (a host-side table lookup once the
// module is loaded): a cached address would outlive a context torn down and
// created again.  Every call shares the array; calls that overlap on the GPU
// race.
constexpr size_t kStaticScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_splitkv_scratch[kStaticScratchBytes];

int static_scratch(void** out) {
  void* a = nullptr;
  if (cudaGetSymbolAddress(&a, g_splitkv_scratch) != cudaSuccess || a == nullptr)
    return ATTN_ERR_CUDA;
  *out = a;
  return ATTN_OK;
}

int run_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int H_kv, int N, int d, float scale, int causal, int window, int dtype, int* status,
             unsigned long long timeout_ns, int skip_loads, cudaStream_t stream,
             const SplitArgs& split = SplitArgs()) {
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  int rc = check_shape(B, H, N, scale, causal);
  if (rc) return rc;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (window < 0 || (window > 0 && !causal)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  size_t lse_off = 0;
  if (split.splits != 0) {
    if (split.splits < 1 || split.splits > kMaxSplits || !split.workspace) return ATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * H * ((N + 255) / 256) * split.splits > 0x7fffffffLL)
      return ATTN_ERR_INVALID_ARG;
    if (split.workspace_bytes < splitkv_bytes(B, H, N, d, split.splits, &lse_off))
      return ATTN_ERR_INVALID_ARG;
  }
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      (lse && !aligned(lse, 4)) || (split.workspace && !aligned(split.workspace, 16)))
    return ATTN_ERR_ALIGNMENT;
  int sms = 0;
  if ((rc = device_check(&sms))) return rc;
  const int BH = B * H, BHk = B * H_kv;
  CUtensorMap mq, mk, mv, mo;
  const uint32_t box_inner = 64;   // 128-byte rows of the swizzle atom
  if (!encode_map_3d(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, box_inner, 128) ||
      !encode_map_3d(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BHk, box_inner, 128) ||
      !encode_map_3d(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BHk, box_inner, 128) ||
      !encode_map_3d(&mo, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, box_inner, 32))
    return ATTN_ERR_CUDA;
  AttnParams p = base_params(o, lse, B, H, H_kv, N, scale, causal, window);
  p.status = status;
  p.timeout_ns = timeout_ns;
  p.skip_load = skip_loads;
  if (split.splits != 0) {
    p.splits = split.splits;
    p.num_units *= split.splits;
    p.o_part = static_cast<float*>(split.workspace);
    p.lse_part = reinterpret_cast<float*>(static_cast<char*>(split.workspace) + lse_off);
    // The kernel stores partial O (f32 [splits * B * H][N][d]) through the O
    // map in 32-row x 32-column boxes; the merge writes O itself.
    if (!encode_map_3d(&mo, p.o_part, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d, N,
                       static_cast<uint64_t>(split.splits) * BH, 32, 32))
      return ATTN_ERR_CUDA;
  }
  const int grid = p.num_units < sms ? p.num_units : sms;
  cudaError_t e = (d == 64) ? launch_attn_bf16_d64(mq, mk, mv, mo, p, grid, stream)
                            : launch_attn_bf16_d128(mq, mk, mv, mo, p, grid, stream);
  if (e == cudaSuccess && split.splits != 0)
    e = launch_splitkv_merge(p.o_part, p.lse_part, o, lse, split.splits, BH, N, d, stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
             int d, float scale, int causal, int dtype, attn_stream_t stream) {
  return run_bf16(q, k, v, o, lse, B, H, H, N, d, scale, causal, 0, dtype, nullptr,
                  kDefaultTimeoutNs, 0, reinterpret_cast<cudaStream_t>(stream));
}

int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int H_kv, int N, int d, float scale, int causal, int window, int dtype,
                attn_stream_t stream) {
  return run_bf16(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, window, dtype, nullptr,
                  kDefaultTimeoutNs, 0, reinterpret_cast<cudaStream_t>(stream));
}

int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int H_kv, int N, int d, float scale, int causal, int window, int dtype,
                     int num_splits, void* workspace, size_t workspace_bytes,
                     attn_stream_t stream) {
  if (num_splits < 1 || num_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  SplitArgs split;
  split.splits = num_splits;
  split.workspace = workspace;
  split.workspace_bytes = workspace_bytes;
  return run_bf16(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, window, dtype, nullptr,
                  kDefaultTimeoutNs, 0, reinterpret_cast<cudaStream_t>(stream), split);
}

int attn_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int H, int H_kv, int N, int d, float scale, int causal,
                            int window, int dtype, int num_splits, attn_stream_t stream) {
  if (num_splits < 1 || num_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  SplitArgs split;
  split.splits = num_splits;
  const size_t need = attn_splitkv_workspace_bytes(B, H, N, d, num_splits);
  if (need != 0) {
    // Valid shape: the request must fit the static scratch.
    if (need > kStaticScratchBytes) return ATTN_ERR_INVALID_ARG;
    const int rc = static_scratch(&split.workspace);
    if (rc) return rc;
    split.workspace_bytes = kStaticScratchBytes;
  }
  // (need == 0: run_bf16 reports the argument error; it launches nothing.)
  return run_bf16(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, window, dtype, nullptr,
                  kDefaultTimeoutNs, 0, reinterpret_cast<cudaStream_t>(stream), split);
}

size_t attn_splitkv_workspace_bytes(int B, int H, int N, int d, int num_splits) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  if (num_splits < 1 || num_splits > kMaxSplits) return 0;
  return splitkv_bytes(B, H, N, d, num_splits, nullptr);
}

int attn_splitkv_default_splits(int B, int H, int N, int d, int causal, int num_sms) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128) || num_sms < 1) return 0;
  const long long bh = static_cast<long long>(B) * H;
  const long long npairs = (N + 255) / 256;
  if (bh * npairs >= num_sms) return 1;
  // Time model in key blocks.  The kernel's dynamic scheduler hands out units
  // in its own order (causal: longest pairs first, split ranges innermost);
  // each SM takes the next one when it is free, and a unit costs its key
  // blocks plus a fixed four (Q load, pipeline fill, epilogue) or one if its
  // range is empty.  S > 1 adds the merge: d floats per row and split
  // written and read again, one key block's time moving about 8.8 MB.
  const long long blocks = (N + 127) / 128;
  const long long cap = blocks < kMaxSplits ? blocks : kMaxSplits;
  const double merge_per_split = static_cast<double>(bh) * N * d * 8.0 / kBytesPerKeyBlock;
  auto model = [&](long long S) {
    std::priority_queue<long long, std::vector<long long>, std::greater<long long>> free_at;
    for (int m = 0; m < num_sms; ++m) free_at.push(0);
    long long span = 0;
    for (long long r = 0; r < npairs; ++r) {
      const long long pair = causal ? npairs - 1 - r : r;
      const long long nb = causal ? std::min(blocks, 2 * pair + 2) : blocks;
      for (long long h = 0; h < bh; ++h) {
        for (long long sp = 0; sp < S; ++sp) {
          const long long sz = (sp + 1) * nb / S - sp * nb / S;
          const long long t = free_at.top() + (sz > 0 ? sz + kUnitOverheadBlocks : 1);
          free_at.pop();
          free_at.push(t);
          span = std::max(span, t);
        }
      }
    }
    return static_cast<double>(span) + (S > 1 ? S * merge_per_split : 0.0);
  };
  long long best = 1;
  double best_t = model(1);
  for (long long S = 2; S <= cap; ++S) {
    const double t = model(S);
    if (t < best_t) {
      best = S;
      best_t = t;
    }
  }
  return static_cast<int>(best);
}

size_t attn_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  const size_t rows = static_cast<size_t>(B) * H * ((static_cast<size_t>(N) + 127) / 128 * 128);
  return 2 * round256(rows * sizeof(float));
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dO, void* dq, void* dk, void* dv, int B, int H, int H_kv, int N, int d,
             float scale, int causal, int window, void* workspace, size_t workspace_bytes,
             attn_stream_t stream) {
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !workspace)
    return ATTN_ERR_INVALID_ARG;
  int rc = check_shape(B, H, N, scale, causal);
  if (rc) return rc;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (window < 0 || (window > 0 && !causal)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (workspace_bytes < attn_bwd_workspace_bytes(B, H, N, d)) return ATTN_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * ((N + 127) / 128) > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dO, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(workspace, 16))
    return ATTN_ERR_ALIGNMENT;
  int sms = 0;
  if ((rc = device_check(&sms))) return rc;
  const int BH = B * H, BHk = B * H_kv;
  CUtensorMap mq, mk, mv, mdo;
  if (!encode_map_3d(&mq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, 64, 128) ||
      !encode_map_3d(&mk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BHk, 64, 128) ||
      !encode_map_3d(&mv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BHk, 64, 128) ||
      !encode_map_3d(&mdo, dO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, 64, 128))
    return ATTN_ERR_CUDA;
  BwdParams p{};
  p.N = N;
  p.Npad = (N + 127) / 128 * 128;
  const size_t half = round256(static_cast<size_t>(BH) * p.Npad * sizeof(float));
  float* lp = static_cast<float*>(workspace);
  float* dd = reinterpret_cast<float*>(static_cast<char*>(workspace) + half);
  p.lp = lp;
  p.dd = dd;
  p.q = static_cast<const uint16_t*>(q);
  p.dO = static_cast<const uint16_t*>(dO);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.BH = BH;
  p.BHk = BHk;
  p.H = H;
  p.Hk = H_kv;
  p.group = H / H_kv;
  p.window = window;
  p.causal = causal;
  p.nb = (N + 127) / 128;
  p.scale = scale;
  set_scale(scale, &p.scale_log2, &p.neg_scale, &p.zero_scale);
  p.timeout_ns = kDefaultTimeoutNs;
  cudaError_t e = launch_attn_bwd(d, mq, mk, mv, mdo, p, o, dO, lse, lp, dd, sms,
                                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_fwd_debug(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int N, int d, float scale, int causal, int* dev_status,
                   unsigned long long timeout_ns, int skip_loads, attn_stream_t stream) {
  if (!dev_status || !aligned(dev_status, 4) || timeout_ns == 0 || skip_loads < 0)
    return ATTN_ERR_INVALID_ARG;
  return run_bf16(q, k, v, o, lse, B, H, H, N, d, scale, causal, 0, ATTN_BF16, dev_status,
                  timeout_ns, skip_loads, reinterpret_cast<cudaStream_t>(stream));
}

int attn_fp8_prep(const void* x, void* x8, float* block_scale, const signed char* signs, int B,
                  int H, int N, int d, int transpose_out, attn_stream_t stream) {
  if (!x || !x8 || !block_scale) return ATTN_ERR_INVALID_ARG;
  int rc = check_shape(B, H, N, 1.0f, 0);
  if (rc) return rc;
  if (transpose_out != 0 && transpose_out != 1) return ATTN_ERR_INVALID_ARG;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(x8, 16) || !aligned(block_scale, 4) || (signs && !aligned(signs, 4)))
    return ATTN_ERR_ALIGNMENT;
  int sms = 0;
  if ((rc = device_check(&sms))) return rc;
  cudaError_t e = launch_fp8_prep(x, x8, block_scale, signs, B * H, H, N, transpose_out, sms,
                                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_fwd_fp8(const void* q8, const void* k8, const void* v8t, const float* q_scale,
                 const float* k_scale, const float* v_scale, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, attn_stream_t stream) {
  if (!q8 || !k8 || !v8t || !q_scale || !k_scale || !v_scale || !o) return ATTN_ERR_INVALID_ARG;
  int rc = check_shape(B, H, N, scale, causal);
  if (rc) return rc;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned(q8, 16) || !aligned(k8, 16) || !aligned(v8t, 16) || !aligned(o, 16) ||
      !aligned(q_scale, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4) ||
      (lse && !aligned(lse, 4)))
    return ATTN_ERR_ALIGNMENT;
  int sms = 0;
  if ((rc = device_check(&sms))) return rc;
  const int BH = B * H;
  const int Npad = ((N + 127) / 128) * 128;
  CUtensorMap mq, mk, mv, mo;
  if (!encode_map_3d(&mq, q8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d, N, BH, 128, 128) ||
      !encode_map_3d(&mk, k8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d, N, BH, 128, 128) ||
      !encode_map_3d(&mv, v8t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Npad, d, BH, 128, 128) ||
      !encode_map_3d(&mo, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, N, BH, 64, 32))
    return ATTN_ERR_CUDA;
  AttnParams p = base_params(o, lse, B, H, H, N, scale, causal, 0);
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  const int grid = p.num_units < sms ? p.num_units : sms;
  cudaError_t e = launch_attn_fp8_d128(mq, mk, mv, mo, p, grid, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_device_status(int clear) {
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  int out = ATTN_OK;
  const int s[5] = {status_attn_bf16_d64(clear != 0), status_attn_bf16_d128(clear != 0),
                    status_attn_fp8_d128(clear != 0), status_attn_bwd(clear != 0),
                    status_fp8_prep(clear != 0)};
  for (int i = 0; i < 5; ++i)
    if (s[i] != 0 && out == ATTN_OK) out = s[i];
  return out;
}

int attn_num_units(int B, int H, int N) {
  if (B < 1 || H < 1 || N < 1) return 0;
  return units_for(B * H, N);
}

int attn_grid_size(int B, int H, int N, int num_sms) {
  const int u = attn_num_units(B, H, N);
  if (num_sms < 1) return 0;
  return u < num_sms ? u : num_sms;
}

const char* attn_status_str(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported head dim, dtype or device";
    case ATTN_ERR_ALIGNMENT: return "tensor base address not 16-byte aligned";
    case ATTN_ERR_CUDA: return "CUDA runtime or driver call failed";
    case ATTN_ERR_TIMEOUT: return "a pipeline wait inside the kernel ran out of time";
    default: return "unknown status";
  }
}

}  // extern "C"
