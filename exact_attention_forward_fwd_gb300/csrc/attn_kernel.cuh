// Fused exact attention forward for sm_103a: O = softmax(scale * Q K^T [+causal]) V
// and lse = log sum exp(scale * Q K^T) per row, without writing the N x N
// score matrix anywhere.
//
// Method (as described on "Learn: The Memory Wall & FlashAttention", section
// 5.1, and "4.3 FlashAttention 2 & 3", sections "Edit 1/2/3" and
// "FlashAttention-3: exploiting Hopper"):
//   * tiled over query blocks, streaming over key/value blocks;
//   * online softmax: running max m, running denominator l, unnormalised
//     accumulator O~ rescaled by alpha = exp(m_old - m_new), one final O~ / l;
//   * causal: key blocks strictly in the future are skipped, the diagonal
//     blocks are masked element-wise (key > query -> -inf);
//   * producer/consumer warp specialisation over a shared-memory ring with
//     mbarriers; the score MMA of the next block overlaps the softmax of the
//     current one.
//
// Blackwell mapping (this file's own design):
//   * one persistent CTA per SM; a work unit is (batch*head, pair of 128-row
//     query tiles); both tiles share every K/V block loaded;
//   * warps 0-3 / 4-7: softmax of tile 0 / tile 1, one thread per query row
//     (224 registers each: warps 8-11 hand theirs over with setmaxnreg),
//     reading S from tensor memory (TMEM) and writing P back over it;
//   * warp 8: TMA loads of Q (once per unit) and of K, V blocks into the ring;
//   * warps 10, 11: no role (they complete the third warpgroup);
//   * warp 9: allocates TMEM and issues every tcgen05.mma (the warp runs its
//     loop converged, one elected lane issues):
//       S_t = Q_t K_j^T  (SS, both operands K-major in shared memory)
//       O_t += P_t V_j   (TS, P from TMEM, V from shared memory; FP8: SS)
//     bf16 at d = 128 in the order PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), ...
//     (P over S: the tensor pipe has the other tile's work while one tile's
//     softmax runs); FP8 issues S_t(j+1) as soon as the softmax has read
//     S_t(j) (P in shared memory); bf16 at d = 64 does the same for S's
//     first 112 keys and issues the rest once the P.V steps over P's last
//     32 keys, stored over S's last 16 columns and signalled first, are in;
//   * TMEM columns: S/P tile 0 [0,128), S/P tile 1 [128,256), O tile 0
//     [256,256+D), O tile 1 [256+D, 256+2D); at d = 64 O_t has 80 columns
//     (the last 16 accumulate l~: P.V runs with N = 80 against V and a block
//     of ones) and P of keys [0, 96) has [416 + 48 t, +48);
//   * scale folded into exp2: p = 2^(s * scale*log2(e) - m), m kept in the
//     same base-2 units; a negative scale runs as s' = Q (-K)^T with |scale|
//     (the MMA negates its B operand, exactly), so the multiplier the softmax
//     sees is always positive; scale = 0 replaces every visible score by 0;
//   * conditional rescaling: the reference max used for the exponentials is
//     only moved (and O~, l rescaled) when the block's values against it grow
//     too large.  Numerator and denominator always share the same reference,
//     so the result stays exact.  The exponentials are taken against the
//     current reference and the block's sum of p decides: a sum of at most
//     2^32 bounds every p by 2^32 and the pass stands (f32 O~ and l then stay
//     below 2^56 times max|V| for any sequence length); otherwise (rare after
//     a unit's first block, even on rows as sharp as scores with a spread of
//     10 in base 2) the reference moves to the block's max and the block,
//     still in registers, is taken again.  No exponential waits for a row
//     max.  The FP8 path takes the block's max first instead and moves the
//     reference only when that max exceeds it by more than 8, so p <= 2^8
//     (P must fit E4M3, whose largest value is 448).
//   * because every tcgen05.commit tracks all earlier MMAs of the issuing
//     thread, in the d = 128 order the arrival of S_t(j) also proves
//     O_t += P_t(j-1) V(j-1) is complete: a rescale of O~ right after waiting
//     for S_t(j) is race-free.  The other orders wait for the commit after
//     the previous P.V (p_free) and, at d = 64 once P's last keys are in,
//     for the commit after their P.V steps (pt_done).
//
// FP8 variant (E4M3 operands, f32 accumulation): per-128-row block scales of
// Q, K, V ("FlashAttention-3: How Warp Specialization ...", section 4); the
// score scale of block j is folded into the exp2 factor, P is quantised to
// E4M3 as p * 1.75 * s_V(j) / max_j s_V(j) (p <= 2^8, so P <= 448, E4M3's
// largest finite value), which folds V's per-block scale into P, and the
// epilogue divides by 1.75 * l / max s_V.
// V arrives transposed ([d][N], keys contiguous) so both MMAs read K-major
// operands.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "ptx.cuh"

namespace gb300 {

enum : int { kStatusOk = 0, kStatusTimeout = -5 };

struct AttnParams {
  void* o;               // bf16 [BH][N][D]
  float* lse;            // fp32 [BH][N] or null
  const float* q_scale;  // FP8 only: [BH][nqb]
  const float* k_scale;  // FP8 only: [BH][nkb]
  const float* v_scale;  // FP8 only: [BH][nkb]
  int* status;           // device status word, or null for the library's own word
  int N;                 // sequence length (queries == keys)
  int BH;                // batch * query heads
  int H;                 // query heads
  int group;             // query heads per KV head (H / H_kv)
  int window;            // > 0: causal sliding window of this many keys; 0: none
  int nkb;               // ceil(N / 128): key blocks (and 128-row query tiles)
  int npairs;            // ceil(N / 256): query-tile pairs per head
  int num_units;         // BH * npairs
  int causal;
  float scale_log2;      // |scale| * log2(e) (log2(e) when scale = 0)
  int neg_scale;         // scale < 0: the score product negates its K operand, so the
                         // softmax always sees a positive multiplier
  int zero_scale;        // scale = 0: every visible score is 0 (uniform weights)
  unsigned long long timeout_ns;
  int skip_load;         // test hook: when > 0, the load warp stops after that many K/V loads
  // Split-KV mode (o_part != null): every (head, query-tile pair) is split into
  // `splits` contiguous key ranges, each a unit of its own, and each unit writes
  // its partial result: O normalised by its own denominator, and its own
  // logsumexp.  A merge kernel combines them.
  int hgroup;            // causal order: heads per group (K/V of a group stay in L2)
  int* sched;            // unit counter for dynamic scheduling (zeroed before launch), or null
  int splits;            // key ranges per (head, pair); 1 without split-KV
  float* o_part;         // [splits][BH][N][D] fp32, or null
  float* lse_part;       // [splits][BH][N] fp32 (natural log), or null
};

template <int D, bool FP8>
struct KCfg {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  static_assert(!FP8 || D == 128, "FP8 path: head dim 128");
  static constexpr int kRowBytes = FP8 ? D : 2 * D;        // one Q/K row in bytes
  static constexpr int kSlabs = kRowBytes / 128;           // 128-byte column slabs per tile
  static constexpr int kTileBytes = 128 * kRowBytes;       // 128-row tile (V / V^T tile the same)
  static constexpr int kStages = (kTileBytes == 32768) ? 4 : 8;
  static constexpr int kOStageBytes = D == 128 ? 16384 : 0;   // per tile: 4 warps x 32 rows x 64 bf16 of O
  // bf16 at d = 64: the normaliser l~ (the sum of P as rounded to bf16) comes
  // from the tensor core instead of two bf16 additions per key pair in the
  // softmax.  P.V runs with N = D + 16: B is the V tile and, one operand atom
  // along N further (the descriptor's 16 KB leading-dimension step), a block
  // of bf16 ones, so columns [D, D + 16) of the tile's accumulator collect
  // sum_k P[r][k] -- every one of them l~ -- in the same instructions as O.
  static constexpr bool kLFused = !FP8 && D == 64;
  static constexpr int kOCols = kLFused ? D + 16 : D;     // TMEM columns of O_t (and l~)
  // Ring: K tiles take the even slots and V tiles the odd ones (items
  // alternate K, V and every unit starts on an even item); with kLFused each
  // V slot is followed by its 16 KB of ones.
  static constexpr int kPairBytes = (kLFused ? 3 : 2) * kTileBytes;
  static constexpr int kRingBytes = kStages / 2 * kPairBytes;
  __host__ __device__ static constexpr uint32_t slot_off(uint32_t s) {
    return kLFused ? (s >> 1) * kPairBytes + (s & 1) * kTileBytes : s * kTileBytes;
  }
  static constexpr int kSmemBytes = 2 * kTileBytes + kRingBytes + 2 * kOStageBytes + 1024;
  static constexpr uint32_t kTmemCols = 512;
  // 12 warps: two softmax warpgroups (warps 0-7), then load (8), MMA (9) and
  // two idle warps (10, 11) that complete the third warpgroup so that it can
  // hand its registers to the softmax warpgroups.
  static constexpr int kThreads = 384;
  static constexpr int kLaunchRegs = 168;                 // 65536 / 384, rounded down to 8
  static constexpr uint32_t kRegsSoftmax = 224;
  static constexpr uint32_t kRegsOther = 56;
  static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsOther <= kThreads * kLaunchRegs,
                "register split exceeds the block's pool");
  static constexpr float kSumLimit = 4294967296.0f;       // bf16: 2^32, bound on a block's sum of p
  static constexpr float kTauLog2 = 8.0f;                 // FP8: move the reference when a block max exceeds it by more
  static constexpr float kPScale = 1.75f;                 // FP8: P' = p * kPScale * s_V(j) / max s_V <= 256 * 1.75 = 448
  // Causal: tile 0 skips a pair's last key block (wholly above its rows).  bf16
  // at d = 128 only: the FP8 and d = 64 kernels measured slower with the
  // extra branches in their issue loop than the work saved (2 %; at d = 64,
  // in the coupled order with the l~ product, 1.3 %).
  static constexpr bool kSkipDiag = !FP8 && D == 128;
  // FP8: P (one byte per key, 128 bytes per row) goes to shared memory -- the
  // region that stages O in the epilogue -- instead of over S in tensor
  // memory, so a tile's next S product can start as soon as its softmax has
  // read S, and P.V reads P as an SS operand.
  static constexpr bool kPSmem = FP8;
  // bf16 at d = 64: P of keys [0, 96) has TMEM columns of its own (tile t at
  // [kPCol + 48 t, +48): the 96 columns left after S, O and l~), and P of
  // keys [96, 128) goes over S's last 16 columns.  The softmax computes and
  // signals those last keys first (p_ready[2 t + 1]); S is issued in two
  // parts: keys [0, 112) as soon as the softmax has read the tile's previous
  // S, and keys [112, 128) right after the P.V steps that read P's last keys,
  // so S_t(j+1) is complete while the softmax still works on block j.
  static constexpr bool kPSep = !FP8 && D == 64;
  static constexpr int kSMainKeys = 112;                  // keys of S's first part
  static constexpr bool kDecoupled = kPSmem;
  // Tile t's P-ready barrier is p_ready[t * kPReadyStride].  Neither the
  // spacing nor the spare word between the bf16 barriers carries a signal;
  // both are what measured fastest (same-box A/B, three repeats): FP8 1.6 %
  // faster with its two barriers adjacent, bf16 d = 128 1 % faster with them
  // 16 bytes apart and the word between them initialised as a barrier too.
  static constexpr int kPReadyStride = FP8 ? 1 : 2;
  static constexpr uint32_t kPCol = 256 + 2 * kOCols;
  static constexpr int kSKSteps = FP8 ? D / 32 : D / 16;  // k-steps of S = Q K^T
  static constexpr int kPVSteps = FP8 ? 4 : 8;            // k-steps of O += P V (128 keys)
  static constexpr uint32_t kIdescS =
      make_idesc(128, 128, FP8 ? 0u : 1u, FP8 ? 0u : 1u, false, false);
  static constexpr uint32_t kIdescPV =
      make_idesc(128, kOCols, FP8 ? 0u : 1u, FP8 ? 0u : 1u, false, !FP8);
  static constexpr uint32_t kIdescSMain = make_idesc(128, kSMainKeys, 1u, 1u, false, false);
  static constexpr uint32_t kIdescSTail = make_idesc(128, 128 - kSMainKeys, 1u, 1u, false, false);
};

struct SmemCtl {
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t s_full[2];
  uint64_t p_ready[4];      // tile t at [t * kPReadyStride]; d = 64: P's last 32 keys at
                            // [t * kPReadyStride + 1]
  uint64_t s_free[2];       // FP8, d = 64: the tile's S has been read (its TMEM columns
                            // may be overwritten)
  uint64_t p_free[2];       // FP8, d = 64: the tile's P.V is done (its P buffer may be
                            // overwritten, O_t rescaled)
  uint64_t o_final[2];
  uint64_t drain;
  uint64_t unit_full[4];    // ring of work-unit indices handed out by the load warp
  uint64_t unit_empty[4];
  int4 unit_ring[4][2];     // decoded work units (Unit fields; valid = 0 ends)
  uint32_t tmem_base;
  int abort_flag;
  uint64_t pt_done[2];      // bf16 d = 64: the tile's P.V over its last 32 keys is done
};

// Status word of launches that pass no status pointer (one per translation
// unit; read back by the host through cudaMemcpyFromSymbol).
static __device__ int g_attn_status;

struct WaitCtx {
  int* abort_flag;   // this CTA's abort flag (shared memory)
  int* status;
  unsigned long long timeout_ns;
};

// Bounded wait on an mbarrier phase.  Returns false if the CTA was told to
// abort or the limit ran out (which sets the abort flag and the status word).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx& wc,
                                             bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (honour_abort && *reinterpret_cast<volatile int*>(wc.abort_flag)) return false;
    if (global_timer_ns() - t0 > wc.timeout_ns) {
      *reinterpret_cast<volatile int*>(wc.abort_flag) = 1;
      atomicCAS(wc.status, kStatusOk, kStatusTimeout);
      return false;
    }
  }
}

struct Unit {
  int bh, bhk, pair, j0, nblocks;   // query head, KV head, pair, first key block, blocks
  int split;                        // key range index (split-KV), 0 otherwise
  bool skip0;                       // causal: the last block lies wholly above tile 0's rows
};

// Work unit u -> (head, query-tile pair, key blocks to visit).  Non-causal:
// consecutive units walk the pairs of one head (K/V of a head stay hot in L2).
// Causal: longest first within groups of `hgroup` heads -- the group's last
// pairs, then the ones before, ...; the groups one after the other, so that
// only one group's K/V (sized by the host to fit L2) is live at a time.  The
// units are handed out dynamically, so the short units at the end of a group
// do not unbalance the SMs.  A sliding window also skips the key blocks
// entirely before the window of the pair's first row.  Query head h of batch b reads KV head h / group.  With
// split-KV, consecutive units are the key ranges of one pair: range s takes
// blocks [s*nb/S, (s+1)*nb/S) of the pair's nb visible blocks (empty when
// nb < S; such a unit only writes an empty partial result).
__device__ __forceinline__ Unit unit_of(int u, const AttnParams& p) {
  Unit w;
  const int S = p.splits > 1 ? p.splits : 1;
  w.split = 0;
  if (S > 1) {
    w.split = u % S;
    u /= S;
  }
  if (p.causal) {
    const int HG = p.hgroup > 0 ? p.hgroup : p.BH;
    const int per_group = HG * p.npairs;
    const int g = u / per_group;
    const int v = u - g * per_group;
    const int hg = min(HG, p.BH - g * HG);   // heads in this group (the last may have fewer)
    const int r = v / hg;
    w.bh = g * HG + (v - r * hg);
    w.pair = p.npairs - 1 - r;
    const int j_hi = min(p.nkb - 1, 2 * w.pair + 1);
    w.j0 = p.window > 0 ? max(0, w.pair * 256 - p.window + 1) / 128 : 0;
    w.nblocks = j_hi - w.j0 + 1;
  } else {
    w.bh = u / p.npairs;
    w.pair = u - w.bh * p.npairs;
    w.j0 = 0;
    w.nblocks = p.nkb;
  }
  if (S > 1) {
    const int nb = w.nblocks;
    const int b0 = (w.split * nb) / S, b1 = ((w.split + 1) * nb) / S;
    w.j0 += b0;
    w.nblocks = b1 - b0;
  }
  // Causal (one key range): the pair's last block 2·pair+1 holds keys
  // 256·pair+128 on, all above the rows of tile 0, which skips it.
  w.skip0 = p.causal && S == 1 && w.nblocks >= 2 && w.j0 + w.nblocks - 1 == 2 * w.pair + 1;
  const int b = w.bh / p.H;
  const int h = w.bh - b * p.H;
  w.bhk = b * (p.H / p.group) + h / p.group;
  return w;
}

template <int D, bool FP8>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const AttnParams p) {
  using C = KCfg<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ SmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_addr(smem);                         // Q tile 0, Q tile 1
  const uint32_t sKV = sQ + 2 * C::kTileBytes;                 // ring of K / V tiles
  const uint32_t sO = sKV + C::kRingBytes;                     // O staging (d = 128), 4 KB per softmax warp
                                                               // (FP8: also P, 128 bytes per row)
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  auto bar = [&](uint64_t& b) { return smem_addr(&b); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(ctl.kv_full[s]), 1);
      mbar_init(bar(ctl.kv_empty[s]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(ctl.q_full[t]), 1);
      mbar_init(bar(ctl.q_empty[t]), 1);
      mbar_init(bar(ctl.s_full[t]), 1);
      // FP8: one arrival per softmax warp of the tile (measured +1 %); bf16: one
      // per thread (a warp-level arrival after __syncwarp measured -2 % there).
      mbar_init(bar(ctl.p_ready[t * C::kPReadyStride]), FP8 ? 4 : 128);
      if (!FP8) mbar_init(bar(ctl.p_ready[t * C::kPReadyStride + 1]), 128);
      mbar_init(bar(ctl.o_final[t]), 1);
      mbar_init(bar(ctl.s_free[t]), 4);
      mbar_init(bar(ctl.p_free[t]), 1);
    }
    mbar_init(bar(ctl.drain), 1);
    if constexpr (C::kPSep)
      for (int t = 0; t < 2; ++t) mbar_init(bar(ctl.pt_done[t]), 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(bar(ctl.unit_full[s]), 1);
      mbar_init(bar(ctl.unit_empty[s]), 9);   // the MMA warp and the 8 softmax warps
    }
    ctl.abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  if constexpr (C::kLFused) {
    // The ones beside each V slot (bf16 1.0 = 0x3F80 in every element: with
    // equal elements the swizzle needs no care), written once.
    constexpr int kChunks = C::kStages / 2 * C::kTileBytes / 16;
    for (int i = threadIdx.x; i < kChunks; i += C::kThreads) {
      const int pr = i / (C::kTileBytes / 16), c = i % (C::kTileBytes / 16);
      st_shared_v4(sKV + C::slot_off(2 * pr + 1) + C::kTileBytes + 16 * c, 0x3F803F80u, 0x3F803F80u,
                   0x3F803F80u, 0x3F803F80u);
    }
    fence_proxy_async_smem();   // generic-proxy writes -> the MMA's operand reads
  }
  if (warp == 9) {
    tmem_alloc(smem_addr(&ctl.tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const WaitCtx wc{&ctl.abort_flag, p.status ? p.status : &g_attn_status, p.timeout_ns};

  // Work units: the load warp takes the next index (atomic counter, or the
  // static stride without one), decodes it once (unit_of divides by runtime
  // values: hundreds of cycles of latency that every role would otherwise pay
  // at each unit boundary) and passes the decoded unit through a 4-entry
  // ring; an entry with valid = 0 ends the kernel.
  auto publish_unit = [&](uint32_t k, bool& ok, Unit& w) -> int {
    int u = p.sched ? atomicAdd(p.sched, 1) : static_cast<int>(blockIdx.x + k * gridDim.x);
    if (u >= p.num_units) u = -1;
    if (u >= 0) w = unit_of(u, p);
    const uint32_t slot = k & 3;
    if (k >= 4 && !(ok = wait_bounded(bar(ctl.unit_empty[slot]), ((k >> 2) - 1) & 1, wc))) return -1;
    ctl.unit_ring[slot][0] = make_int4(w.bh, w.bhk, w.pair, w.j0);
    ctl.unit_ring[slot][1] = make_int4(w.nblocks, w.split, w.skip0 ? 1 : 0, u >= 0 ? 1 : 0);
    mbar_arrive(bar(ctl.unit_full[slot]));
    return u;
  };
  // Consumer side (a whole warp; lane 0 frees the slot).  Returns false at the end.
  auto take_unit = [&](uint32_t k, bool& ok, Unit& w) -> bool {
    const uint32_t slot = k & 3;
    ok = wait_bounded(bar(ctl.unit_full[slot]), (k >> 2) & 1, wc);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return false;
    const int4 a = ld_shared_v4_s32(smem_addr(&ctl.unit_ring[slot][0]));
    const int4 b = ld_shared_v4_s32(smem_addr(&ctl.unit_ring[slot][1]));
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(ctl.unit_empty[slot]));
    w.bh = a.x;
    w.bhk = a.y;
    w.pair = a.z;
    w.j0 = a.w;
    w.nblocks = b.x;
    w.split = b.y;
    w.skip0 = b.z != 0;
    return b.w != 0;
  };

  // Each role sets its warpgroup's register budget first (warps 8-11 give
  // registers up, warps 0-7 take them).
  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    regs_dec<C::kRegsOther>();
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      const uint64_t pol_kv = l2_policy_evict_last();
      const uint64_t pol_q = l2_policy_evict_first();
      uint32_t item = 0;        // K/V ring items issued
      uint32_t uit = 0;         // units started
      uint32_t qn[2] = {0, 0};  // Q tiles issued per tile slot
      bool ok = true;
      int loads = 0;
      for (uint32_t k = 0; ok; ++k) {
        Unit w{};
        const int u = publish_unit(k, ok, w);
        if (u < 0) break;
        if (w.nblocks == 0) continue;   // empty key range (split-KV)
        // No L2 prefetch of the unit's Q tiles or first key blocks here: the
        // prefetch instructions (a dozen, issued at unit boundaries) delayed
        // the Q loads below by more than the prefetch saved (measured: 1-2.6 %
        // faster on every bf16 workload without them).
        for (int t = 0; t < 2 && ok; ++t) {
          if (uit > 0) ok = wait_bounded(bar(ctl.q_empty[t]), (uit - 1) & 1, wc);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(ctl.q_full[t]), C::kTileBytes);
          ++qn[t];
          const int row0 = w.pair * 256 + t * 128;
          for (int s = 0; s < C::kSlabs; ++s)
            tma_load_3d_hint(sQ + t * C::kTileBytes + s * 16384, &tmQ, bar(ctl.q_full[t]),
                             s * (FP8 ? 128 : 64), row0, w.bh, pol_q);
        }
        for (int jj = 0; jj < w.nblocks && ok; ++jj) {
          const int j = w.j0 + jj;   // key block
          for (int kv = 0; kv < 2 && ok; ++kv, ++item) {
            if (p.skip_load > 0 && loads >= p.skip_load) break;   // test hook only
            const uint32_t slot = item % C::kStages;
            const uint32_t ph = (item / C::kStages) & 1;
            ok = wait_bounded(bar(ctl.kv_empty[slot]), ph ^ 1, wc);
            if (!ok) break;
            const uint32_t dst = sKV + C::slot_off(slot);
            mbar_arrive_expect_tx(bar(ctl.kv_full[slot]), C::kTileBytes);
            if (kv == 0) {
              for (int s = 0; s < C::kSlabs; ++s)
                tma_load_3d_hint(dst + s * 16384, &tmK, bar(ctl.kv_full[slot]),
                                 s * (FP8 ? 128 : 64), j * 128, w.bhk, pol_kv);
            } else if (FP8) {
              // V^T [BH][D][Npad]: one 128-key x D tile
              tma_load_3d_hint(dst, &tmV, bar(ctl.kv_full[slot]), j * 128, 0, w.bhk, pol_kv);
            } else {
              for (int s = 0; s < C::kSlabs; ++s)
                tma_load_3d_hint(dst + s * 16384, &tmV, bar(ctl.kv_full[slot]), s * 64, j * 128,
                                 w.bhk, pol_kv);
            }
            ++loads;
          }
        }
        ++uit;
      }
      // Let every copy this warp started land before the CTA can exit.
      const uint32_t issued = item;
      for (uint32_t s = 0; s < (uint32_t)C::kStages && s < issued; ++s) {
        const uint32_t last = s + ((issued - 1 - s) / C::kStages) * C::kStages;
        wait_bounded(bar(ctl.kv_full[s]), (last / C::kStages) & 1, wc, false);
      }
      for (int t = 0; t < 2; ++t)
        if (qn[t] > 0) wait_bounded(bar(ctl.q_full[t]), (qn[t] - 1) & 1, wc, false);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    regs_dec<C::kRegsOther>();
    // The whole warp runs this loop converged; each MMA and commit is issued by
    // one elected lane (the *_w forms), every wait is taken by all lanes.
    {
      uint32_t item = 0, uit = 0, pr[2] = {0, 0};
      bool ok = true;
      auto wait_w = [&](uint64_t& b, uint32_t parity) {
        return __all_sync(0xffffffffu, wait_bounded(bar(b), parity, wc));
      };
      // Descriptor bases, computed once: K-major Q and K tiles (and FP8 V^T),
      // MN-major bf16 V tiles.  A k-step adds its offset in 16-byte units to
      // the address field (tiles lie below 256 KB, so it never carries).
      constexpr uint64_t kTileUnits = C::kTileBytes >> 4;
      const uint64_t dQ = make_smem_desc(sQ, 16, 1024, kSwizzle128B);
      const uint64_t dK = make_smem_desc(sKV, 16, 1024, kSwizzle128B);
      const uint64_t dV = make_smem_desc(sKV, FP8 ? 16 : 16384, 1024, kSwizzle128B);
      const uint32_t idesc_s = C::kIdescS | (p.neg_scale ? kIdescNegateB : 0u);
      auto s_mma = [&](int t, uint32_t kslot) {
        const uint64_t da = dQ + t * kTileUnits;
        const uint64_t db = dK + (C::slot_off(kslot) >> 4);
#pragma unroll
        for (int g = 0; g < C::kSKSteps / 4; ++g) {
          const uint64_t o = FP8 ? 0 : g * 1024;   // next 128-byte column slab (bf16, d = 128)
          mma_ss_x4_w<FP8>(tmem + 128 * t, da + o, da + o + 2, da + o + 4, da + o + 6, db + o,
                           db + o + 2, db + o + 4, db + o + 6, idesc_s, g > 0 ? 1u : 0u);
        }
      };
      // bf16 with P over S (d = 128): O_t += P_t V over the keys of half `hf` of
      // the block, P from the tile's S columns.
      auto pv_mma = [&](int t, uint32_t vslot, bool acc, int hf) {
        const uint64_t db = dV + (C::slot_off(vslot) >> 4);
        const uint32_t ta = tmem + 128 * t;
        const uint32_t acc0 = (acc || hf > 0) ? 1u : 0u;
        const int k = 4 * hf;   // 16-key steps: P columns advance by 8, V rows by 2048 bytes
        mma_ts_x4_w<false>(tmem + 256 + C::kOCols * t, ta + k * 8, ta + k * 8 + 8, ta + k * 8 + 16,
                           ta + k * 8 + 24, db + k * 128, db + k * 128 + 128, db + k * 128 + 256,
                           db + k * 128 + 384, C::kIdescPV, acc0);
      };
      auto wait_item = [&](uint32_t it) {
        return wait_w(ctl.kv_full[it % C::kStages], (it / C::kStages) & 1);
      };
      if constexpr (C::kDecoupled) {
        // FP8: P outside the S columns, in shared memory.  S_t(j+1) is issued
        // once the softmax has read S_t(j) (s_free) and K_{j+1} has landed;
        // P_t(j).V_j once P_t(j) is stored.  A tile's softmax therefore never
        // waits for its own products: the next S is computed while it works
        // on the current block.  p_free (a commit after each P.V) tells the
        // softmax that the P buffer may be refilled and O rescaled.
        uint32_t ns[2] = {0, 0};   // S products issued per tile
        uint32_t npv = 0;          // P.V products issued per tile
        const uint64_t dP = make_smem_desc(sO, 16, 1024, kSwizzle128B);
        auto issue_s = [&](int t, uint32_t kslot) -> bool {
          if (ns[t] > 0 && !wait_w(ctl.s_free[t], (ns[t] - 1) & 1)) return false;
          ++ns[t];
          tc_fence_after();
          s_mma(t, kslot);
          mma_commit_w(bar(ctl.s_full[t]));
          return true;
        };
        // O_t (+)= P_t V over the block's 128 keys once P_t is stored: four
        // K = 32 steps with P from shared memory.
        auto issue_pv = [&](int t, uint32_t vslot, bool acc) -> bool {
          const uint64_t db = dV + (C::slot_off(vslot) >> 4);
          if (!wait_w(ctl.p_ready[t * C::kPReadyStride], npv & 1)) return false;
          tc_fence_after();
          const uint64_t da = dP + t * (uint64_t)(C::kOStageBytes >> 4);
          mma_ss_x4_w<true>(tmem + 256 + D * t, da, da + 2, da + 4, da + 6, db, db + 2, db + 4,
                            db + 6, C::kIdescPV, acc ? 1u : 0u);
          mma_commit_w(bar(ctl.p_free[t]));
          return true;
        };
        for (uint32_t k = 0; ok; ++k) {
          Unit w{};
          if (!take_unit(k, ok, w)) break;
          const int J = w.nblocks;
          if (J == 0) continue;
          ok = wait_w(ctl.q_full[0], uit & 1) && wait_w(ctl.q_full[1], uit & 1);
          if (!ok) break;
          const uint32_t base = item;   // K_j = base + 2j, V_j = base + 2j + 1
          item += 2 * J;
          if (!(ok = wait_item(base))) break;
          if (!(ok = issue_s(0, base % C::kStages) && issue_s(1, base % C::kStages))) break;
          mma_commit_w(bar(ctl.kv_empty[base % C::kStages]));
          if (J == 1) {
            mma_commit_w(bar(ctl.q_empty[0]));
            mma_commit_w(bar(ctl.q_empty[1]));
          }
          for (int j = 0; j < J && ok; ++j) {
            const uint32_t iv = base + 2 * j + 1, ik = base + 2 * j + 2;
            if (j + 1 < J) {
              if (!(ok = wait_item(ik))) break;
              if (!(ok = issue_s(0, ik % C::kStages) && issue_s(1, ik % C::kStages))) break;
              mma_commit_w(bar(ctl.kv_empty[ik % C::kStages]));
              if (j + 2 == J) {
                mma_commit_w(bar(ctl.q_empty[0]));
                mma_commit_w(bar(ctl.q_empty[1]));
              }
            }
            if (!(ok = wait_item(iv))) break;
            if (!(ok = issue_pv(0, iv % C::kStages, j > 0))) break;
            if (j == J - 1) mma_commit_w(bar(ctl.o_final[0]));
            if (!(ok = issue_pv(1, iv % C::kStages, j > 0))) break;
            mma_commit_w(bar(ctl.kv_empty[iv % C::kStages]));
            if (j == J - 1) mma_commit_w(bar(ctl.o_final[1]));
            ++npv;
          }
          ++uit;
        }
      } else if constexpr (C::kPSep) {
        // bf16 d = 64 (P outside S but for its last 32 keys).  Per block:
        // S(j+1) for keys [0, 112) of each tile once its softmax has read S(j)
        // (s_free) and K(j+1) has landed; then, for each tile once P(j) of
        // keys [96, 128) is stored (p_ready[2 t + 1]), the P.V steps over those
        // keys -- P from S's last 16 columns -- with a commit to pt_done, and
        // S(j+1) for keys [112, 128) over those columns with s_full; then, for
        // each tile once the rest of P(j) is stored (p_ready[2 t]), the P.V
        // steps over keys [0, 96) and p_free.
        uint32_t ns[2] = {0, 0};   // S products issued per tile
        uint32_t npv = 0;          // P.V products issued per tile
        const uint32_t idesc_main = C::kIdescSMain | (p.neg_scale ? kIdescNegateB : 0u);
        const uint32_t idesc_tail = C::kIdescSTail | (p.neg_scale ? kIdescNegateB : 0u);
        auto s_main = [&](int t, uint32_t kslot) -> bool {
          if (ns[t] > 0 && !wait_w(ctl.s_free[t], (ns[t] - 1) & 1)) return false;
          ++ns[t];
          tc_fence_after();
          const uint64_t da = dQ + t * kTileUnits;
          const uint64_t db = dK + (C::slot_off(kslot) >> 4);
          mma_ss_x4_w<false>(tmem + 128 * t, da, da + 2, da + 4, da + 6, db, db + 2, db + 4, db + 6,
                             idesc_main, 0u);
          return true;
        };
        auto s_tail = [&](int t, uint32_t kslot) {
          const uint64_t da = dQ + t * kTileUnits;
          const uint64_t db = dK + ((C::slot_off(kslot) + C::kSMainKeys * 128) >> 4);
          mma_ss_x4_w<false>(tmem + 128 * t + C::kSMainKeys, da, da + 2, da + 4, da + 6, db, db + 2,
                             db + 4, db + 6, idesc_tail, 0u);
          mma_commit_w(bar(ctl.s_full[t]));
        };
        // P.V over 16-key step k: P from the tile's own columns (k < 6) or
        // from S's last 16 columns (k = 6, 7); V rows 2048 bytes apart.
        auto pa = [&](int t, int k) -> uint32_t {
          return k < 6 ? tmem + C::kPCol + 48 * t + 8 * k : tmem + 128 * t + C::kSMainKeys + 8 * (k - 6);
        };
        for (uint32_t k = 0; ok; ++k) {
          Unit w{};
          if (!take_unit(k, ok, w)) break;
          const int J = w.nblocks;
          if (J == 0) continue;
          ok = wait_w(ctl.q_full[0], uit & 1) && wait_w(ctl.q_full[1], uit & 1);
          if (!ok) break;
          const uint32_t base = item;   // K_j = base + 2j, V_j = base + 2j + 1
          item += 2 * J;
          if (!(ok = wait_item(base))) break;
          // The previous unit's last P.V steps (already issued) read P's last
          // keys before these products overwrite them.
          if (!(ok = s_main(0, base % C::kStages))) break;
          s_tail(0, base % C::kStages);
          if (!(ok = s_main(1, base % C::kStages))) break;
          s_tail(1, base % C::kStages);
          mma_commit_w(bar(ctl.kv_empty[base % C::kStages]));
          if (J == 1) {
            mma_commit_w(bar(ctl.q_empty[0]));
            mma_commit_w(bar(ctl.q_empty[1]));
          }
          for (int j = 0; j < J && ok; ++j) {
            const uint32_t iv = base + 2 * j + 1, ik = base + 2 * j + 2;
            const uint32_t vslot = iv % C::kStages, kslot = ik % C::kStages;
            const bool nxt = j + 1 < J;
            if (nxt) {
              if (!(ok = wait_item(ik))) break;
              if (!(ok = s_main(0, kslot) && s_main(1, kslot))) break;
            }
            if (!(ok = wait_item(iv))) break;
            const uint64_t db = dV + (C::slot_off(vslot) >> 4);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (!(ok = wait_w(ctl.p_ready[t * C::kPReadyStride + 1], npv & 1))) break;
              tc_fence_after();
              mma_ts_x2_w(tmem + 256 + C::kOCols * t, pa(t, 6), pa(t, 7), db + 6 * 128, db + 7 * 128,
                          C::kIdescPV, j > 0 ? 1u : 0u);
              mma_commit_w(bar(ctl.pt_done[t]));
              if (nxt) s_tail(t, kslot);
            }
            if (!ok) break;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (!(ok = wait_w(ctl.p_ready[t * C::kPReadyStride], npv & 1))) break;
              tc_fence_after();
              const uint32_t dO = tmem + 256 + C::kOCols * t;
              mma_ts_x4_w<false>(dO, pa(t, 0), pa(t, 1), pa(t, 2), pa(t, 3), db, db + 128, db + 256,
                                 db + 384, C::kIdescPV, 1u);
              mma_ts_x2_w(dO, pa(t, 4), pa(t, 5), db + 4 * 128, db + 5 * 128, C::kIdescPV, 1u);
              mma_commit_w(bar(ctl.p_free[t]));
              if (j == J - 1) mma_commit_w(bar(ctl.o_final[t]));
            }
            if (!ok) break;
            mma_commit_w(bar(ctl.kv_empty[vslot]));
            if (nxt) {
              mma_commit_w(bar(ctl.kv_empty[kslot]));
              if (j + 2 == J) {
                mma_commit_w(bar(ctl.q_empty[0]));
                mma_commit_w(bar(ctl.q_empty[1]));
              }
            }
            ++npv;
          }
          ++uit;
        }
      } else
      for (uint32_t k = 0; ok; ++k) {
        Unit w{};
        if (!take_unit(k, ok, w)) break;
        const int J = w.nblocks;
        if (J == 0) continue;   // empty key range (split-KV)
        ok = wait_w(ctl.q_full[0], uit & 1) && wait_w(ctl.q_full[1], uit & 1);
        if (!ok) break;
        const uint32_t base = item;            // K_j = base + 2j, V_j = base + 2j + 1
        item += 2 * J;
        if (!(ok = wait_item(base))) break;
        tc_fence_after();
        s_mma(0, base % C::kStages);
        mma_commit_w(bar(ctl.s_full[0]));
        s_mma(1, base % C::kStages);
        mma_commit_w(bar(ctl.s_full[1]));
        mma_commit_w(bar(ctl.kv_empty[base % C::kStages]));
        if (J == 1) {
          mma_commit_w(bar(ctl.q_empty[0]));
          mma_commit_w(bar(ctl.q_empty[1]));
        }
        const int J0 = (C::kSkipDiag && w.skip0) ? J - 1 : J;   // blocks of tile 0
        for (int j = 0; j < J && ok; ++j) {
          const uint32_t iv = base + 2 * j + 1, ik = base + 2 * j + 2;
          const uint32_t vslot = iv % C::kStages, kslot = ik % C::kStages;
          if (!(ok = wait_item(iv))) break;
          if (j < J0) {
            if (!(ok = wait_w(ctl.p_ready[0], pr[0] & 1))) break;
            tc_fence_after();
            pv_mma(0, vslot, j > 0, 0);
            ++pr[0];
            tc_fence_after();
            pv_mma(0, vslot, j > 0, 1);
            if (j == J0 - 1) mma_commit_w(bar(ctl.o_final[0]));
          }
          if (j + 1 < J) {
            if (!(ok = wait_item(ik))) break;
            tc_fence_after();
            if (j + 1 < J0) {
              s_mma(0, kslot);
              mma_commit_w(bar(ctl.s_full[0]));
            }
          }
          if (!(ok = wait_w(ctl.p_ready[C::kPReadyStride], pr[1] & 1))) break;
          tc_fence_after();
          pv_mma(1, vslot, j > 0, 0);
          ++pr[1];
          tc_fence_after();
          pv_mma(1, vslot, j > 0, 1);
          mma_commit_w(bar(ctl.kv_empty[vslot]));
          if (j == J - 1) mma_commit_w(bar(ctl.o_final[1]));
          if (j + 1 < J) {
            s_mma(1, kslot);
            mma_commit_w(bar(ctl.s_full[1]));
            mma_commit_w(bar(ctl.kv_empty[kslot]));
            if (j + 2 == J) {
              mma_commit_w(bar(ctl.q_empty[0]));
              mma_commit_w(bar(ctl.q_empty[1]));
            }
          }
        }
        ++uit;
      }
      // Every MMA issued must finish before TMEM is released.
      __syncwarp();
      mma_commit_w(bar(ctl.drain));
      wait_bounded(bar(ctl.drain), 0, wc, false);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax
    regs_inc<C::kRegsSoftmax>();
    const int t = warp >> 2;                 // query tile of the pair
    const int wq = warp & 3;                 // TMEM lane quarter
    const int r = wq * 32 + lane;            // row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + 128 * t;
    const uint32_t tO = tmem + lane_off + 256 + C::kOCols * t;
    // bf16 P: over S (d = 128), or in its own columns but for its last 32
    // keys, which go over S's last 16 columns (d = 64).
    const uint32_t tP = C::kPSep ? tmem + lane_off + C::kPCol + 48 * t : tS;
    const uint32_t tL = tO + D;   // bf16 d = 64: l~ of this row (16 equal columns)
    const float NEG_INF = __int_as_float(0xff800000);
    const bool zero_scale = p.zero_scale != 0;
    uint32_t sit = 0, uit = 0;
    uint32_t np = 0;   // FP8: P blocks this tile has written (phase of p_free)
    bool ok = true;
    // 64 columns of this thread's row of O_t from TMEM, times inv, as bf16 pairs.
    auto load_o_bf16 = [&](int col, float inv_o, uint32_t (&pk)[32]) {
      uint32_t ov[64];
      __syncwarp();
      tmem_ld32(tO + col, *reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
      tmem_ld32(tO + col + 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
      tmem_wait_ld();
      reg_fence(ov);
#pragma unroll
      for (int i = 0; i < 32; ++i)
        pk[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_o, __uint_as_float(ov[2 * i + 1]) * inv_o);
    };
    // Row i of a staging buffer (128 bytes at addr) in the 128-byte swizzle.
    auto stage_row = [&](uint32_t addr, int i, const uint32_t (&pk)[32]) {
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(addr + ((c ^ (i & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();   // generic-proxy writes -> the tensor copy's reads
      __syncwarp();
    };
    for (uint32_t k = 0; ok; ++k) {
      Unit w{};
      if (!take_unit(k, ok, w)) break;
      const int row = w.pair * 256 + t * 128 + r;
      if (w.nblocks == 0) {
        // Empty key range: O_part = 0 and lse_part = -inf (weight 0 in the merge).
        if (row < p.N) {
          const size_t prow = ((size_t)w.split * p.BH + w.bh) * p.N + row;
          float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll 4
          for (int i = 0; i < D / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          p.lse_part[prow] = NEG_INF;
        }
        continue;
      }
      const int lim_row = p.causal ? min(row, p.N - 1) : p.N - 1;   // last visible key
      const int lo_row = p.window > 0 ? row - p.window + 1 : 0;      // first visible key
      float m_ref = NEG_INF, ell = 0.0f;   // reference max (base 2), sum of f32 p
      float ell_r = 0.0f;                   // sum of p as rounded into P (bf16 path)
      float q_s = 1.0f, v_smax = 1.0f, inv_vmax = 1.0f;
      float ks_nx = 1.0f, vs_nx = 1.0f;   // FP8: K and V scales of the next block, loaded a block ahead
      const float* ksc = FP8 ? p.k_scale + (size_t)w.bhk * p.nkb : nullptr;
      const float* vsc = FP8 ? p.v_scale + (size_t)w.bhk * p.nkb : nullptr;
      if (FP8) {
        const int qb = w.pair * 2 + t;
        q_s = (qb < p.nkb) ? __ldg(p.q_scale + (size_t)w.bh * p.nkb + qb) : 1.0f;
        float mx = 0.0f;
        for (int b = lane; b < p.nkb; b += 32) mx = fmaxf(mx, __ldg(vsc + b));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        v_smax = mx;
        inv_vmax = C::kPScale / v_smax;
        ks_nx = __ldg(ksc + w.j0);
        vs_nx = __ldg(vsc + w.j0);
      }
      const int nb_t = w.nblocks - ((C::kSkipDiag && t == 0 && w.skip0) ? 1 : 0);   // tile 0 may skip the last
      for (int jj = 0; jj < nb_t; ++jj) {
        const int j = w.j0 + jj;   // key block
        // FP8: the block's score factor and P fold (V's block scale over the
        // head's largest, times 1.75), from scales loaded one block ahead.
        float cj = p.scale_log2;
        float v_fold = 1.0f, inv_vfold = 1.0f, lg_vfold = 0.0f;
        if (FP8) {
          cj *= q_s * ks_nx;
          v_fold = vs_nx * inv_vmax;
          if (jj + 1 < nb_t) {
            ks_nx = __ldg(ksc + j + 1);
            vs_nx = __ldg(vsc + j + 1);
          }
          // The reciprocal only scales the block's sum of p into l: the
          // approximate instruction (within 1 ulp, subnormals kept) is enough,
          // and measured 2.6 % faster than the correctly rounded one.
          asm("rcp.approx.f32 %0, %1;" : "=f"(inv_vfold) : "f"(v_fold));
          lg_vfold = __log2f(v_fold);
        }
        ok = mbar_test_wait(bar(ctl.s_full[t]), sit & 1) || wait_bounded(bar(ctl.s_full[t]), sit & 1, wc);
        ++sit;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // With P outside the S columns, the previous block's P.V must be done
        // before O_t is rescaled or the P buffer refilled (it was issued as
        // that block's P landed, so this is rarely a wait).
        bool pfree = np == 0;
        auto wait_pfree = [&]() {
          if (pfree) return true;
          pfree = true;
          const uint32_t pb = bar(ctl.p_free[t]), ph = (np - 1) & 1;
          const bool w_ok = __all_sync(0xffffffffu, mbar_test_wait(pb, ph) || wait_bounded(pb, ph, wc));
          tc_fence_after();
          return w_ok;
        };
        const int lim = lim_row - j * 128;    // columns > lim are invisible
        const int lo = lo_row - j * 128;      // columns < lo are invisible (window)
        // S of this block -> x (raw scores; invisible columns -inf).
        auto load_s = [&](float (&x)[128]) {
          uint32_t sr[128];
          tmem_ld128(tS, sr);
          tmem_wait_ld();
          reg_fence(sr);
#pragma unroll
          for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(sr[c]);
          if (lim < 127 || lo > 0 || zero_scale) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              x[c] = (c > lim || c < lo) ? NEG_INF : (zero_scale ? 0.0f : x[c]);
          }
        };
        auto row_max = [&](const float (&x)[128]) {
          float m0 = fmaxf(x[0], x[1]), m1 = fmaxf(x[2], x[3]);
          float m2 = fmaxf(x[4], x[5]), m3 = fmaxf(x[6], x[7]);
#pragma unroll
          for (int c = 8; c < 128; c += 8) {
            m0 = max3(m0, x[c], x[c + 1]);
            m1 = max3(m1, x[c + 2], x[c + 3]);
            m2 = max3(m2, x[c + 4], x[c + 5]);
            m3 = max3(m3, x[c + 6], x[c + 7]);
          }
          return max3(m0, m1, fmaxf(m2, m3));
        };
        // O_t *= alpha (per row); only called when some row of the warp needs it.
        auto rescale_o = [&](float alpha) {
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 32) {
            uint32_t orow[32];
            tmem_ld32(tO + cc, orow);
            tmem_wait_ld();
            reg_fence(orow);
#pragma unroll
            for (int i = 0; i < 32; ++i) orow[i] = __float_as_uint(__uint_as_float(orow[i]) * alpha);
            tmem_st32(tO + cc, orow);
          }
          if constexpr (C::kLFused) {
            uint32_t lrow[16];
            tmem_ld16(tL, lrow);
            tmem_wait_ld();
            reg_fence(lrow);
#pragma unroll
            for (int i = 0; i < 16; ++i) lrow[i] = __float_as_uint(__uint_as_float(lrow[i]) * alpha);
            tmem_st16(tL, lrow);
          }
        };
        if constexpr (FP8) {
          // p' = p * v_fold = 2^(s c - (m - log2 v_fold)) against the running
          // reference m (V's block scale rides in the exponent).  m moves to the
          // block's max only when that max exceeds m by more than 8 (base 2), so
          // p <= 2^8 and P' = p * v_fold <= 256 * kPScale = 448, inside E4M3's
          // range.
          uint32_t pk[32];
          float e_sum;
          // Exponentials of keys [64hf, 64hf + 64) into pk[16hf, 16hf + 16);
          // returns their sum of p.
          auto exps_half = [&](const float (&x)[128], int hf) -> float {
            const float m_use = (m_ref == NEG_INF) ? 0.0f : m_ref;
            const float m_f = m_use - lg_vfold;
            const uint64_t c2 = f32x2_pack(cj, cj);
            const uint64_t nm2 = f32x2_pack(-m_f, -m_f);
            uint64_t s01 = 0, s23 = 0;   // (0.f, 0.f)
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) {
              const int i = 16 * hf + ii;
              const int c = 4 * i;
              float t0, t1, t2, t3;
              f32x2_unpack(f32x2_fma(f32x2_pack(x[c], x[c + 1]), c2, nm2), t0, t1);
              f32x2_unpack(f32x2_fma(f32x2_pack(x[c + 2], x[c + 3]), c2, nm2), t2, t3);
              const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
              const float p2 = ex2_approx(t2), p3 = ex2_approx(t3);
              s01 = f32x2_add(s01, f32x2_pack(p0, p1));
              s23 = f32x2_add(s23, f32x2_pack(p2, p3));
              pk[i] = pack_e4m3x4(p0, p1, p2, p3);
            }
            float a0, a1;
            f32x2_unpack(f32x2_add(s01, s23), a0, a1);
            return (a0 + a1) * inv_vfold;
          };
          {
            // The block's max first: E4M3 P must never saturate, and with the
            // outliers FP8 inputs carry, large rises of a row's max are common
            // enough that retaking a block would cost more than this pass.
            float x[128];
            load_s(x);
            // S is in registers now: the tile's next S product may overwrite it.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(ctl.s_free[t]));
            const float m_blk = row_max(x) * cj;
            const bool need = m_blk > m_ref + C::kTauLog2;
            const float m_new = need ? m_blk : m_ref;
            const float alpha = need ? ex2_approx(m_ref - m_new) : 1.0f;   // 0 when m_ref = -inf
            if (jj > 0 && __any_sync(0xffffffffu, need)) {
              if (!(ok = wait_pfree())) break;
              rescale_o(alpha);
              tmem_wait_st();   // the rescaled O is in TMEM before P.V (signalled below) adds to it
              tc_fence_before();
            }
            ell *= alpha;
            m_ref = m_new;
            // keys [64hf, 64hf+64) -> bytes [64hf, 64hf+64) of this row of the
            // tile's P buffer (the 128-byte swizzle of a K-major operand: 16-byte
            // chunk c of row r at position c ^ (r & 7)); the first half is stored
            // while the second half's exponentials run, and P.V is signalled once
            // (it is off the softmax's path: the next S is already computed).
            const uint32_t prow = sO + t * C::kOStageBytes + r * 128;
            e_sum = 0.0f;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              e_sum += exps_half(x, hf);
              if (hf == 0) {
                if (!(ok = wait_pfree())) break;
                if (jj == 0 && uit > 0) {
                  // The previous unit's O left through this buffer: its tensor
                  // stores must have read it.
                  if (lane == 0) bulk_wait_read_all();
                  __syncwarp();
                }
              }
#pragma unroll
              for (int c = 4 * hf; c < 4 * hf + 4; ++c)
                st_shared_v4(prow + ((c ^ (r & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                             pk[4 * c + 3]);
            }
            fence_proxy_async_smem();   // generic-proxy writes -> the MMA's operand reads
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(ctl.p_ready[t * C::kPReadyStride]));
            ++np;
            if (!ok) break;
          }
          ell += e_sum;
        } else if constexpr (C::kPSep) {
          // bf16, d = 64.  p = 2^(s*c - m) against the running reference m, as
          // at d = 128 below (the block's sum bounds every p; a block whose sum
          // passes 2^32 moves m to its max and is taken again), with two
          // differences: l~ comes from the tensor core (the ones beside V), and
          // P of keys [96, 128) is computed, tested, stored over S's last 16
          // columns and signalled first, so that the tile's P.V over those keys
          // and the rest of its next S run while the softmax works on keys
          // [0, 96).  If the whole block's sum then fails the test, O and l~
          // already hold P.V over the last keys at the old reference: once that
          // product is done (pt_done) they are rescaled with the rest, and the
          // sum of those keys' p is scaled by the same factor.
          uint32_t pk[64];
          // Exponentials of key pairs [i0, i0 + n) into pk[i0, i0 + n); returns
          // their sum of p.
          auto exps_pairs = [&](const float (&x)[128], int i0, int n) -> float {
            const float m_use = (m_ref == NEG_INF) ? 0.0f : m_ref;
            const uint64_t c2 = f32x2_pack(cj, cj);
            const uint64_t nm2 = f32x2_pack(-m_use, -m_use);
            uint64_t ex0 = 0, ex1 = 0;   // (0.f, 0.f)
#pragma unroll
            for (int ii = 0; ii < n; ++ii) {
              const int i = i0 + ii;
              float t0, t1;
              f32x2_unpack(f32x2_fma(f32x2_pack(x[2 * i], x[2 * i + 1]), c2, nm2), t0, t1);
              const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
              pk[i] = pack_bf16x2(p0, p1);
              if (ii & 1)
                ex1 = f32x2_add(ex1, f32x2_pack(p0, p1));
              else
                ex0 = f32x2_add(ex0, f32x2_pack(p0, p1));
            }
            float b0, b1;
            f32x2_unpack(f32x2_add(ex0, ex1), b0, b1);
            return b0 + b1;
          };
          // Rows with `redo` move m to the block's max; returns their factor.
          auto move_ref = [&](const float (&x)[128], bool redo) -> float {
            const float m_blk = row_max(x) * cj;
            const float m_new = redo ? fmaxf(m_ref, m_blk) : m_ref;
            const float alpha = redo ? ex2_approx(m_ref - m_new) : 1.0f;   // 0 when m_ref = -inf
            ell *= alpha;
            m_ref = m_new;
            return alpha;
          };
          float x[128];
          load_s(x);
          // S is in registers now: the tile's next S product may overwrite it.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(ctl.s_free[t]));
          if (!__all_sync(0xffffffffu, m_ref != NEG_INF)) {
            const float m_blk0 = row_max(x) * cj;
            if (m_ref == NEG_INF) m_ref = m_blk0;
          }
          float sum_tail = exps_pairs(x, 48, 16);
          // Stored before its sum is tested (a retake stores it again before
          // the signal): 0.5 % faster than storing after the test.
          __syncwarp();   // tcgen05.st is warp-collective
          tmem_st16(tS + C::kSMainKeys, *reinterpret_cast<uint32_t(*)[16]>(&pk[48]));
          if (__any_sync(0xffffffffu, !(sum_tail <= C::kSumLimit))) {
            const float alpha = move_ref(x, !(sum_tail <= C::kSumLimit));
            if (jj > 0) {
              if (!(ok = wait_pfree())) break;
              rescale_o(alpha);
            }
            sum_tail = exps_pairs(x, 48, 16);
            tmem_wait_st();
            __syncwarp();
            tmem_st16(tS + C::kSMainKeys, *reinterpret_cast<uint32_t(*)[16]>(&pk[48]));
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(ctl.p_ready[t * C::kPReadyStride + 1]));
          float sum_main = exps_pairs(x, 0, 32);
          if (!(ok = wait_pfree())) break;
          __syncwarp();
          tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
          sum_main += exps_pairs(x, 32, 16);
          __syncwarp();
          tmem_st16(tP + 32, *reinterpret_cast<uint32_t(*)[16]>(&pk[32]));
          if (__any_sync(0xffffffffu, !(sum_tail + sum_main <= C::kSumLimit))) {
            const uint32_t pb = bar(ctl.pt_done[t]), ph = np & 1;
            if (!(ok = __all_sync(0xffffffffu, mbar_test_wait(pb, ph) || wait_bounded(pb, ph, wc)))) break;
            tc_fence_after();
            const float alpha = move_ref(x, !(sum_tail + sum_main <= C::kSumLimit));
            rescale_o(alpha);
            sum_tail *= alpha;
            sum_main = exps_pairs(x, 0, 32) + exps_pairs(x, 32, 16);
            tmem_wait_st();   // this block's first stores are done before they are replaced
            __syncwarp();
            tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
            tmem_st16(tP + 32, *reinterpret_cast<uint32_t(*)[16]>(&pk[32]));
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(ctl.p_ready[t * C::kPReadyStride]));
          ++np;
          ell += sum_tail + sum_main;
        } else {
          // p = 2^(s*c - m) against the running reference max m, so no
          // exponential waits for the block's max.  The block's sum of p bounds
          // every p in it: if the sum is at most 2^32 the pass stands (p <= 2^32;
          // bf16 P and the f32 sums have the range for it, and their relative
          // precision does not depend on the reference).  Otherwise (rare after
          // the first block: the block's max is then more than 25 above m) m
          // moves to the block's max, O and the sums are rescaled and the block
          // (still in registers; P is not signalled yet) is taken again.  P is rounded to
          // bf16 for the PV MMA; the sum of exactly those rounded values (l~)
          // normalises O, so numerator and denominator use the same weights,
          // while the sum of the f32 values (l) gives the logsumexp.
          uint32_t pk[64];
          float e_sum, r_sum;
          // Exponentials of keys [64h, 64h + 64) into P pairs pk[32h, 32h + 32),
          // with their sums (f32 p and bf16-rounded p).
          auto exps_half = [&](const float (&x)[128], int h, float& es, float& rs) {
            const float m_use = (m_ref == NEG_INF) ? 0.0f : m_ref;
            const uint64_t c2 = f32x2_pack(cj, cj);
            const uint64_t nm2 = f32x2_pack(-m_use, -m_use);
            uint64_t ex0 = 0, ex1 = 0;   // (0.f, 0.f)
            float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) {
              const int i = 32 * h + ii;
              float t0, t1;
              f32x2_unpack(f32x2_fma(f32x2_pack(x[2 * i], x[2 * i + 1]), c2, nm2), t0, t1);
              const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
              const uint32_t pb = pack_bf16x2(p0, p1);
              pk[i] = pb;
              const uint64_t e = f32x2_pack(p0, p1);
              if (ii & 1) {
                r2 = add_bf16_lo(pb, r2);
                r3 = add_bf16_hi(pb, r3);
                ex1 = f32x2_add(ex1, e);
              } else {
                r0 = add_bf16_lo(pb, r0);
                r1 = add_bf16_hi(pb, r1);
                ex0 = f32x2_add(ex0, e);
              }
            }
            float b0, b1;
            f32x2_unpack(f32x2_add(ex0, ex1), b0, b1);
            es = b0 + b1;
            rs = (r0 + r1) + (r2 + r3);
          };
          // S stays in registers for the whole block (a retaken block needs no
          // reload), and P of keys [0, 64) is stored over S columns [0, 32) --
          // already read -- while the second half's exponentials run; P is
          // signalled only once the block's sum has passed.  A row with no
          // visible key yet (every row at a unit's first block) takes its
          // reference from the block's max first; its O and sums are still 0, so
          // nothing is rescaled.
          float x[128];
          load_s(x);
          if (!__all_sync(0xffffffffu, m_ref != NEG_INF)) {
            const float m_blk0 = row_max(x) * cj;
            if (m_ref == NEG_INF) m_ref = m_blk0;
          }
          float es0, rs0, es1, rs1;
          exps_half(x, 0, es0, rs0);
          __syncwarp();   // tcgen05.st is warp-collective
          tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
          exps_half(x, 1, es1, rs1);
          e_sum = es0 + es1;
          r_sum = rs0 + rs1;
          // A sum of 128 terms above 2^32 has a term above 2^25; moving m to the
          // block's max makes every term <= 1, so one more pass suffices.
          const bool redo = !(e_sum <= C::kSumLimit);
          if (__any_sync(0xffffffffu, redo)) {
            const float m_blk = row_max(x) * cj;
            const float m_new = redo ? fmaxf(m_ref, m_blk) : m_ref;
            const float alpha = redo ? ex2_approx(m_ref - m_new) : 1.0f;
            if (jj > 0) rescale_o(alpha);
            ell *= alpha;
            ell_r *= alpha;
            m_ref = m_new;
            exps_half(x, 0, es0, rs0);
            exps_half(x, 1, es1, rs1);
            e_sum = es0 + es1;
            r_sum = rs0 + rs1;
            tmem_wait_st();   // this block's first stores are done before they are replaced
            __syncwarp();
            tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
          }
          // P of keys [64, 128), after the sum test (storing it before the test
          // measured 4 % slower here).
          __syncwarp();   // tcgen05.st is warp-collective
          tmem_st32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
          // bf16: one signal for all keys of the block (P·V waits for it once).
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(ctl.p_ready[t * C::kPReadyStride]));
          ell_r += r_sum;
          ell += e_sum;
        }
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      ok = wait_bounded(bar(ctl.o_final[t]), uit & 1, wc);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float inv;
      if (FP8)
        inv = (ell > 0.0f) ? v_smax / C::kPScale / ell : 0.0f;
      else {
        if constexpr (C::kLFused) {
          // l~ as the tensor core summed the block products' P (all 16 columns equal).
          uint32_t lrow[16];
          tmem_ld16(tL, lrow);
          tmem_wait_ld();
          reg_fence(lrow);
          ell_r = __uint_as_float(lrow[0]);
        }
        inv = (ell_r > 0.0f) ? 1.0f / ell_r : 0.0f;
      }
      const bool live = row < p.N;
      const float l2e = (ell > 0.0f) ? (m_ref + __log2f(ell)) * 0.69314718055994531f : NEG_INF;
      if (p.o_part != nullptr) {
        // Split-KV: this key range's O (normalised by its own sum) in fp32.
        const size_t prow = ((size_t)w.split * p.BH + w.bh) * p.N + row;
        float* orow_p = p.o_part + prow * D;
        // d = 128: staged per warp like the bf16 epilogue below, in 32-column
        // boxes (32 rows x 128 bytes) of the f32 partial-O tensor map.
        const uint32_t wstage = sO + t * C::kOStageBytes + wq * 4096;
        const int wrow0 = w.pair * 256 + t * 128 + wq * 32;
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t ov[32];
          __syncwarp();
          tmem_ld32(tO + cc, ov);
          tmem_wait_ld();
          reg_fence(ov);
          if constexpr (D == 128) {
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * inv);
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c)
              st_shared_v4(wstage + lane * 128 + ((c ^ (lane & 7)) << 4), ov[4 * c], ov[4 * c + 1],
                           ov[4 * c + 2], ov[4 * c + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && wrow0 < p.N) {
              tma_store_3d(&tmO, wstage, cc, wrow0, w.split * p.BH + w.bh);
              bulk_commit();
            }
          } else if (live) {
            float4* dst = reinterpret_cast<float4*>(orow_p + cc);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(ov[4 * i]) * inv, __uint_as_float(ov[4 * i + 1]) * inv,
                                   __uint_as_float(ov[4 * i + 2]) * inv, __uint_as_float(ov[4 * i + 3]) * inv);
          }
        }
        if (live) p.lse_part[prow] = l2e;
      } else {
        // O_t in bf16 through shared memory: each thread writes its row of a
        // 64-column slab into a staging buffer in the 128-byte swizzled layout
        // of the O tensor map (row i at 128 i, 16-byte chunk c at position
        // c ^ (i & 7): conflict-free), and one lane stores the buffer with a
        // tensor copy (rows past N are clipped).  Full lines reach L2 and the
        // warps go on while the copy drains; a buffer is written again only
        // after the copy out of it has read it.
        // Each warp stages and stores its own 32 rows (4 KB buffers), so that
        // no warp waits on another.
        if constexpr (D == 128) {
          const uint32_t wstage = sO + t * C::kOStageBytes + wq * 4096;
          const int wrow0 = w.pair * 256 + t * 128 + wq * 32;
          // All 128 columns of the row in one TMEM round trip (the softmax's
          // registers are free here), then the two 64-column slabs through
          // the staging buffer one after the other.
          uint32_t pk[2][32];
          {
            uint32_t ov[128];
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tO + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&ov[32 * c]));
            tmem_wait_ld();
            reg_fence(ov);
#pragma unroll
            for (int i = 0; i < 64; ++i)
              pk[i >> 5][i & 31] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv, __uint_as_float(ov[2 * i + 1]) * inv);
          }
#pragma unroll
          for (int sl = 0; sl < 2; ++sl) {
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            stage_row(wstage + lane * 128, lane, pk[sl]);
            if (lane == 0 && wrow0 < p.N) {
              tma_store_3d(&tmO, wstage, 64 * sl, wrow0, w.bh);
              bulk_commit();
            }
          }
        } else {
          // d = 64: each thread stores its 128-byte row directly (staging it
          // measured slower here).
          uint32_t pk[32];
          load_o_bf16(0, inv, pk);
          if (live) {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.o) +
                                                  ((size_t)w.bh * p.N + row) * D);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
        if (live && p.lse != nullptr) p.lse[(size_t)w.bh * p.N + row] = l2e;
      }
      ++uit;
      // The next unit's first P arrive (after this epilogue) releases O_t.
    }
    // The staging buffers must outlive every copy out of them.
    if (D == 128 && lane == 0) bulk_wait_all();
  } else {
    regs_dec<C::kRegsOther>();   // warps 10, 11: no role
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, C::kTmemCols);
}

}  // namespace gb300

namespace gb300 {

// Host-side launch of one instantiation (defined in this header so that each
// translation unit instantiates exactly one configuration).
// Unit counters of the dynamic scheduler (one file-scope array per translation
// unit).  Each launch takes the next of 64 counters in turn and zeroes it on
// its stream first, so launches in flight on different streams do not share a
// counter (unless 64 of them overlap).  The array's device address is looked
// up on every launch, for the device current then: a cached address would
// outlive a context torn down and created again (cudaDeviceReset).
static __device__ int g_unit_counter[64];

static cudaError_t unit_counter(cudaStream_t stream, int** out) {
  static std::atomic<unsigned> next{0};
  void* a = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&a, g_unit_counter);
  if (e != cudaSuccess) return e;
  if (a == nullptr) return cudaErrorInvalidSymbol;
  int* c = static_cast<int*>(a) + (next.fetch_add(1u, std::memory_order_relaxed) % 64u);
  if ((e = cudaMemsetAsync(c, 0, sizeof(int), stream)) != cudaSuccess) return e;
  *out = c;
  return cudaSuccess;
}

template <int D, bool FP8>
cudaError_t launch_attn(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                        const CUtensorMap& o, const AttnParams& p, int grid, cudaStream_t stream) {
  using C = KCfg<D, FP8>;
  auto kern = attn_fwd_kernel<D, FP8>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  // The register split inside the kernel draws on the pool the launch
  // allocates; refuse to launch a build whose register count would leave the
  // softmax warps' increase waiting forever.
  cudaFuncAttributes fa{};
  if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
  if (fa.numRegs < C::kLaunchRegs) return cudaErrorInvalidConfiguration;
  AttnParams pd = p;
  if ((e = unit_counter(stream, &pd.sched)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kern, q, k, v, o, pd);
}

// Status word of this translation unit's kernels.
inline int read_tu_status(bool clear) {
  int s = 0;
  if (cudaMemcpyFromSymbol(&s, g_attn_status, sizeof(int)) != cudaSuccess) return -4;
  if (clear && s != 0) {
    int z = 0;
    if (cudaMemcpyToSymbol(g_attn_status, &z, sizeof(int)) != cudaSuccess) return -4;
  }
  return s;
}

}  // namespace gb300
