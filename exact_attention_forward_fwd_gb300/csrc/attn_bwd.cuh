// Exact attention backward for sm_103a: dQ, dK, dV of O = softmax(scale Q K^T
// [+mask]) V given dO, the forward's O and its logsumexp L.
//
// Method ("4.3 FlashAttention 2 & 3: Work Partitioning, Warp Specialization &
// FP8", section "The backward pass: recompute, and the one identity that makes
// it tile-able"; "Learn: The Memory Wall & FlashAttention", section 5.3):
//   * S and P are recomputed tile by tile, never stored: P_ij = exp(S_ij - L_i);
//   * D_i = rowdot(dO_i, O_i) is computed once by a small preprocessing kernel;
//   * dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = scale dS K,
//     dK = scale dS^T Q;
//   * dK, dV are reductions over query blocks: one work unit owns a key block
//     and loops over the query blocks that see it, so they accumulate locally.
//     dQ, the reduction over key blocks, is computed by a second kernel that
//     owns a query block and loops over key blocks -- the "separate pass" the
//     page names as the alternative to atomic adds -- so the result is
//     deterministic.  That recomputes S and dP once more (7 tile products per
//     (query block, key block) instead of 5).
//
// Blackwell mapping (this file's own design), both kernels one persistent CTA
// per SM, 576 threads: warps 0-15 element-wise work (warp w owns TMEM lane
// quarter w & 3 and the 32 tile columns [32(w >> 2), +32)), warp 16 TMA, warp
// 17 TMEM allocation and every tcgen05.mma from one thread.  Sixteen
// element-wise warps (four per SM sub-partition) hide the latency of the TMEM
// loads; the per-query L and D of the dK/dV kernel arrive in shared memory by
// bulk copy with each Q tile.
//   dK/dV kernel (keys on the TMEM lanes): S^T = K Q^T and dP^T = V dO^T (SS);
//     P^T (bf16) over S^T, dS^T (bf16) over dP^T; dV += P^T dO and
//     dK += dS^T Q (TS, P^T / dS^T straight from TMEM, Q and dO as MN-major
//     B operands -- the tiles TMA loaded for the SS products).  TMEM: S^T
//     [0,128), dP^T [128,256), dV [256,256+D), dK [256+D,256+2D).  The
//     element-wise pass first writes P^T (dV can start) and then dS^T.
//   dQ kernel (queries on the lanes, L and D per thread): S = Q K^T into one of
//     two buffers [0,128) / [384,512), dP = dO V^T [128,256), dS (bf16) over S,
//     dQ += dS K (TS, K as MN-major B) [256,256+D).  S(j+1) runs during the
//     element-wise pass of block j.
// Every wait is bounded (status word + abort flag, as in the forward).
#pragma once

#include "attn_kernel.cuh"

namespace gb300 {

struct BwdParams {
  const float* lp;       // [BH][Npad] L * log2(e) (+inf past N)
  const float* dd;       // [BH][Npad] D = rowdot(dO, O) (0 past N)
  const uint16_t* q;     // bf16 [BH][N][D] (read directly by the dQ kernel)
  const uint16_t* dO;    // bf16 [BH][N][D]
  void* dq;              // bf16 [BH][N][D]
  void* dk;              // bf16 [BHk][N][D]
  void* dv;              // bf16 [BHk][N][D]
  int* status;           // device status word, or null for the library's own word
  int N, Npad;           // sequence length; N rounded up to 128
  int BH, BHk, H, Hk;    // batch * query heads, batch * KV heads, heads per batch
  int group;             // query heads per KV head
  int window, causal;
  int nb;                // ceil(N / 128): query blocks == key blocks
  int num_units;
  int hgroup;            // causal order: heads per group (their streamed tiles stay in L2)
  int* sched;            // unit counter for dynamic scheduling (zeroed before launch), or null
  float scale_log2;      // |scale| * log2(e) (log2(e) when scale = 0)
  int neg_scale;         // scale < 0: the score products negate their B operand
  int zero_scale;        // scale = 0: every visible score is 0
  float scale;           // signed: multiplies dQ and dK
  unsigned long long timeout_ns;
};

template <int D>
struct BCfg {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  static constexpr int kTile = 128 * D * 2;                 // 128 rows x D bf16
  static constexpr int kSlabs = D / 64;                     // 128-byte column slabs
  // Ring of tiles: dK/dV kernel Q/dO tiles (K, V fixed per unit; L', D come
  // from global memory); dQ kernel K/V tiles (its Q and dO live in TMEM, so the
  // ring gets the rest).  Five 32 KB stages at d = 128 (230 KB with K and V):
  // with four, the next block's Q tile still in flight stalled the MMA warp.
  static constexpr int kStages = (D == 128) ? 5 : 12;
  static constexpr int kStagesDQ = (D == 128) ? 6 : 12;
  static constexpr int kSmemBytes = (2 + kStages) * kTile + 1024;
  static constexpr int kSmemBytesDQ = kStagesDQ * kTile + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kEW = 16;                            // element-wise warps
  static constexpr int kThreads = (kEW + 2) * 32;
  static constexpr int kSSteps = D / 16;                    // K = D for S, dP
  static constexpr uint32_t kIdescSS = make_idesc(128, 128, 1, 1, false, false);
  static constexpr uint32_t kIdescTS = make_idesc(128, D, 1, 1, false, true);
};

// Bulk copy (no tensor map) of `bytes` (multiple of 16, both addresses 16-byte
// aligned) into this CTA's shared memory, completing on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

struct BwdCtl {
  uint64_t full[16];       // ring slot loaded
  uint64_t empty[16];      // ring slot free
  uint64_t fix_full;       // the unit's fixed tiles (K, V or Q, dO) loaded
  uint64_t fix_empty;      // ... free again
  uint64_t s_full;         // S (dK/dV: S^T) of a block computed
  uint64_t dp_full;        // dP (dK/dV: dP^T) of a block computed
  uint64_t s_read;         // dQ kernel: S of a block read by all element-wise warps
  uint64_t p_ready;        // dK/dV: P^T written; dQ: dS written (16 warp arrivals)
  uint64_t ds_ready;       // dK/dV: dS^T written (16 warp arrivals)
  uint64_t unit_done;      // the unit's accumulators final
  uint64_t drain;
  uint64_t unit_full[4];   // ring of work-unit indices handed out by the load warp
  uint64_t unit_empty[4];
  int unit_ring[4];
  uint32_t tmem_base;
  int abort_flag;
};

// Causal unit order shared by both kernels: longest first within groups of
// `hgroup` heads (bigger first when `ascending` is false), the groups one after
// the other.  Returns (head, block).
__device__ __forceinline__ void bwd_causal_order(int u, int heads, int nb, int hgroup, bool ascending,
                                                 int& head, int& blk) {
  const int HG = hgroup > 0 ? min(hgroup, heads) : heads;
  const int per_group = HG * nb;
  const int g = u / per_group;
  const int v = u - g * per_group;
  const int hg = min(HG, heads - g * HG);
  const int rr = v / hg;
  head = g * HG + (v - rr * hg);
  blk = ascending ? rr : nb - 1 - rr;
}

// Query blocks [i_lo, i_hi] that see key block j.
__device__ __forceinline__ void bwd_qrange(int j, const BwdParams& p, int& i_lo, int& i_hi) {
  i_lo = p.causal ? j : 0;
  i_hi = p.nb - 1;
  if (p.window > 0) i_hi = min(i_hi, (j * 128 + 126 + p.window) / 128);
}

// Key blocks [j_lo, j_hi] that query block i sees.
__device__ __forceinline__ void bwd_krange(int i, const BwdParams& p, int& j_lo, int& j_hi) {
  j_hi = p.causal ? i : p.nb - 1;
  j_lo = p.window > 0 ? max(0, i * 128 - p.window + 1) / 128 : 0;
}

// Element (key k, query q) visible under the mask (k, q global; q < N assumed).
__device__ __forceinline__ bool bwd_visible(int k, int q, const BwdParams& p) {
  return k < p.N && (!p.causal || k <= q) && (p.window <= 0 || k > q - p.window);
}

// ============================================================================
// dK, dV: one unit = (batch * KV head, 128-key block j).
// ============================================================================
template <int D>
__global__ void __launch_bounds__(576, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                         const BwdParams p) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sK = smem_addr(smem);
  const uint32_t sV = sK + C::kTile;
  const uint32_t sRing = sV + C::kTile;     // Q_i / dO_i tiles, alternating
  // L' and D of the query block of the Q item in ring slot s: 128 + 128 floats
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](uint64_t& b) { return smem_addr(&b); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(ctl.full[s]), 1);
      mbar_init(bar(ctl.empty[s]), 1);
    }
    mbar_init(bar(ctl.fix_full), 1);
    mbar_init(bar(ctl.fix_empty), 1);
    mbar_init(bar(ctl.s_full), 1);
    mbar_init(bar(ctl.dp_full), 1);
    mbar_init(bar(ctl.p_ready), C::kEW);
    mbar_init(bar(ctl.ds_ready), C::kEW);
    mbar_init(bar(ctl.unit_done), 1);
    mbar_init(bar(ctl.drain), 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(bar(ctl.unit_full[s]), 1);
      mbar_init(bar(ctl.unit_empty[s]), C::kEW + 1);   // the MMA thread and the element-wise warps
    }
    ctl.abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  if (warp == C::kEW + 1) {
    tmem_alloc(smem_addr(&ctl.tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const WaitCtx wc{&ctl.abort_flag, p.status ? p.status : &g_attn_status, p.timeout_ns};
  // Work units: the load warp takes the next index (atomic counter, or the
  // static stride without one) and passes it through a 4-entry ring; -1 ends.
  auto publish_unit = [&](uint32_t k, bool& ok) -> int {
    int u = p.sched ? atomicAdd(p.sched, 1) : static_cast<int>(blockIdx.x + k * gridDim.x);
    if (u >= p.num_units) u = -1;
    const uint32_t slot = k & 3;
    if (k >= 4 && !(ok = wait_bounded(bar(ctl.unit_empty[slot]), ((k >> 2) - 1) & 1, wc))) return -1;
    ctl.unit_ring[slot] = u;
    mbar_arrive(bar(ctl.unit_full[slot]));
    return u;
  };
  auto take_unit = [&](uint32_t k, bool& ok) -> int {   // a whole warp; lane 0 frees the slot
    const uint32_t slot = k & 3;
    ok = wait_bounded(bar(ctl.unit_full[slot]), (k >> 2) & 1, wc);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return -1;
    const int u = *reinterpret_cast<volatile int*>(&ctl.unit_ring[slot]);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(ctl.unit_empty[slot]));
    return u;
  };

  // Unit u -> (bhk, j).  Causal: ascending j (key block 0 sees the most query
  // blocks) across all heads first; otherwise the key blocks of one head in turn.
  auto unit = [&](int u, int& bhk, int& j) {
    if (p.causal) {
      bwd_causal_order(u, p.BHk, p.nb, p.hgroup, true, bhk, j);   // key block 0 sees the most
    } else {
      bhk = u / p.nb;
      j = u - bhk * p.nb;
    }
  };

  if (warp == C::kEW) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      prefetch_tensormap(&tmdO);
      const uint64_t pol_fix = l2_policy_evict_first();
      const uint64_t pol_ring = l2_policy_evict_last();
      uint32_t item = 0, uit = 0;
      bool ok = true;
      for (uint32_t k = 0; ok; ++k, ++uit) {
        const int u = publish_unit(k, ok);
        if (u < 0) break;
        int bhk, j;
        unit(u, bhk, j);
        int i_lo, i_hi;
        bwd_qrange(j, p, i_lo, i_hi);
        const int nI = i_hi - i_lo + 1;
        const int b = bhk / p.Hk, g = bhk - (bhk / p.Hk) * p.Hk;
        if (uit > 0 && !(ok = wait_bounded(bar(ctl.fix_empty), (uit - 1) & 1, wc))) break;
        mbar_arrive_expect_tx(bar(ctl.fix_full), 2 * C::kTile);
        for (int s = 0; s < C::kSlabs; ++s) {
          tma_load_3d_hint(sK + s * 16384, &tmK, bar(ctl.fix_full), s * 64, j * 128, bhk, pol_fix);
          tma_load_3d_hint(sV + s * 16384, &tmV, bar(ctl.fix_full), s * 64, j * 128, bhk, pol_fix);
        }
        for (int t = 0; t < p.group * nI && ok; ++t) {
          const int hh = t / nI, i = i_lo + (t - hh * nI);
          const int bh = b * p.H + g * p.group + hh;
          for (int w2 = 0; w2 < 2 && ok; ++w2, ++item) {   // Q_i (+ L', D), then dO_i
            const uint32_t slot = item % C::kStages;
            if (!(ok = wait_bounded(bar(ctl.empty[slot]), ((item / C::kStages) & 1) ^ 1, wc))) break;
            mbar_arrive_expect_tx(bar(ctl.full[slot]), C::kTile);
            for (int s = 0; s < C::kSlabs; ++s)
              tma_load_3d_hint(sRing + slot * C::kTile + s * 16384, w2 == 0 ? &tmQ : &tmdO,
                               bar(ctl.full[slot]), s * 64, i * 128, bh, pol_ring);
          }
        }
      }
      // Let every copy started land before the CTA can exit.
      const uint32_t issued = item;
      for (uint32_t s = 0; s < (uint32_t)C::kStages && s < issued; ++s) {
        const uint32_t last = s + ((issued - 1 - s) / C::kStages) * C::kStages;
        wait_bounded(bar(ctl.full[s]), (last / C::kStages) & 1, wc, false);
      }
      if (uit > 0) wait_bounded(bar(ctl.fix_full), (uit - 1) & 1, wc, false);
    }
  } else if (warp == C::kEW + 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop converged; one elected lane issues each
    // MMA and commit (the *_w forms), every wait is taken by all lanes.
    {
      uint32_t item = 0, uit = 0, gblk = 0;
      auto wait_w = [&](uint32_t b, uint32_t parity) {
        return __all_sync(0xffffffffu, wait_bounded(b, parity, wc));
      };
      bool ok = true;
      auto wait_slot = [&](uint32_t it) {
        return wait_w(bar(ctl.full[it % C::kStages]), (it / C::kStages) & 1);
      };
      // SS product [M = 128 rows of a] x [N = 128 rows of b]^T over K = D, four
      // k-steps per election; a k-step adds its offset (16-byte units) to the
      // descriptors' address field.
      // S^T = K Q^T negates Q (its B operand) for a negative scale; dP^T does not.
      const uint32_t idesc_s = C::kIdescSS | (p.neg_scale ? kIdescNegateB : 0u);
      auto ss = [&](uint32_t d_col, uint32_t a0, uint32_t b0, uint32_t idesc) {
        const uint64_t da = make_smem_desc(a0, 16, 1024, kSwizzle128B);
        const uint64_t db = make_smem_desc(b0, 16, 1024, kSwizzle128B);
#pragma unroll
        for (int g = 0; g < C::kSSteps / 4; ++g) {
          const uint64_t o = g * 1024;   // next 128-byte column slab
          mma_ss_x4_w<false>(tmem + d_col, da + o, da + o + 2, da + o + 4, da + o + 6, db + o,
                             db + o + 2, db + o + 4, db + o + 6, idesc, g > 0 ? 1u : 0u);
        }
      };
      // TS product: A = 128 x 128 bf16 in TMEM, queries [32h, 32h+32) at
      // columns a_col + 32h + [0,16); B = a [queries x D] tile as MN-major operand.
      auto ts = [&](uint32_t d_col, uint32_t a_col, uint32_t b0, bool acc) {
        const uint64_t db = make_smem_desc(b0, 16384, 1024, kSwizzle128B);
        const uint32_t ta = tmem + a_col;
#pragma unroll
        for (int g = 0; g < 2; ++g) {   // k-steps 4g .. 4g+3: A columns 64g + {0, 8, 32, 40}, B rows 2048 bytes apart
          mma_ts_x4_w<false>(tmem + d_col, ta + 64 * g, ta + 64 * g + 8, ta + 64 * g + 32,
                             ta + 64 * g + 40, db + 512 * g, db + 512 * g + 128,
                             db + 512 * g + 256, db + 512 * g + 384, C::kIdescTS,
                             (acc || g > 0) ? 1u : 0u);
        }
      };
      for (uint32_t k = 0; ok; ++k, ++uit) {
        const int u = take_unit(k, ok);
        if (u < 0) break;
        int bhk, j;
        unit(u, bhk, j);
        int i_lo, i_hi;
        bwd_qrange(j, p, i_lo, i_hi);
        const int T = p.group * (i_hi - i_lo + 1);
        if (!(ok = wait_w(bar(ctl.fix_full), uit & 1))) break;
        // Block t: Q item = base + 2t, dO item = base + 2t + 1.
        const uint32_t base = item;
        item += 2 * T;
        // prologue: S^T(0), dP^T(0)
        if (!(ok = wait_slot(base) && wait_slot(base + 1))) break;
        tc_fence_after();
        ss(0, sK, sRing + (base % C::kStages) * C::kTile, idesc_s);
        mma_commit_w(bar(ctl.s_full));
        ss(128, sV, sRing + ((base + 1) % C::kStages) * C::kTile, C::kIdescSS);
        mma_commit_w(bar(ctl.dp_full));
        for (int t = 0; t < T && ok; ++t, ++gblk) {
          const uint32_t iq = base + 2 * t, io = iq + 1;
          const uint32_t sQ = sRing + (iq % C::kStages) * C::kTile;
          const uint32_t sdO = sRing + (io % C::kStages) * C::kTile;
          // dV += P^T dO once P^T is written
          if (!(ok = wait_w(bar(ctl.p_ready), gblk & 1))) break;
          tc_fence_after();
          ts(256, 0, sdO, t > 0);
          mma_commit_w(bar(ctl.empty[io % C::kStages]));    // dO_i done (dP^T(t) was earlier)
          // S^T(t+1): the S^T columns are free once dV(t) has read P^T
          const bool more = t + 1 < T;
          if (more) {
            if (!(ok = wait_slot(iq + 2))) break;
            tc_fence_after();
            ss(0, sK, sRing + ((iq + 2) % C::kStages) * C::kTile, idesc_s);
            mma_commit_w(bar(ctl.s_full));   // P^T(t+1) can start during dK(t), dP^T(t+1)
          }
          // dK += dS^T Q once dS^T is written
          if (!(ok = wait_w(bar(ctl.ds_ready), gblk & 1))) break;
          tc_fence_after();
          ts(256 + D, 128, sQ, t > 0);
          mma_commit_w(bar(ctl.empty[iq % C::kStages]));    // Q_i done
          if (more) {
            if (!(ok = wait_slot(io + 2))) break;
            tc_fence_after();
            ss(128, sV, sRing + ((io + 2) % C::kStages) * C::kTile, C::kIdescSS);
            mma_commit_w(bar(ctl.dp_full));
          }
        }
        mma_commit_w(bar(ctl.unit_done));
        mma_commit_w(bar(ctl.fix_empty));
      }
      __syncwarp();
      mma_commit_w(bar(ctl.drain));
      wait_bounded(bar(ctl.drain), 0, wc, false);
    }
  } else {
    // ------------------------------------------------------------ element-wise
    const int qd = warp & 3;             // TMEM lane quarter: keys 32qd .. 32qd+31
    const int h = warp >> 2;             // queries [32h, 32h+32) of each block
    const int r = qd * 32 + lane;        // key row within the block
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    const float cl = p.scale_log2;
    const bool zero_scale = p.zero_scale != 0;
    uint32_t uit = 0, gblk = 0, item = 0;
    bool ok = true;
    for (uint32_t k = 0; ok; ++k, ++uit) {
      const int u = take_unit(k, ok);
      if (u < 0) break;
      int bhk, j;
      unit(u, bhk, j);
      int i_lo, i_hi;
      bwd_qrange(j, p, i_lo, i_hi);
      const int nI = i_hi - i_lo + 1;
      const int key = j * 128 + r;
      // L' and D of block t's queries 32h + lane, read from global memory one
      // block ahead (lane i holds query 32h + i; shuffles hand the values to the
      // other lanes): shared-memory loads queue behind the score products'
      // operand traffic for hundreds of cycles.
      const int T = p.group * nI;
      const int hb = bhk / p.Hk, hg = bhk - hb * p.Hk;
      auto stat_off = [&](int tt) {
        const int hh = tt / nI, ii = i_lo + (tt - hh * nI);
        return (size_t)(hb * p.H + hg * p.group + hh) * p.Npad + (size_t)ii * 128 + 32 * h + lane;
      };
      float l_next = 0.0f, d_next = 0.0f;
      if (T > 0) {
        l_next = __ldg(p.lp + stat_off(0));
        d_next = __ldg(p.dd + stat_off(0));
      }
      for (int t = 0; t < T; ++t, ++gblk, item += 2) {
        const int i = i_lo + (t - (t / nI) * nI);
        const float l_lane = l_next, d_lane = d_next;
        if (t + 1 < T) {
          l_next = __ldg(p.lp + stat_off(t + 1));
          d_next = __ldg(p.dd + stat_off(t + 1));
        }
        const int q0 = i * 128 + 32 * h;   // first query of this thread's columns
        // Mask needed unless every (key, query) of the block is visible.
        const bool full_vis = (!p.causal || j * 128 + 127 <= i * 128) &&
                              (p.window <= 0 || j * 128 > i * 128 + 127 - p.window);
        ok = wait_bounded(bar(ctl.s_full), gblk & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;   // a timed-out wait also set the abort flag every other wait honours
        tc_fence_after();
        // ---- phase A: P^T = exp2(S^T * c - L') for this thread's 32 queries
        float pr[32];
        {
          uint32_t sv[32];
          tmem_ld32(tmem + lane_off + 32 * h, sv);
          tmem_wait_ld();
          reg_fence(sv);
          if (!full_vis || zero_scale) {
            // Diagonal / window-edge block: 2^-inf = 0 for the invisible scores
            // (scale = 0: every visible score is 0).
#pragma unroll
            for (int col = 0; col < 32; ++col)
              sv[col] = !bwd_visible(key, q0 + col, p) ? 0xff800000u : (zero_scale ? 0u : sv[col]);
          }
          const uint64_t c2 = f32x2_pack(cl, cl);
          uint32_t pk[16];
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4) {
            const float4 L = make_float4(__shfl_sync(0xffffffffu, l_lane, 4 * v4),
                                         __shfl_sync(0xffffffffu, l_lane, 4 * v4 + 1),
                                         __shfl_sync(0xffffffffu, l_lane, 4 * v4 + 2),
                                         __shfl_sync(0xffffffffu, l_lane, 4 * v4 + 3));
            float a0, a1, a2, a3;
            f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(sv[4 * v4]), __uint_as_float(sv[4 * v4 + 1])), c2,
                                   f32x2_pack(-L.x, -L.y)), a0, a1);
            f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(sv[4 * v4 + 2]), __uint_as_float(sv[4 * v4 + 3])), c2,
                                   f32x2_pack(-L.z, -L.w)), a2, a3);
            pr[4 * v4] = ex2_approx(a0);
            pr[4 * v4 + 1] = ex2_approx(a1);
            pr[4 * v4 + 2] = ex2_approx(a2);
            pr[4 * v4 + 3] = ex2_approx(a3);
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(pr[2 * e], pr[2 * e + 1]);
          // P^T of queries [32h, +32) -> columns [32h, 32h+16): inside the S^T
          // columns this warp has already read.
          tmem_st16(tmem + lane_off + 32 * h, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(ctl.p_ready));
        // ---- phase B: dS^T = P^T o (dP^T - D), once dP^T is computed
        ok = wait_bounded(bar(ctl.dp_full), gblk & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t dv[32];
          tmem_ld32(tmem + lane_off + 128 + 32 * h, dv);
          tmem_wait_ld();
          reg_fence(dv);
          uint32_t pk[16];
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4) {
            const float Dd[4] = {__shfl_sync(0xffffffffu, d_lane, 4 * v4),
                                 __shfl_sync(0xffffffffu, d_lane, 4 * v4 + 1),
                                 __shfl_sync(0xffffffffu, d_lane, 4 * v4 + 2),
                                 __shfl_sync(0xffffffffu, d_lane, 4 * v4 + 3)};
            float ds[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) ds[e] = pr[4 * v4 + e] * (__uint_as_float(dv[4 * v4 + e]) - Dd[e]);
            pk[2 * v4] = pack_bf16x2(ds[0], ds[1]);
            pk[2 * v4 + 1] = pack_bf16x2(ds[2], ds[3]);
          }
          tmem_st16(tmem + lane_off + 128 + 32 * h, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(ctl.ds_ready));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      ok = wait_bounded(bar(ctl.unit_done), uit & 1, wc);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const bool live = key < p.N;
      constexpr int kW = D / 4;   // output columns of this thread: [kW h, kW h + kW)
      const size_t orow = ((size_t)bhk * p.N + key) * D + kW * h;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {   // dV, then dK (times scale)
        const float mul = which == 0 ? 1.0f : p.scale;
        uint16_t* dst_row = reinterpret_cast<uint16_t*>(which == 0 ? p.dv : p.dk) + orow;
        const uint32_t src = tmem + lane_off + 256 + which * D + kW * h;
        uint32_t pk[kW / 2];
        __syncwarp();
        if (kW == 32) {
          uint32_t av[32];
          tmem_ld32(src, av);
          tmem_wait_ld();
          reg_fence(av);
#pragma unroll
          for (int e = 0; e < kW / 2; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(av[2 * e]) * mul, __uint_as_float(av[2 * e + 1]) * mul);
        } else {
          uint32_t av[16];
          tmem_ld16(src, av);
          tmem_wait_ld();
          reg_fence(av);
#pragma unroll
          for (int e = 0; e < kW / 2; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(av[2 * e]) * mul, __uint_as_float(av[2 * e + 1]) * mul);
        }
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(dst_row);
#pragma unroll
          for (int e = 0; e < kW / 8; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
      tc_fence_before();   // accumulators read: the next unit's first products may overwrite them
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::kEW + 1) tmem_dealloc(tmem, C::kTmemCols);
}

// ============================================================================
// dQ: one unit = (batch * query head, 128-query block i).  Q_i and dO_i stay in
// TMEM for the whole unit (written by the element-wise warps from global
// memory), so S = Q K^T and dP = dO V^T are TS products that read only K_j and
// V_j from shared memory.  TMEM: Q [0, D/2), dO [D/2, D) (bf16 pairs), S
// [D, D+128), dP [D+128, D+256) with dS (bf16) written over it, dQ after that.
// ============================================================================
template <int D>
__global__ void __launch_bounds__(576, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const BwdParams p) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sRing = smem_addr(smem);   // K_j / V_j tiles, alternating
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](uint64_t& b) { return smem_addr(&b); };
  constexpr uint32_t kColQ = 0, kColdO = D / 2, kColS = D, kColDP = D + 128, kColDQ = D + 256;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStagesDQ; ++s) {
      mbar_init(bar(ctl.full[s]), 1);
      mbar_init(bar(ctl.empty[s]), 1);
    }
    mbar_init(bar(ctl.fix_full), C::kEW);   // Q_i, dO_i written into TMEM
    mbar_init(bar(ctl.s_full), 1);
    mbar_init(bar(ctl.dp_full), 1);
    mbar_init(bar(ctl.s_read), C::kEW);     // S read: its columns may be overwritten
    mbar_init(bar(ctl.p_ready), C::kEW);    // dS written
    mbar_init(bar(ctl.unit_done), 1);
    mbar_init(bar(ctl.drain), 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(bar(ctl.unit_full[s]), 1);
      mbar_init(bar(ctl.unit_empty[s]), C::kEW + 1);   // the MMA thread and the element-wise warps
    }
    ctl.abort_flag = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  if (warp == C::kEW + 1) {
    tmem_alloc(smem_addr(&ctl.tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const WaitCtx wc{&ctl.abort_flag, p.status ? p.status : &g_attn_status, p.timeout_ns};
  // Work units: the load warp takes the next index (atomic counter, or the
  // static stride without one) and passes it through a 4-entry ring; -1 ends.
  auto publish_unit = [&](uint32_t k, bool& ok) -> int {
    int u = p.sched ? atomicAdd(p.sched, 1) : static_cast<int>(blockIdx.x + k * gridDim.x);
    if (u >= p.num_units) u = -1;
    const uint32_t slot = k & 3;
    if (k >= 4 && !(ok = wait_bounded(bar(ctl.unit_empty[slot]), ((k >> 2) - 1) & 1, wc))) return -1;
    ctl.unit_ring[slot] = u;
    mbar_arrive(bar(ctl.unit_full[slot]));
    return u;
  };
  auto take_unit = [&](uint32_t k, bool& ok) -> int {   // a whole warp; lane 0 frees the slot
    const uint32_t slot = k & 3;
    ok = wait_bounded(bar(ctl.unit_full[slot]), (k >> 2) & 1, wc);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return -1;
    const int u = *reinterpret_cast<volatile int*>(&ctl.unit_ring[slot]);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(ctl.unit_empty[slot]));
    return u;
  };

  // Unit u -> (bh, i).  Causal: longest first (last query blocks of all heads).
  auto unit = [&](int u, int& bh, int& i) {
    if (p.causal) {
      bwd_causal_order(u, p.BH, p.nb, p.hgroup, false, bh, i);    // the last query block sees the most
    } else {
      bh = u / p.nb;
      i = u - bh * p.nb;
    }
  };
  auto kv_head = [&](int bh) {
    const int b = bh / p.H, hq = bh - (bh / p.H) * p.H;
    return b * p.Hk + hq / p.group;
  };

  if (warp == C::kEW) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      const uint64_t pol_ring = l2_policy_evict_last();
      uint32_t item = 0;
      bool ok = true;
      for (uint32_t k = 0; ok; ++k) {
        const int u = publish_unit(k, ok);
        if (u < 0) break;
        int bh, i;
        unit(u, bh, i);
        int j_lo, j_hi;
        bwd_krange(i, p, j_lo, j_hi);
        const int bhk = kv_head(bh);
        for (int jj = j_lo; jj <= j_hi && ok; ++jj) {
          for (int w2 = 0; w2 < 2 && ok; ++w2, ++item) {   // K_j, then V_j
            const uint32_t slot = item % C::kStagesDQ;
            if (!(ok = wait_bounded(bar(ctl.empty[slot]), ((item / C::kStagesDQ) & 1) ^ 1, wc))) break;
            mbar_arrive_expect_tx(bar(ctl.full[slot]), C::kTile);
            for (int s = 0; s < C::kSlabs; ++s)
              tma_load_3d_hint(sRing + slot * C::kTile + s * 16384, w2 == 0 ? &tmK : &tmV,
                               bar(ctl.full[slot]), s * 64, jj * 128, bhk, pol_ring);
          }
        }
      }
      const uint32_t issued = item;
      for (uint32_t s = 0; s < (uint32_t)C::kStagesDQ && s < issued; ++s) {
        const uint32_t last = s + ((issued - 1 - s) / C::kStagesDQ) * C::kStagesDQ;
        wait_bounded(bar(ctl.full[s]), (last / C::kStagesDQ) & 1, wc, false);
      }
    }
  } else if (warp == C::kEW + 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop converged; one elected lane issues each
    // MMA and commit (the *_w forms), every wait is taken by all lanes.
    {
      uint32_t item = 0, uit = 0, gblk = 0;
      auto wait_w = [&](uint32_t b, uint32_t parity) {
        return __all_sync(0xffffffffu, wait_bounded(b, parity, wc));
      };
      bool ok = true;
      auto wait_slot = [&](uint32_t it) {
        return wait_w(bar(ctl.full[it % C::kStagesDQ]), (it / C::kStagesDQ) & 1);
      };
      auto slot_addr = [&](uint32_t it) { return sRing + (it % C::kStagesDQ) * C::kTile; };
      // [128 rows in TMEM at a_col] x [128 rows of the K-major tile b0]^T over K = D,
      // four k-steps per election.
      // S = Q K^T negates K (its B operand) for a negative scale; dP does not.
      const uint32_t idesc_s = C::kIdescSS | (p.neg_scale ? kIdescNegateB : 0u);
      auto ts_k = [&](uint32_t d_col, uint32_t a_col, uint32_t b0, uint32_t idesc) {
        const uint64_t db = make_smem_desc(b0, 16, 1024, kSwizzle128B);
        const uint32_t ta = tmem + a_col;
#pragma unroll
        for (int g = 0; g < C::kSSteps / 4; ++g) {
          const uint64_t o = g * 1024;
          mma_ts_x4_w<false>(tmem + d_col, ta + 32 * g, ta + 32 * g + 8, ta + 32 * g + 16,
                             ta + 32 * g + 24, db + o, db + o + 2, db + o + 4, db + o + 6,
                             idesc, g > 0 ? 1u : 0u);
        }
      };
      // [128 x 128 bf16 in TMEM at a_col, keys [32h, 32h+32) at columns a_col +
      // 32h + [0,16)] x [MN-major K tile b0]
      auto ts_mn = [&](uint32_t d_col, uint32_t a_col, uint32_t b0, bool acc) {
        const uint64_t db = make_smem_desc(b0, 16384, 1024, kSwizzle128B);
        const uint32_t ta = tmem + a_col;
#pragma unroll
        for (int g = 0; g < 2; ++g)
          mma_ts_x4_w<false>(tmem + d_col, ta + 64 * g, ta + 64 * g + 8, ta + 64 * g + 32,
                             ta + 64 * g + 40, db + 512 * g, db + 512 * g + 128,
                             db + 512 * g + 256, db + 512 * g + 384, C::kIdescTS,
                             (acc || g > 0) ? 1u : 0u);
      };
      for (uint32_t k = 0; ok; ++k, ++uit) {
        const int u = take_unit(k, ok);
        if (u < 0) break;
        int bh, i;
        unit(u, bh, i);
        int j_lo, j_hi;
        bwd_krange(i, p, j_lo, j_hi);
        const int J = j_hi - j_lo + 1;
        if (!(ok = wait_w(bar(ctl.fix_full), uit & 1))) break;   // Q_i, dO_i in TMEM
        const uint32_t base = item;            // K_j item = base + 2jj, V_j = base + 2jj + 1
        item += 2 * J;
        if (!(ok = wait_slot(base) && wait_slot(base + 1))) break;
        tc_fence_after();
        ts_k(kColS, kColQ, slot_addr(base), idesc_s);
        mma_commit_w(bar(ctl.s_full));
        ts_k(kColDP, kColdO, slot_addr(base + 1), C::kIdescSS);
        mma_commit_w(bar(ctl.dp_full));
        mma_commit_w(bar(ctl.empty[(base + 1) % C::kStagesDQ]));   // V_0 done
        for (int jj = 0; jj < J && ok; ++jj, ++gblk) {
          const uint32_t ik = base + 2 * jj;
          const bool more = jj + 1 < J;
          // S(jj+1) once the element-wise pass has read S(jj)
          if (more) {
            if (!(ok = wait_w(bar(ctl.s_read), gblk & 1) && wait_slot(ik + 2))) break;
            tc_fence_after();
            ts_k(kColS, kColQ, slot_addr(ik + 2), idesc_s);
            mma_commit_w(bar(ctl.s_full));
          }
          // dQ += dS K_j once dS is written (over dP)
          if (!(ok = wait_w(bar(ctl.p_ready), gblk & 1))) break;
          tc_fence_after();
          ts_mn(kColDQ, kColDP, slot_addr(ik), jj > 0);
          mma_commit_w(bar(ctl.empty[ik % C::kStagesDQ]));   // K_j done
          // dP(jj+1) over dS(jj): after dQ(jj) in issue order
          if (more) {
            if (!(ok = wait_slot(ik + 3))) break;
            tc_fence_after();
            ts_k(kColDP, kColdO, slot_addr(ik + 3), C::kIdescSS);
            mma_commit_w(bar(ctl.dp_full));
            mma_commit_w(bar(ctl.empty[(ik + 3) % C::kStagesDQ]));   // V_{jj+1} done
          }
        }
        mma_commit_w(bar(ctl.unit_done));
      }
      __syncwarp();
      mma_commit_w(bar(ctl.drain));
      wait_bounded(bar(ctl.drain), 0, wc, false);
    }
  } else {
    // ------------------------------------------------------------ element-wise
    const int qd = warp & 3;             // TMEM lane quarter: queries 32qd .. 32qd+31
    const int h = warp >> 2;             // keys [32h, 32h+32) of each block; head dims [D/4 h, +D/4)
    const int r = qd * 32 + lane;        // query row within the block
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    const float cl = p.scale_log2;
    const bool zero_scale = p.zero_scale != 0;
    uint32_t uit = 0, gblk = 0;
    bool ok = true;
    for (uint32_t k = 0; ok; ++k, ++uit) {
      const int u = take_unit(k, ok);
      if (u < 0) break;
      int bh, i;
      unit(u, bh, i);
      int j_lo, j_hi;
      bwd_krange(i, p, j_lo, j_hi);
      const int q = i * 128 + r;
      const float Lq = __ldg(p.lp + (size_t)bh * p.Npad + q);   // +inf past N: P = 0
      const float Dq = __ldg(p.dd + (size_t)bh * p.Npad + q);
      // Q_i and dO_i rows into TMEM (zeros past N).  The previous unit's products
      // that read them are complete: its unit_done was waited for.
      {
        constexpr int kE = D / 4;   // elements of this thread: [kE h, kE h + kE)
        uint32_t qv[kE / 2], ov[kE / 2];
        if (q < p.N) {
          const uint4* sq = reinterpret_cast<const uint4*>(p.q + ((size_t)bh * p.N + q) * D + kE * h);
          const uint4* so = reinterpret_cast<const uint4*>(p.dO + ((size_t)bh * p.N + q) * D + kE * h);
#pragma unroll
          for (int e = 0; e < kE / 8; ++e) {
            const uint4 a = __ldg(sq + e), c = __ldg(so + e);
            qv[4 * e] = a.x; qv[4 * e + 1] = a.y; qv[4 * e + 2] = a.z; qv[4 * e + 3] = a.w;
            ov[4 * e] = c.x; ov[4 * e + 1] = c.y; ov[4 * e + 2] = c.z; ov[4 * e + 3] = c.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < kE / 2; ++e) qv[e] = ov[e] = 0u;
        }
        if (kE == 32) {
          tmem_st16(tmem + lane_off + kColQ + 16 * h, *reinterpret_cast<const uint32_t(*)[16]>(qv));
          tmem_st16(tmem + lane_off + kColdO + 16 * h, *reinterpret_cast<const uint32_t(*)[16]>(ov));
        } else {
          tmem_st8(tmem + lane_off + kColQ + 8 * h, *reinterpret_cast<const uint32_t(*)[8]>(qv));
          tmem_st8(tmem + lane_off + kColdO + 8 * h, *reinterpret_cast<const uint32_t(*)[8]>(ov));
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(ctl.fix_full));
      }
      for (int jj = j_lo; jj <= j_hi; ++jj, ++gblk) {
        const int k0 = jj * 128 + 32 * h;   // first key of this thread's columns
        const bool full_vis = (jj * 128 + 127 < p.N) && (!p.causal || jj * 128 + 127 <= i * 128) &&
                              (p.window <= 0 || jj * 128 > i * 128 + 127 - p.window);
        // Exponentials as soon as S is there; dS once dP is there too.
        ok = wait_bounded(bar(ctl.s_full), gblk & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;   // a timed-out wait also set the abort flag every other wait honours
        tc_fence_after();
        float pr[32];
        {
          uint32_t sv[32];
          tmem_ld32(tmem + lane_off + kColS + 32 * h, sv);
          tmem_wait_ld();
          reg_fence(sv);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(ctl.s_read));   // S(jj+1) may overwrite S now
          if (!full_vis || zero_scale) {
            // Diagonal / window-edge / ragged block: 2^-inf = 0 for invisible scores
            // (scale = 0: every visible score is 0).
#pragma unroll
            for (int col = 0; col < 32; ++col)
              sv[col] = !bwd_visible(k0 + col, q, p) ? 0xff800000u : (zero_scale ? 0u : sv[col]);
          }
          const uint64_t c2 = f32x2_pack(cl, cl);
          const uint64_t nl2 = f32x2_pack(-Lq, -Lq);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float a0, a1;
            f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), c2, nl2),
                         a0, a1);
            pr[2 * e] = ex2_approx(a0);
            pr[2 * e + 1] = ex2_approx(a1);
          }
        }
        ok = wait_bounded(bar(ctl.dp_full), gblk & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t dv[32];
        tmem_ld32(tmem + lane_off + kColDP + 32 * h, dv);
        tmem_wait_ld();
        reg_fence(dv);
        const uint64_t nd2 = f32x2_pack(-Dq, -Dq);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float g0, g1;
          f32x2_unpack(f32x2_add(f32x2_pack(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1])), nd2), g0, g1);
          pk[e] = pack_bf16x2(pr[2 * e] * g0, pr[2 * e + 1] * g1);
        }
        // dS of keys [32h, +32) -> columns [32h, 32h+16) of the dP region (read above)
        tmem_st16(tmem + lane_off + kColDP + 32 * h, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(ctl.p_ready));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      ok = wait_bounded(bar(ctl.unit_done), uit & 1, wc);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const bool live = q < p.N;
      constexpr int kW = D / 4;   // output columns of this thread: [kW h, kW h + kW)
      uint16_t* dst_row = reinterpret_cast<uint16_t*>(p.dq) + ((size_t)bh * p.N + q) * D + kW * h;
      const uint32_t src = tmem + lane_off + kColDQ + kW * h;
      uint32_t pk[kW / 2];
      __syncwarp();
      if (kW == 32) {
        uint32_t av[32];
        tmem_ld32(src, av);
        tmem_wait_ld();
        reg_fence(av);
#pragma unroll
        for (int e = 0; e < kW / 2; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(av[2 * e]) * p.scale, __uint_as_float(av[2 * e + 1]) * p.scale);
      } else {
        uint32_t av[16];
        tmem_ld16(src, av);
        tmem_wait_ld();
        reg_fence(av);
#pragma unroll
        for (int e = 0; e < kW / 2; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(av[2 * e]) * p.scale, __uint_as_float(av[2 * e + 1]) * p.scale);
      }
      if (live) {
        uint4* dst = reinterpret_cast<uint4*>(dst_row);
#pragma unroll
        for (int e = 0; e < kW / 8; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::kEW + 1) tmem_dealloc(tmem, C::kTmemCols);
}

// ============================================================================
// Preprocessing: D_i = rowdot(dO_i, O_i) and L'_i = L_i * log2(e), padded to
// Npad rows (L' = +inf, D = 0 past N so that padded queries get P = 0).  One
// warp per row.
// ============================================================================
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const uint16_t* __restrict__ o,
                                                            const uint16_t* __restrict__ dO,
                                                            const float* __restrict__ lse,
                                                            float* __restrict__ lp, float* __restrict__ dd,
                                                            int N, int Npad, long long rows_pad) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows_pad) return;
  const long long bh = row / Npad;
  const int n = static_cast<int>(row - bh * Npad);
  float acc = 0.0f;
  if (n < N) {
    const size_t base = ((size_t)bh * N + n) * D;
    constexpr int V = D / 32;   // elements per lane (4 or 2)
    const uint16_t* po = o + base + V * lane;
    const uint16_t* pd = dO + base + V * lane;
#pragma unroll
    for (int e = 0; e < V; ++e)
      acc = fmaf(__uint_as_float(static_cast<uint32_t>(po[e]) << 16),
                 __uint_as_float(static_cast<uint32_t>(pd[e]) << 16), acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    dd[row] = acc;
    lp[row] = n < N ? lse[(size_t)bh * N + n] * 1.4426950408889634f : __int_as_float(0x7f800000);
  }
}

}  // namespace gb300
