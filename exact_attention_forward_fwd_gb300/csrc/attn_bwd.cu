// Instantiation and launch of the attention backward (head dims 64 and 128).
#include "attn_bwd.cuh"
#include "launchers.h"

namespace gb300 {

namespace {

template <int D>
cudaError_t run_bwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                    const CUtensorMap& dO, const BwdParams& base, const void* o, const void* dO_ptr,
                    const float* lse, float* lp, float* dd, int sms, cudaStream_t stream) {
  using C = BCfg<D>;
  const long long rows_pad = static_cast<long long>(base.BH) * base.Npad;
  const long long blocks = (rows_pad + 7) / 8;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  attn_bwd_prep_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      reinterpret_cast<const uint16_t*>(o), reinterpret_cast<const uint16_t*>(dO_ptr), lse, lp, dd,
      base.N, base.Npad, rows_pad);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kdkdv = attn_bwd_dkdv_kernel<D>;
  auto kdq = attn_bwd_dq_kernel<D>;
  if ((e = cudaFuncSetAttribute(kdkdv, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(kdq, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytesDQ)) !=
          cudaSuccess)
    return e;
  // Causal order: groups of heads whose streamed tiles (Q and dO of all the
  // query heads of a KV head for dK/dV; K and V for dQ) take at most 48 MiB.
  const long long per_head = 4LL * base.N * 128;
  auto group_of = [&](long long bytes, int heads) {
    long long hg = (48LL << 20) / (bytes > 0 ? bytes : 1);
    return static_cast<int>(hg < 1 ? 1 : (hg > heads ? heads : hg));
  };
  BwdParams p1 = base;
  p1.num_units = base.BHk * base.nb;
  p1.hgroup = group_of(per_head * base.group, base.BHk);
  if ((e = unit_counter(stream, &p1.sched)) != cudaSuccess) return e;
  const int g1 = p1.num_units < sms ? p1.num_units : sms;
  kdkdv<<<g1, C::kThreads, C::kSmemBytes, stream>>>(q, k, v, dO, p1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  BwdParams p2 = base;
  p2.num_units = base.BH * base.nb;
  p2.hgroup = group_of(per_head, base.BH);
  if ((e = unit_counter(stream, &p2.sched)) != cudaSuccess) return e;
  const int g2 = p2.num_units < sms ? p2.num_units : sms;
  kdq<<<g2, C::kThreads, C::kSmemBytesDQ, stream>>>(q, k, v, dO, p2);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dO, const BwdParams& p, const void* o,
                            const void* dO_ptr, const float* lse, float* lp, float* dd, int sms,
                            cudaStream_t stream) {
  return d == 64 ? run_bwd<64>(q, k, v, dO, p, o, dO_ptr, lse, lp, dd, sms, stream)
                 : run_bwd<128>(q, k, v, dO, p, o, dO_ptr, lse, lp, dd, sms, stream);
}

int status_attn_bwd(bool clear) { return read_tu_status(clear); }

}  // namespace gb300
