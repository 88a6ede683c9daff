// Backward-pass kernel instantiations (Dk = Dv in {64, 128}) and launchers.
#include "fa_bwd.cuh"
#include "fa_internal.h"

namespace fa {
namespace {
template <int D, int MOD, bool BM>
cudaError_t launch_d(const BwdLaunch &L) {
  using Cfg = BwdCfg<D>;
  constexpr int kSmem = Cfg::kSmemBytes;
  static unsigned long long done_dq = 0, done_kv = 0;
  cudaError_t e = ensure_smem_attr(fa_bwd_dq_kernel<D, MOD, BM>, kSmem, &done_dq);
  if (e == cudaSuccess) e = ensure_smem_attr(fa_bwd_dkdv_kernel<D, MOD, BM>, kSmem, &done_kv);
  if (e != cudaSuccess) return e;
  fa_bwd_delta_kernel<<<L.delta_blocks, 256, 0, L.stream>>>(L.dp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fa_bwd_dkdv_kernel<D, MOD, BM><<<L.grid_kv, Cfg::kThreads, kSmem, L.stream>>>(L.tm_q, L.tm_k, L.tm_v, L.tm_do, L.p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fa_bwd_dq_kernel<D, MOD, BM><<<L.grid_q, Cfg::kThreads, kSmem, L.stream>>>(L.tm_q, L.tm_k, L.tm_v, L.tm_do, L.p);
  return cudaGetLastError();
}
template <int D, bool BM>
cudaError_t by_mod(const BwdLaunch &L) {
  if (L.mod == 1) return launch_d<D, 1, BM>(L);
  if (L.mod == 2) return launch_d<D, 2, BM>(L);
  return launch_d<D, 0, BM>(L);
}
template <int D>
cudaError_t by_mask(const BwdLaunch &L) {
  return L.p.block_mask ? by_mod<D, true>(L) : by_mod<D, false>(L);
}
}  // namespace

cudaError_t launch_bwd(int d, const BwdLaunch &L) {
  return d == 64 ? by_mask<64>(L) : by_mask<128>(L);
}
}  // namespace fa
