// Prefill kernel instantiations for (Dk, Dv) = (128, 128): the two-query-tile
// ping-pong kernel (bf16 K/V).
#include "fa_internal.h"
#include "fa_prefill2.cuh"

namespace fa {
namespace {
template <bool PAGED, int MOD>
cudaError_t launch_one(const PrefillLaunch &L) {
  using Cfg = Prefill2Cfg<128, 128, PAGED, MOD>;
  static unsigned long long done = 0;
  auto kern = fa_prefill2_kernel<128, 128, PAGED, MOD>;
  cudaError_t e = ensure_smem_attr(kern, Cfg::kSmemBytes, &done);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, Cfg::kThreads, Cfg::kSmemBytes, L.stream>>>(L.tm_q, L.tm_k, L.tm_v, L.p);
  return cudaGetLastError();
}
template <bool PAGED>
cudaError_t by_mod(const PrefillLaunch &L) {
  switch (L.mod) {
    case 0: return launch_one<PAGED, 0>(L);
    case 1: return launch_one<PAGED, 1>(L);
    default: return launch_one<PAGED, 2>(L);
  }
}
}  // namespace

cudaError_t launch_prefill_128_128(const PrefillLaunch &L) {
  if (L.fp8) return cudaErrorNotSupported;
  return L.paged ? by_mod<true>(L) : by_mod<false>(L);
}
}  // namespace fa
