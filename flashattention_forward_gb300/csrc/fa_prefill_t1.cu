// Ping-pong prefill kernels with one 128-row query tile per CTA, so that two
// CTAs share an SM (bf16 K/V, Dk = Dv in {64, 128}, plain, ALiBi, soft-cap
// and ALiBi with its bias in the contraction (MOD 5), packed or paged K/V
// with pages of >= 16 keys).
#include "fa_prefill2_launch.cuh"

namespace fa {
template <int D, bool PAGED>
static cudaError_t t1_by_mod(const PrefillLaunch &L) {
  switch (L.mod) {
    case 0: return prefill2_launch_t1<D, PAGED, 0>(L);
    case 1: return prefill2_launch_t1<D, PAGED, 1>(L);
    case 2: return prefill2_launch_t1<D, PAGED, 2>(L);
    case 5: return prefill2_launch_t1<D, PAGED, 5>(L);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_prefill2_t1(int d, const PrefillLaunch &L) {
  if (d == 64) return L.paged ? t1_by_mod<64, true>(L) : t1_by_mod<64, false>(L);
  if (d == 128) return L.paged ? t1_by_mod<128, true>(L) : t1_by_mod<128, false>(L);
  return cudaErrorNotSupported;
}
}  // namespace fa
