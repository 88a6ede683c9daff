// Prefill kernel instantiations for (Dk, Dv) = (128, 128): the two-query-tile
// ping-pong kernel for bf16 K/V; e4m3 K/V runs its converter-warp form.
#include "fa_prefill2_launch.cuh"
#include "fa_prefill3_launch.cuh"

namespace fa {
cudaError_t launch_prefill_128_128(const PrefillLaunch &L) {
  if (L.fp8) {   // byte K/V
    if (L.q8) return launch_prefill_128_128_q8(L);
    return L.int8 ? launch_prefill_128_128_i8(L) : launch_prefill3<128, 128, true>(L);
  }
  return L.paged ? prefill2_by_mod<128, true>(L) : prefill2_by_mod<128, false>(L);
}
}  // namespace fa
