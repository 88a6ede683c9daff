// Prefill kernel instantiations for (Dk, Dv) = (64, 64): the two-query-tile
// ping-pong kernel for bf16 K/V; e4m3 K/V runs its converter-warp form.
#include "fa_prefill2_launch.cuh"
#include "fa_prefill3_launch.cuh"

namespace fa {
cudaError_t launch_prefill_64_64(const PrefillLaunch &L) {
  if (L.fp8) return L.int8 ? launch_prefill_64_64_i8(L) : launch_prefill3<64, 64, true>(L);   // byte K/V
  return L.paged ? prefill2_by_mod<64, true>(L) : prefill2_by_mod<64, false>(L);
}
}  // namespace fa
