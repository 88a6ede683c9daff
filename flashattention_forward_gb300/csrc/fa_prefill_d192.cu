// Prefill kernel instantiations for (Dk, Dv) = (192, 128): the single-query-
// tile kernel, bf16 or e4m3 K/V.
#include "fa_prefill1_launch.cuh"

namespace fa {
cudaError_t launch_prefill_192_128(const PrefillLaunch &L) {
  if (L.fp8) return launch_prefill1_fp8<192, 128>(L);
  return L.paged ? launch_prefill1_mod<192, 128, true, false>(L) : launch_prefill1_mod<192, 128, false, false>(L);
}
}  // namespace fa
