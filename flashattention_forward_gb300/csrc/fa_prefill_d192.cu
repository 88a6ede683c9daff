// Prefill kernel instantiations for (Dk, Dv) = (192, 128): the chunked-ring
// ping-pong kernel, bf16 K/V.
#include "fa_prefill3_launch.cuh"

namespace fa {
cudaError_t launch_prefill_192_128(const PrefillLaunch &L) {
  if (L.fp8) return launch_prefill_192_128_fp8(L);
  return launch_prefill3<192, 128, false>(L);
}
}  // namespace fa
