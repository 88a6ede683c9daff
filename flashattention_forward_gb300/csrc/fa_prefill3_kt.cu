// Chunked-ring prefill kernels with the per-key score term of a prologue's Q
// add (MOD 3, 4): bf16 K/V at Dk 192 and e4m3 caches at every head-dim pair.
#include "fa_prefill3_launch.cuh"

namespace fa {
cudaError_t launch_prefill3_kt(int dk, bool fp8, const PrefillLaunch &L) {
  if (!fp8) return launch_prefill3_kt_one<192, 128, false, false>(L);
  if (dk == 64) return launch_prefill3_kt_one<64, 64, true, false>(L);
  if (dk == 128) return launch_prefill3_kt_one<128, 128, true, false>(L);
  return launch_prefill3_kt_one<192, 128, true, false>(L);
}
}  // namespace fa
