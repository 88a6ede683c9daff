// Chunked-ring prefill kernels with the per-key score term of a prologue's Q
// add (MOD 3, 4) for int8 caches at every head-dim pair.
#include "fa_prefill3_launch.cuh"

namespace fa {
cudaError_t launch_prefill3_kt_i8(int dk, const PrefillLaunch &L) {
  if (dk == 64) return launch_prefill3_kt_one<64, 64, true, true>(L);
  if (dk == 128) return launch_prefill3_kt_one<128, 128, true, true>(L);
  return launch_prefill3_kt_one<192, 128, true, true>(L);
}
}  // namespace fa
