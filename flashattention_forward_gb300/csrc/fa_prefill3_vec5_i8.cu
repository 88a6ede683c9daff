// Chunked-ring prefill kernels for int8 caches in the vectorized 5-D page
// layouts at every head-dim pair.
#include "fa_prefill3_launch.cuh"

namespace fa {
cudaError_t launch_prefill3_vec5_i8(int dk, const PrefillLaunch &L) {
  if (dk == 64) return launch_prefill3_vec5_one<64, 64, true>(L);
  if (dk == 128) return launch_prefill3_vec5_one<128, 128, true>(L);
  return launch_prefill3_vec5_one<192, 128, true>(L);
}
}  // namespace fa
