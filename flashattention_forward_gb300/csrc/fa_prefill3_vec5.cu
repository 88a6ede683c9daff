// Chunked-ring prefill kernels for e4m3 caches in the vectorized 5-D page
// layouts (K [N_pg, Hkv, Dk/16, P_s, 16], V [N_pg, Hkv, P_s/16, Dv, 16]) at
// every head-dim pair; int8 caches in fa_prefill3_vec5_i8.cu.
#include "fa_prefill3_launch.cuh"

namespace fa {
cudaError_t launch_prefill3_vec5(int dk, bool i8, const PrefillLaunch &L) {
  if (i8) return launch_prefill3_vec5_i8(dk, L);
  if (dk == 64) return launch_prefill3_vec5_one<64, 64, false>(L);
  if (dk == 128) return launch_prefill3_vec5_one<128, 128, false>(L);
  return launch_prefill3_vec5_one<192, 128, false>(L);
}
}  // namespace fa
