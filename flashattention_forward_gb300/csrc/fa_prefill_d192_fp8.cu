// Prefill kernel instantiations for (Dk, Dv) = (192, 128) with e4m3 K/V (the
// chunked-ring kernel with converter warps), in a translation unit of their own
// so that the build compiles them in parallel with the bf16 ones.
#include "fa_prefill3_launch.cuh"

namespace fa {
cudaError_t launch_prefill_192_128_fp8(const PrefillLaunch &L) {
  if (L.q8) return launch_prefill_192_128_q8(L);
  return L.int8 ? launch_prefill_192_128_i8(L) : launch_prefill3<192, 128, true>(L);
}
}  // namespace fa
