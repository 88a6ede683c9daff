// Prefill kernel instantiations for e4m3 Q with e4m3 K/V at (Dk, Dv) =
// (128, 128) and (192, 128): the converter-warp kernel with its QK on the
// e4m3 bytes (kind::f8f6f4), in a translation unit of its own so that the
// build compiles it in parallel with the others.
#include "fa_prefill3_launch.cuh"

namespace fa {
cudaError_t launch_prefill_128_128_q8(const PrefillLaunch &L) { return launch_prefill3<128, 128, true, false, true>(L); }
cudaError_t launch_prefill_192_128_q8(const PrefillLaunch &L) { return launch_prefill3<192, 128, true, false, true>(L); }
}  // namespace fa
