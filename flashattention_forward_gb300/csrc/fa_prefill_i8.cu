// Prefill kernel instantiations for int8 K/V caches with per-token scales (the
// converter-warp kernel, every head-dim pair), in a translation unit of their
// own so that the build compiles them in parallel with the others.
#include "fa_prefill3_launch.cuh"

namespace fa {
cudaError_t launch_prefill_64_64_i8(const PrefillLaunch &L) { return launch_prefill3<64, 64, true, true>(L); }
cudaError_t launch_prefill_128_128_i8(const PrefillLaunch &L) { return launch_prefill3<128, 128, true, true>(L); }
cudaError_t launch_prefill_192_128_i8(const PrefillLaunch &L) { return launch_prefill3<192, 128, true, true>(L); }
}  // namespace fa
