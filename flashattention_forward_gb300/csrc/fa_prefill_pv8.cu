// Chunked-ring prefill kernels with e4m3 Q and the opt-in e4m3 P * V (P in
// e4m3 in shared memory, V transposed to a K-major e4m3 operand): Dk 128 and
// 192, Dv 128, plain, ALiBi and soft-cap scores, packed or paged.
#include "fa_prefill3_launch.cuh"

namespace fa {
cudaError_t launch_prefill3_pv8(int dk, const PrefillLaunch &L) {
  if (dk == 128) return launch_prefill3_pv8_one<128>(L);
  if (dk == 192) return launch_prefill3_pv8_one<192>(L);
  return cudaErrorNotSupported;
}
}  // namespace fa
