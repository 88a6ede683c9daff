// Ping-pong prefill kernels with the per-key score term of a prologue's Q add
// (MOD 3: the general score with ALiBi, whose slope may be 0; MOD 4: the
// soft-cap), bf16 K/V at Dk = Dv in {64, 128}.  A translation unit of their
// own: the kernels without the term carry no trace of it.
#include "fa_prefill2_launch.cuh"

namespace fa {
namespace {
template <int D>
cudaError_t kt(const PrefillLaunch &L) {
  if (L.paged) return L.mod == 3 ? prefill2_pick<D, true, 3>(L) : prefill2_pick<D, true, 4>(L);
  return L.mod == 3 ? prefill2_pick<D, false, 3>(L) : prefill2_pick<D, false, 4>(L);
}
}  // namespace

cudaError_t launch_prefill2_kt(int d, const PrefillLaunch &L) {
  if (L.mod != 3 && L.mod != 4) return cudaErrorInvalidValue;
  return d == 64 ? kt<64>(L) : kt<128>(L);
}
}  // namespace fa
