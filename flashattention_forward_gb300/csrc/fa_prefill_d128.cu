// Prefill kernel instantiations for (Dk, Dv) = (128, 128): the two-query-tile
// ping-pong kernel for bf16 K/V; e4m3 K/V runs its converter-warp form.
#include "fa_prefill2.cuh"
#include "fa_prefill3_launch.cuh"

namespace fa {
namespace {
// The 12-warp variant raises the softmax warps to Cfg::kRegsSoftmax registers
// with setmaxnreg.inc, which waits until other warps of the CTA release
// registers.  It is launched only when the compiled launch register count
// makes the whole split fit the CTA's pool; otherwise the 10-warp variant runs.
template <bool PAGED, int MOD>
bool bigreg_fits() {
  using Big = Prefill2Cfg<128, 128, PAGED, MOD, true>;
  static int verdict = -1;   // per process: all devices run the same binary
  if (verdict < 0) {
    cudaFuncAttributes a;
    const bool ok = cudaFuncGetAttributes(&a, fa_prefill2_kernel<128, 128, PAGED, MOD, true>) == cudaSuccess &&
                    a.numRegs >= Big::kMinLaunchRegs && a.numRegs * Big::kThreads >=
                    8 * 32 * Big::kRegsSoftmax + 4 * 32 * Big::kRegsOther;
    verdict = ok ? 1 : 0;
  }
  return verdict == 1;
}

template <bool PAGED, int MOD, bool BIG>
cudaError_t launch_one(const PrefillLaunch &L) {
  using Cfg = Prefill2Cfg<128, 128, PAGED, MOD, BIG>;
  static unsigned long long done = 0;
  auto kern = fa_prefill2_kernel<128, 128, PAGED, MOD, BIG>;
  cudaError_t e = ensure_smem_attr(kern, Cfg::kSmemBytes, &done);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, Cfg::kThreads, Cfg::kSmemBytes, L.stream>>>(L.tm_q, L.tm_k, L.tm_v, L.p);
  return cudaGetLastError();
}
template <bool PAGED, int MOD>
cudaError_t pick(const PrefillLaunch &L) {
  if (L.variant != 1 && bigreg_fits<PAGED, MOD>()) return launch_one<PAGED, MOD, true>(L);
  return launch_one<PAGED, MOD, false>(L);
}
template <bool PAGED>
cudaError_t by_mod(const PrefillLaunch &L) {
  switch (L.mod) {
    case 0: return pick<PAGED, 0>(L);
    case 1: return pick<PAGED, 1>(L);
    default: return pick<PAGED, 2>(L);
  }
}
}  // namespace

cudaError_t launch_prefill_128_128(const PrefillLaunch &L) {
  if (L.fp8) {   // byte K/V
    if (L.q8) return launch_prefill_128_128_q8(L);
    return L.int8 ? launch_prefill_128_128_i8(L) : launch_prefill3<128, 128, true>(L);
  }
  return L.paged ? by_mod<true>(L) : by_mod<false>(L);
}
}  // namespace fa
