// Launcher of the two-query-tile ping-pong kernel (fa_prefill2.cuh), shared
// by the translation units that instantiate it for one head dim each.
#pragma once
#include "fa_internal.h"
#include "fa_prefill2.cuh"

namespace fa {

// The 12-warp variant raises the softmax warps to Cfg::kRegsSoftmax registers
// with setmaxnreg.inc, which waits until other warps of the CTA release
// registers.  It is launched only when the compiled launch register count
// makes the whole split fit the CTA's pool; otherwise the 10-warp variant runs.
template <int D, bool PAGED, int MOD, int NT = 2>
bool prefill2_bigreg_fits() {
  using Big = Prefill2Cfg<D, D, PAGED, MOD, true, NT>;
  static int fits = -1;   // per process: all devices run the same binary
  if (fits < 0) {
    cudaFuncAttributes a;
    const bool ok = cudaFuncGetAttributes(&a, fa_prefill2_kernel<D, D, PAGED, MOD, true, NT>) == cudaSuccess &&
                    a.numRegs >= Big::kMinLaunchRegs && a.numRegs * Big::kThreads >= Big::kPoolNeeded;
    fits = ok ? 1 : 0;
  }
  return fits == 1;
}

template <int D, bool PAGED, int MOD, bool BIG, int NT = 2>
cudaError_t prefill2_launch_one(const PrefillLaunch &L) {
  using Cfg = Prefill2Cfg<D, D, PAGED, MOD, BIG, NT>;
  static unsigned long long done = 0;
  auto kern = fa_prefill2_kernel<D, D, PAGED, MOD, BIG, NT>;
  cudaError_t e = ensure_smem_attr(kern, Cfg::kSmemBytes, &done);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, Cfg::kThreads, Cfg::kSmemBytes, L.stream>>>(L.tm_q, L.tm_k, L.tm_v, L.p);
  return cudaGetLastError();
}

template <int D, bool PAGED, int MOD>
cudaError_t prefill2_pick(const PrefillLaunch &L) {
  if constexpr (MOD == 5) {   // the one-pass softmax only
    if (!prefill2_bigreg_fits<D, PAGED, MOD>()) return cudaErrorNotSupported;
    return prefill2_launch_one<D, PAGED, MOD, true>(L);
  } else {
    if (L.variant != 1 && prefill2_bigreg_fits<D, PAGED, MOD>()) return prefill2_launch_one<D, PAGED, MOD, true>(L);
    return prefill2_launch_one<D, PAGED, MOD, false>(L);
  }
}

// MOD 0 plain, 1 ALiBi, 2 soft-cap; 3 and 4 (a prologue's per-key score
// term) are instantiated in fa_prefill_kt.cu.
// One query tile per CTA, two CTAs per SM (L.tiles_per_cta == 1; MOD 0-2):
// instantiated in fa_prefill_t1.cu.
template <int D, bool PAGED, int MOD>
cudaError_t prefill2_launch_t1(const PrefillLaunch &L) {
  if (!prefill2_bigreg_fits<D, PAGED, MOD, 1>()) return cudaErrorNotSupported;
  return prefill2_launch_one<D, PAGED, MOD, true, 1>(L);
}

template <int D, bool PAGED>
cudaError_t prefill2_by_mod(const PrefillLaunch &L) {
  if (L.tiles_per_cta == 1) return launch_prefill2_t1(D, L);
  switch (L.mod) {
    case 0: return prefill2_pick<D, PAGED, 0>(L);
    case 1: return prefill2_pick<D, PAGED, 1>(L);
    case 2: return prefill2_pick<D, PAGED, 2>(L);
    case 5: return prefill2_pick<D, PAGED, 5>(L);
    default: return launch_prefill2_kt(D, L);
  }
}

}  // namespace fa
