// Launcher of the single-query-tile kernel (fa_prefill.cuh), shared by the
// per-head-dim translation units: bf16 K/V for Dk = 192, e4m3 K/V for all Dk.
#pragma once
#include "fa_internal.h"

namespace fa {

template <int DK, int DV, bool PAGED, bool FP8, int MOD>
cudaError_t launch_prefill1_one(const PrefillLaunch &L) {
  using Cfg = PrefillCfg<DK, DV, PAGED, FP8, MOD>;
  static unsigned long long done = 0;
  auto kern = fa_prefill_kernel<DK, DV, PAGED, FP8, MOD>;
  if constexpr (FP8) {
    // The e4m3 variant moves registers between warpgroups with setmaxnreg;
    // setmaxnreg.inc waits for registers that other warps release, so launch
    // only when the compiled launch register count covers the whole split.
    static int verdict = -1;
    if (verdict < 0) {
      cudaFuncAttributes a;
      verdict = (cudaFuncGetAttributes(&a, kern) == cudaSuccess && a.numRegs >= 168 &&
                 a.numRegs * Cfg::kThreads >= Cfg::kPoolNeeded)
                    ? 1
                    : 0;
    }
    if (verdict != 1) return cudaErrorNotSupported;
  }
  cudaError_t e = ensure_smem_attr(kern, Cfg::kSmemBytes, &done);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, Cfg::kThreads, Cfg::kSmemBytes, L.stream>>>(L.tm_q, L.tm_k, L.tm_v, L.p);
  return cudaGetLastError();
}

template <int DK, int DV, bool PAGED, bool FP8>
cudaError_t launch_prefill1_mod(const PrefillLaunch &L) {
  switch (L.mod) {
    case 0: return launch_prefill1_one<DK, DV, PAGED, FP8, 0>(L);
    case 1: return launch_prefill1_one<DK, DV, PAGED, FP8, 1>(L);
    default: return launch_prefill1_one<DK, DV, PAGED, FP8, 2>(L);
  }
}

template <int DK, int DV>
cudaError_t launch_prefill1_fp8(const PrefillLaunch &L) {
  return L.paged ? launch_prefill1_mod<DK, DV, true, true>(L) : launch_prefill1_mod<DK, DV, false, true>(L);
}

}  // namespace fa
