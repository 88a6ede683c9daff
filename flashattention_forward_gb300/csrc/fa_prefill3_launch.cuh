// Launcher of the chunked-ring ping-pong kernel (fa_prefill3.cuh), shared by
// the per-head-dim translation units: bf16 K/V with Dk = 192, e4m3 and int8
// K/V, and e4m3 Q with e4m3 K/V.
#pragma once
#include "fa_internal.h"
#include "fa_prefill3.cuh"

namespace fa {

// A register-split variant raises the softmax warps with setmaxnreg.inc,
// which waits until other warps of the CTA release registers: it may run only
// when the compiled launch register count covers the whole split.
template <int DK, int DV, bool PAGED, bool FP8, int MOD, bool BIGREG, bool I8, bool Q8, bool V5 = false,
          bool PV8 = false>
bool prefill3_split_fits() {
  using Cfg = Prefill3Cfg<DK, DV, PAGED, FP8, MOD, BIGREG, Q8, PV8>;
  if constexpr (!Cfg::kSplitRegs) return true;
  static int fits = -1;   // per process: all devices run the same binary
  if (fits < 0) {
    cudaFuncAttributes a;
    fits = (cudaFuncGetAttributes(&a, fa_prefill3_kernel<DK, DV, PAGED, FP8, MOD, BIGREG, I8, Q8, V5, PV8>) == cudaSuccess &&
               a.numRegs * Cfg::kThreads >= Cfg::kPoolNeeded)
                  ? 1
                  : 0;
  }
  return fits == 1;
}

template <int DK, int DV, bool PAGED, bool FP8, int MOD, bool BIGREG, bool I8, bool Q8, bool V5 = false,
          bool PV8 = false>
cudaError_t launch_prefill3_one(const PrefillLaunch &L) {
  using Cfg = Prefill3Cfg<DK, DV, PAGED, FP8, MOD, BIGREG, Q8, PV8>;
  if (!prefill3_split_fits<DK, DV, PAGED, FP8, MOD, BIGREG, I8, Q8, V5, PV8>()) return cudaErrorNotSupported;
  static unsigned long long done = 0;
  auto kern = fa_prefill3_kernel<DK, DV, PAGED, FP8, MOD, BIGREG, I8, Q8, V5, PV8>;
  cudaError_t e = ensure_smem_attr(kern, Cfg::kSmemBytes, &done);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, Cfg::kThreads, Cfg::kSmemBytes, L.stream>>>(L.tm_q, L.tm_k, L.tm_v, L.p);
  return cudaGetLastError();
}

// bf16: the 12-warp split variant when it fits (and is not overridden), else
// the 10-warp two-half softmax.  e4m3: the 16-warp split variant only.
template <int DK, int DV, bool PAGED, bool FP8, int MOD, bool I8, bool Q8>
cudaError_t launch_prefill3_pick(const PrefillLaunch &L) {
  if constexpr (FP8) {
    return launch_prefill3_one<DK, DV, PAGED, true, MOD, false, I8, Q8>(L);
  } else {
    if (L.variant != 1 && prefill3_split_fits<DK, DV, PAGED, false, MOD, true, false, false>())
      return launch_prefill3_one<DK, DV, PAGED, false, MOD, true, false, false>(L);
    return launch_prefill3_one<DK, DV, PAGED, false, MOD, false, false, false>(L);
  }
}

// FP8: byte caches with per-token scales; I8 selects int8 values over e4m3;
// Q8 (e4m3 caches) takes e4m3 Q and runs QK on the bytes.  MOD 0 plain, 1
// ALiBi, 2 soft-cap; 3 and 4 (a prologue's per-key score term, never with
// Q8) are instantiated in translation units of their own.
template <int DK, int DV, bool FP8, bool I8 = false, bool Q8 = false>
cudaError_t launch_prefill3(const PrefillLaunch &L) {
  if constexpr (FP8 && !Q8) {
    if (L.p.vec5) return launch_prefill3_vec5(DK, I8, L);
  }
  if constexpr (Q8) {
    if (L.pv8) return launch_prefill3_pv8(DK, L);
  }
  if (L.mod >= 3) {
    if (Q8) return cudaErrorInvalidValue;
    return I8 ? launch_prefill3_kt_i8(DK, L) : launch_prefill3_kt(DK, FP8, L);
  }
  auto by_mod = [&](auto paged_tag) -> cudaError_t {
    constexpr bool PG = decltype(paged_tag)::value;
    switch (L.mod) {
      case 0: return launch_prefill3_pick<DK, DV, PG, FP8, 0, I8, Q8>(L);
      case 1: return launch_prefill3_pick<DK, DV, PG, FP8, 1, I8, Q8>(L);
      default: return launch_prefill3_pick<DK, DV, PG, FP8, 2, I8, Q8>(L);
    }
  };
  return L.paged ? by_mod(std::true_type{}) : by_mod(std::false_type{});
}

// The 5-D page kernels of one (Dk, Dv, cache) combination (MOD 0-2; the
// host takes no prologue score terms with 5-D pages).
template <int DK, int DV, bool I8>
cudaError_t launch_prefill3_vec5_one(const PrefillLaunch &L) {
  switch (L.mod) {
    case 0: return launch_prefill3_one<DK, DV, true, true, 0, false, I8, false, true>(L);
    case 1: return launch_prefill3_one<DK, DV, true, true, 1, false, I8, false, true>(L);
    case 2: return launch_prefill3_one<DK, DV, true, true, 2, false, I8, false, true>(L);
    default: return cudaErrorInvalidValue;
  }
}

// The e4m3 P * V kernels (with e4m3 Q) of one Dk (MOD 0-2).
template <int DK>
cudaError_t launch_prefill3_pv8_one(const PrefillLaunch &L) {
  auto by_mod = [&](auto paged_tag) -> cudaError_t {
    constexpr bool PG = decltype(paged_tag)::value;
    switch (L.mod) {
      case 0: return launch_prefill3_one<DK, 128, PG, true, 0, false, false, true, false, true>(L);
      case 1: return launch_prefill3_one<DK, 128, PG, true, 1, false, false, true, false, true>(L);
      case 2: return launch_prefill3_one<DK, 128, PG, true, 2, false, false, true, false, true>(L);
      default: return cudaErrorInvalidValue;
    }
  };
  return L.paged ? by_mod(std::true_type{}) : by_mod(std::false_type{});
}

// The MOD 3 and 4 kernels of one (Dk, Dv, cache) combination.
template <int DK, int DV, bool FP8, bool I8>
cudaError_t launch_prefill3_kt_one(const PrefillLaunch &L) {
  if (L.paged)
    return L.mod == 3 ? launch_prefill3_pick<DK, DV, true, FP8, 3, I8, false>(L)
                      : launch_prefill3_pick<DK, DV, true, FP8, 4, I8, false>(L);
  return L.mod == 3 ? launch_prefill3_pick<DK, DV, false, FP8, 3, I8, false>(L)
                    : launch_prefill3_pick<DK, DV, false, FP8, 4, I8, false>(L);
}

}  // namespace fa
