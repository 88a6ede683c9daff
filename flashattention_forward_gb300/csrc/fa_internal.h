// fa_internal.h -- launch descriptors shared by the C-ABI front end and the
// kernel translation units (one per head-dim family, compiled in parallel).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa_gb300.h"
#include "fa_decode.cuh"
#include "fa_prefill.cuh"
#include "fa_bwd_params.h"

namespace fa {

struct PrefillLaunch {
  CUtensorMap tm_q, tm_k, tm_v;
  PrefillParams p;
  int paged, fp8;
  int mod;       // 0 plain, 1 ALiBi, 2 soft-cap; 3, 4: 1, 2 with a Q add's per-key term
  int int8;      // with fp8: the byte cache holds int8 values (else e4m3)
  int q8;        // with fp8 (e4m3): Q is e4m3 and QK runs on the bytes
  int variant;   // 0: fastest available, 1: force the 10-warp two-pass softmax
  int tiles_per_cta;   // 128-row query tiles per CTA: 2 (ping-pong), or 1 (two CTAs per SM)
  int pv8;             // with q8: P * V on e4m3 P and V (opt-in precision mode)
  dim3 grid;
  cudaStream_t stream;
};

struct DecodeLaunch {
  CUtensorMap tm_k, tm_v;
  DecodeParams p;
  int kv;        // cache: 0 bf16, 1 e4m3, 2 int8 (the last two with per-token scales)
  int rows8;     // every CTA has at most 8 query rows (max_seqlen_q * Hq/Hkv <= 8)
  dim3 grid;
  cudaStream_t stream;
};

struct BwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  BwdParams p;
  BwdDeltaParams dp;
  unsigned delta_blocks;
  int mod;       // score mod: 0 none, 1 ALiBi, 2 soft-cap
  dim3 grid_q, grid_kv;
  cudaStream_t stream;
};

// The per-key score term of a Q add (fa_prologue.cu): col_bias[b][hk][j] =
// factor * k_scale * sum_d k_j[d] for j < Sk_b, 0 for Sk_b <= j < ld.
struct ColBiasParams {
  const uint8_t *k;             // cache base
  int kv;                       // 0 bf16, 1 e4m3, 2 int8
  int64_t s_page, s_slot, s_head;   // byte strides: page (packed: token row), slot, kv head
  const int32_t *block_table;   // [B, bt_stride] or null (packed)
  int64_t bt_stride, max_pages; // block-table row stride and entries per row
  int32_t page_size, page_shift;
  int64_t n_pages;              // pages in the pool (packed: rows of the cache)
  const int32_t *cu_k;
  const float *k_scale;         // byte caches: per (token, kv head)
  int32_t dk, hkv, num_seqs;
  int64_t ld;
  float factor;
  float *out;
  int *err;
};
cudaError_t launch_col_bias(const ColBiasParams &p, cudaStream_t stream);

// The largest |v_scale| of each (sequence, kv head), for the e4m3 P * V mode.
struct VmaxParams {
  const float *v_scale;         // [N_pg, P_s, Hkv] (paged) or [T_k, Hkv]
  const int32_t *block_table;   // [B, bt_stride] or null (packed)
  int64_t bt_stride, max_pages;
  int32_t page_size, page_shift;
  int64_t n_pages;              // pages in the pool (packed: tokens of the cache)
  const int32_t *cu_k;
  int32_t hkv, num_seqs;
  float *out;                   // [B][Hkv]
  int *err;
};
cudaError_t launch_vscale_max(const VmaxParams &p, cudaStream_t stream);

cudaError_t launch_bwd(int d, const BwdLaunch &L);
cudaError_t launch_prefill_64_64(const PrefillLaunch &L);
cudaError_t launch_prefill_128_128(const PrefillLaunch &L);
cudaError_t launch_prefill_192_128(const PrefillLaunch &L);
cudaError_t launch_prefill_192_128_fp8(const PrefillLaunch &L);
cudaError_t launch_prefill_64_64_i8(const PrefillLaunch &L);
cudaError_t launch_prefill_128_128_i8(const PrefillLaunch &L);
cudaError_t launch_prefill_192_128_i8(const PrefillLaunch &L);
cudaError_t launch_prefill_128_128_q8(const PrefillLaunch &L);
cudaError_t launch_prefill_192_128_q8(const PrefillLaunch &L);
// Kernels with a prologue's per-key score term (PrefillLaunch::mod 3 or 4), in
// translation units of their own: the ping-pong kernel (bf16 K/V, Dk = Dv in
// {64, 128}) and the chunked-ring kernel (bf16 Dk 192, e4m3 and int8 caches).
cudaError_t launch_prefill2_kt(int d, const PrefillLaunch &L);
// The ping-pong kernel with one query tile per CTA (two CTAs per SM; bf16
// K/V, Dk = Dv in {64, 128}, MOD 0-2), in a translation unit of its own.
cudaError_t launch_prefill2_t1(int d, const PrefillLaunch &L);
cudaError_t launch_prefill3_kt(int dk, bool fp8, const PrefillLaunch &L);
cudaError_t launch_prefill3_kt_i8(int dk, const PrefillLaunch &L);
// Chunked-ring kernels for byte caches in the vectorized 5-D page layouts
// (MOD 0-2), in translation units of their own.
cudaError_t launch_prefill3_vec5(int dk, bool i8, const PrefillLaunch &L);
cudaError_t launch_prefill3_vec5_i8(int dk, const PrefillLaunch &L);
// Chunked-ring kernels with e4m3 Q and P * V on e4m3 P and V (Dk 128 or 192,
// Dv 128, MOD 0-2), in a translation unit of their own.
cudaError_t launch_prefill3_pv8(int dk, const PrefillLaunch &L);
cudaError_t launch_decode(int d, const DecodeLaunch &L);
cudaError_t launch_combine(const float *o_part, const float *lse_part, int num_splits, int64_t n_rows, int hq,
                           int dv, void *out, float *lse, cudaStream_t stream);

// Records a host-side error message for fa_last_error() and returns `st`.
fa_status_t set_host_error(fa_status_t st, const char *msg);

// Sets the dynamic shared-memory attribute once per (kernel, device).
template <typename K>
cudaError_t ensure_smem_attr(K kernel, int bytes, unsigned long long *done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  // all shared memory, none as L1, so that kernels sized for two CTAs per
  // SM get them
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) __atomic_fetch_or(done_mask, bit, __ATOMIC_ACQ_REL);
  return e;
}

}  // namespace fa
