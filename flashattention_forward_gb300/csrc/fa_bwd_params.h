// fa_bwd_params.h -- kernel parameter blocks of the backward pass (shared by
// the C-ABI front end and the kernels in fa_bwd.cuh).
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace fa {

struct BwdParams {
  const int32_t *cu_q, *cu_k;
  const float *lse;          // [Hq, T_q], natural log
  const float *delta;        // [Hq, T_q]
  __nv_bfloat16 *dq;         // [T_q, Hq, D] (strides in elements)
  int64_t dq_stride_t, dq_stride_h;
  __nv_bfloat16 *dk, *dv;    // [T_k, Hkv, D]
  int64_t dk_stride_t, dk_stride_h, dv_stride_t, dv_stride_h;
  int64_t total_q;
  int32_t num_seqs, hq, hkv, group;
  int32_t n_qtiles, n_ktiles;   // grid extents: cdiv(max_seqlen, 128)
  int32_t causal, window;
  float scale_log2;             // softmax_scale * log2(e)
  float scale;                  // softmax_scale
  int *err;
  const uint8_t *block_mask;    // [B*Hq, n_qblk, n_kblk] (128 x 128 blocks, 0 = skipped) or null
  int n_qblk, n_kblk;
  float softcap_arg;            // soft-cap: softmax_scale / cap
  float softcap_log2;           // soft-cap: cap * log2(e)
  float alibi_log2;             // ALiBi: slope * log2(e)
};

struct BwdDeltaParams {
  const __nv_bfloat16 *out, *dout;
  int64_t o_stride_t, o_stride_h, do_stride_t, do_stride_h;
  float *delta;                 // [Hq, T_q]
  int64_t total_q;
  int32_t hq, d;
};

}  // namespace fa
