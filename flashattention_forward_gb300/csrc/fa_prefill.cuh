// fa_prefill.cuh -- definitions shared by the prefill kernels (fa_prefill2.cuh,
// fa_prefill3.cuh): tile sizes, the kernel parameter block and the order in
// which CTAs take (sequence, head, query-tile pair) work items.
//
// The method is the tiled online-softmax forward of RL-Kernel PR #237 ("SM90
// TMA + mma.sync FlashAttention": TMA loads, QK^T, softmax, PV, LSE export) and
// FlyDSL PR #1066 (paged KV via block_table, lazy O rescaling with a threshold
// of 8 in scaled log2 units, logit scale folded into the max subtraction),
// with the contractions on the fifth-generation tensor cores and the
// accumulators in tensor memory.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "fa_gather.cuh"
#include "sm103_ptx.cuh"

namespace fa {

constexpr int kBlockM = 128;   // query rows per tile (MMA M)
constexpr int kBlockN = 128;   // keys per tile (MMA N of QK^T, K of PV)
constexpr float kRescaleThreshold = 8.0f;   // lazy O rescale, scaled log2 units
constexpr float kGuardSum = 0x1p64f;        // tile row sum above which the deferred max is taken

struct PrefillParams {
  const int32_t *cu_q;
  const int32_t *cu_k;
  const int32_t *block_table;   // [B, bt_stride] or null
  int64_t bt_stride;
  const float *k_scale;         // per token and kv head (e4m3 only)
  const float *v_scale;
  __nv_bfloat16 *out;
  int64_t out_stride_t, out_stride_h;   // elements
  float *lse;                   // [Hq, T_q] or null
  int64_t total_q;
  const uint8_t *block_mask;    // [B*Hq, n_qblk, n_kblk] or null
  int32_t n_qblk, n_kblk;
  int32_t num_seqs, hq, hkv, group;
  int32_t page_size, page_shift, pages_per_tile, rows_per_box;
  int32_t n_qtiles;
  int32_t causal, window;
  float scale_log2;     // softmax_scale * log2(e)
  float softcap_arg;    // softmax_scale / cap
  float softcap_log2;   // cap * log2(e)
  float alibi_log2;     // slope * log2(e)
  int *err;             // device error word
  int32_t head_group;   // heads interleaved per group in the block order
  int32_t n_hgroups;    // ceil(hq / head_group)
  int32_t n_items;      // work items (persistent kernels stride over them)
  int32_t gather;       // pages of < 16 keys: K/V rows by cp.async (fa_gather.cuh), not TMA boxes
  KvGather gk, gv;      // the caches' byte geometry for the gather
  // folded prologue: out = pro_vmul * o + pro_vadd on rows that see keys;
  // the row term of the score, pro_lse_k * sum_d q[d] + pro_lse_c, is added
  // to the LSE (bf16 q read back only when pro_lse_k != 0); under the
  // soft-cap it enters the capped score instead, as pro_row_k * sum_d q[d] +
  // pro_row_c in 2u*log2(e) units
  float pro_vmul, pro_vadd, pro_lse_k, pro_lse_c, pro_row_k, pro_row_c;
  const __nv_bfloat16 *q;
  int64_t q_stride_t, q_stride_h;   // elements
  // the prologue's per-key score term (a Q add), [B][Hkv][cb_ld] fp32 in the
  // units of the kernel's score (log2, or 2u*log2(e) under the soft-cap);
  // null when there is none
  const float *col_bias;
  int64_t cb_ld;
  // byte caches in the vectorized 5-D layouts (paged, pages of >= 16 keys):
  // K [N_pg, Hkv, Dk/16, P_s, 16], V [N_pg, Hkv, P_s/16, Dv, 16]
  int32_t vec5;
  // e4m3 P * V (opt-in): the largest |v_scale| of each (sequence, kv head),
  // [B][Hkv] fp32 written by a pre-pass; null otherwise
  const float *pv_vmax;
};


// sum_d q[d] of one bf16 query row (16-byte loads), for the prologue's LSE term.
template <int D>
__device__ __forceinline__ float q_row_sum(const __nv_bfloat16 *row) {
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    const uint4 u = *reinterpret_cast<const uint4 *>(row + c * 8);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) acc += __uint_as_float(w[e] << 16) + __uint_as_float(w[e] & 0xFFFF0000u);
  }
  return acc;
}

// Row term of the prologue inside the soft-cap argument (0 without one).
template <int D>
__device__ __forceinline__ float softcap_row_term(const PrefillParams &p, int64_t t, int h) {
  float rb = p.pro_row_c;
  if (p.pro_row_k != 0.f) rb += p.pro_row_k * q_row_sum<D>(p.q + t * p.q_stride_t + (int64_t)h * p.q_stride_h);
  return rb;
}

// Block order: for each sequence, for each group of `head_group` heads, query
// tiles from the latest (longest under a causal mask) to the first, the heads
// of the group interleaved.  Concurrent CTAs then share the K/V of a few
// heads through L2, and long tiles start first.  Returns false for padding.
__device__ __forceinline__ bool decode_block(const PrefillParams &p, int item, int &b, int &h, int &qt) {
  unsigned L = (unsigned)item;
  const int g_in = (int)(L % (unsigned)p.head_group);
  L /= (unsigned)p.head_group;
  const int pr = (int)(L % (unsigned)p.n_qtiles);
  L /= (unsigned)p.n_qtiles;
  const int hg = (int)(L % (unsigned)p.n_hgroups);
  b = (int)(L / (unsigned)p.n_hgroups);
  h = hg * p.head_group + g_in;
  qt = p.n_qtiles - 1 - pr;
  return h < p.hq;
}

}  // namespace fa
