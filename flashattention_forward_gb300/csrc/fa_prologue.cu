// fa_prologue.cu -- pre-passes over the keys: the per-key score term of a
// prologue that adds a constant to Q (fkl_python PR #7, prologue-fusion
// commit: op chains fused onto the Q/K/V reads), and the largest V scale of
// each sequence for the e4m3 P * V mode.
//
// With q' = a_q q + b_q and k' = a_k k + b_k, the score scale * <q'_i, k'_j>
// holds the term scale * b_q * a_k * sum_d k_j[d], which depends on the key
// only.  This pass computes it once per (sequence, kv head, key) from the
// stored cache -- bf16 values, or e4m3 / int8 bytes times the key's per-token
// scale -- into col_bias[b][hk][j] (fp32, already multiplied by the factor that
// puts it in the attention kernel's score units), so that the kernels add one
// value per score column instead of rewriting K.  Entries j in [Sk, ld) are 0.
//
// One thread per key row: the row is read with 16-byte loads and summed in
// fp32 (e4m3 and int8 values are exact in fp32, as are bf16 values).
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "fa_internal.h"

namespace fa {
namespace {

__device__ __forceinline__ float sum_bf16x8(const uint4 u) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) acc += __uint_as_float(w[e] << 16) + __uint_as_float(w[e] & 0xFFFF0000u);
  return acc;
}

__device__ __forceinline__ float sum_e4m3x16(const uint4 u) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const __half2_raw hr =
          __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)((w[e] >> (16 * hf)) & 0xFFFFu), __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
      acc += f.x + f.y;
    }
  }
  return acc;
}

__device__ __forceinline__ int sum_i8x16(const uint4 u) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  int acc = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc += (int)(int8_t)((w[e] >> (8 * b)) & 0xFFu);
  return acc;
}

__global__ void __launch_bounds__(128) fa_col_bias_kernel(const ColBiasParams p) {
  const int b = blockIdx.z, hk = blockIdx.y;
  const int64_t j = (int64_t)blockIdx.x * 128 + threadIdx.x;
  if (j >= p.ld) return;
  float *dst = p.out + ((int64_t)b * p.hkv + hk) * p.ld + j;
  const int sk = __ldg(p.cu_k + b + 1) - __ldg(p.cu_k + b);
  // A sequence longer than the launch's max_seqlen_k would need key terms
  // past ld: flag it (the attention kernels read no term past ld).
  if (j == 0 && sk > p.ld) atomicCAS(p.err, 0, (int)FA_ERR_DEVICE_BOUNDS);
  if (j >= sk) {
    *dst = 0.f;
    return;
  }
  int64_t tok;   // row of the [*, Hkv] token view (scales are indexed the same way)
  const uint8_t *row;
  if (p.block_table) {
    const int64_t pi = j >> p.page_shift;
    const int page = pi < p.max_pages ? __ldg(p.block_table + (int64_t)b * p.bt_stride + pi) : -1;
    if (page < 0 || page >= p.n_pages) {
      atomicCAS(p.err, 0, (int)FA_ERR_DEVICE_BOUNDS);
      *dst = 0.f;
      return;
    }
    const int64_t slot = j & (p.page_size - 1);
    tok = (int64_t)page * p.page_size + slot;
    row = p.k + (int64_t)page * p.s_page + slot * p.s_slot + (int64_t)hk * p.s_head;
  } else {
    tok = (int64_t)__ldg(p.cu_k + b) + j;
    if (tok < 0 || tok >= p.n_pages) {   // packed: n_pages counts the cache's rows
      atomicCAS(p.err, 0, (int)FA_ERR_DEVICE_BOUNDS);
      *dst = 0.f;
      return;
    }
    row = p.k + tok * p.s_page + (int64_t)hk * p.s_head;
  }
  const uint4 *r4 = reinterpret_cast<const uint4 *>(row);
  float sum = 0.f;
  if (p.kv == 0) {
    for (int c = 0; c < p.dk / 8; ++c) sum += sum_bf16x8(__ldg(r4 + c));
  } else if (p.kv == 1) {
    for (int c = 0; c < p.dk / 16; ++c) sum += sum_e4m3x16(__ldg(r4 + c));
  } else {
    int isum = 0;
    for (int c = 0; c < p.dk / 16; ++c) isum += sum_i8x16(__ldg(r4 + c));
    sum = (float)isum;
  }
  if (p.kv != 0) sum *= __ldg(p.k_scale + tok * p.hkv + hk);
  *dst = p.factor * sum;
}

// The largest |v_scale| over the keys of one (sequence, kv head): 256
// threads stride over the keys (page-table lookups for paged caches) and
// reduce through shared memory.  Page ids outside the pool are flagged
// (FA_ERR_DEVICE_BOUNDS) and skipped.
__global__ void __launch_bounds__(256) fa_vscale_max_kernel(const VmaxParams p) {
  const int hk = blockIdx.x, b = blockIdx.y;
  const int k0 = __ldg(p.cu_k + b), sk = __ldg(p.cu_k + b + 1) - k0;
  float m = 0.f;
  for (int j = threadIdx.x; j < sk; j += 256) {
    int64_t tok;
    if (p.block_table) {
      const int64_t pi = j >> p.page_shift;
      const int page = pi < p.max_pages ? __ldg(p.block_table + (int64_t)b * p.bt_stride + pi) : -1;
      if (page < 0 || page >= p.n_pages) {
        atomicCAS(p.err, 0, (int)FA_ERR_DEVICE_BOUNDS);
        continue;
      }
      tok = (int64_t)page * p.page_size + (j & (p.page_size - 1));
    } else {
      tok = (int64_t)k0 + j;
      if (tok >= p.n_pages) {
        atomicCAS(p.err, 0, (int)FA_ERR_DEVICE_BOUNDS);
        continue;
      }
    }
    m = fmaxf(m, fabsf(__ldg(p.v_scale + tok * p.hkv + hk)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) r = fmaxf(r, red[w]);
    p.out[(int64_t)b * p.hkv + hk] = r;
  }
}

}  // namespace

cudaError_t launch_vscale_max(const VmaxParams &p, cudaStream_t stream) {
  fa_vscale_max_kernel<<<dim3((unsigned)p.hkv, (unsigned)p.num_seqs), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_col_bias(const ColBiasParams &p, cudaStream_t stream) {
  const dim3 grid((unsigned)((p.ld + 127) / 128), (unsigned)p.hkv, (unsigned)p.num_seqs);
  fa_col_bias_kernel<<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fa
