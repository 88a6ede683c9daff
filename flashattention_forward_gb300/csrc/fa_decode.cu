// Split-KV decode and combine kernel instantiations.
#include "fa_internal.h"

namespace fa {

template <int D, int KV, bool V5, bool R8 = false>
static cudaError_t launch_decode_d(const DecodeLaunch &L) {
  static unsigned long long done = 0;
  auto kern = fa_decode_kernel<D, KV, V5, R8>;
  constexpr int kSmem = DecodeCfg<D, KV, dec_direct<D, KV, V5>(), dec_direct<D, KV, V5>() && R8>::kSmemBytes;
  cudaError_t e = ensure_smem_attr(kern, kSmem, &done);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, kDecThreads, kSmem, L.stream>>>(L.tm_k, L.tm_v, L.p);
  return cudaGetLastError();
}

template <int KV>
static cudaError_t launch_decode_kv(int d, const DecodeLaunch &L) {
  if constexpr (KV != 0) {
    if (L.p.vec5) {
      if (d == 64) return launch_decode_d<64, KV, true>(L);
      if (d == 128 && L.rows8) return launch_decode_d<128, KV, true, true>(L);
      if (d == 128) return launch_decode_d<128, KV, true>(L);
      return cudaErrorNotSupported;
    }
  }
  if (d == 64) return launch_decode_d<64, KV, false>(L);
  if constexpr (KV != 0) {
    if (d == 128 && L.rows8) return launch_decode_d<128, KV, false, true>(L);
  }
  if (d == 128) return launch_decode_d<128, KV, false>(L);
  return cudaErrorNotSupported;
}

cudaError_t launch_decode(int d, const DecodeLaunch &L) {
  if (L.kv == 1) return launch_decode_kv<1>(d, L);
  if (L.kv == 2) return launch_decode_kv<2>(d, L);
  return launch_decode_kv<0>(d, L);
}

cudaError_t launch_combine(const float *o_part, const float *lse_part, int num_splits, int64_t n_rows, int hq,
                           int dv, void *out, float *lse, cudaStream_t stream) {
  const int64_t warps = n_rows * hq;
  if (warps == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (warps * 32 + threads - 1) / threads;
  auto *o = reinterpret_cast<__nv_bfloat16 *>(out);
  if (dv == 64)
    fa_combine_kernel<64><<<(unsigned)blocks, threads, 0, stream>>>(o_part, lse_part, num_splits, n_rows, hq, o, lse);
  else if (dv == 128)
    fa_combine_kernel<128><<<(unsigned)blocks, threads, 0, stream>>>(o_part, lse_part, num_splits, n_rows, hq, o, lse);
  else
    return cudaErrorNotSupported;
  return cudaGetLastError();
}

}  // namespace fa
