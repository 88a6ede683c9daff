// fa_noalloc.cu -- split-KV decode for callers that cannot allocate memory.
//
// Some callers of this library have no way to obtain device memory at the
// moment they run attention: plugins and custom ops inside an inference
// server that are handed only their input and output buffers, real-time
// serving loops whose memory is carved up once at start-up and may not grow,
// and code paths that must not call cudaMalloc because it can synchronise the
// device or fail under memory pressure in the middle of a request.  The
// split-KV decode needs scratch for its per-split partial outputs, so for
// these callers the scratch lives in a fixed, statically sized device array
// that the library owns.
//
// The array is a file-scope __device__ object: every GPU that loads the
// library holds FA_NOALLOC_SCRATCH_BYTES of it until the process exits.  Its
// device address is looked up once per device with cudaGetSymbolAddress (the
// host-side name is only a stand-in and must never be handed to a kernel).
#include <cstdio>
#include <mutex>

#include "../../include/fa_gb300.h"
#include "fa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device; the first call
// on a device performs the lookup (with that device current).
fa_status_t scratch_address(void **addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    char m[160];
    snprintf(m, sizeof m, "cudaGetDevice: %s", cudaGetErrorString(e));
    return fa::set_host_error(FA_ERR_CUDA, m);
  }
  if (dev < 0 || dev >= kMaxDevices) return fa::set_host_error(FA_ERR_UNSUPPORTED, "device ordinal >= 64");
  std::lock_guard<std::mutex> g(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char m[160];
      snprintf(m, sizeof m, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
      return fa::set_host_error(FA_ERR_CUDA, m);
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return FA_OK;
}

}  // namespace

extern "C" fa_status_t fa_fwd_varlen_noalloc(const fa_tensor_t *q, const fa_tensor_t *k_cache,
                                             const fa_tensor_t *v_cache, const fa_tensor_t *block_table,
                                             const fa_tensor_t *cu_seqlens_q, const fa_tensor_t *cu_seqlens_k,
                                             const fa_tensor_t *k_scale, const fa_tensor_t *v_scale,
                                             fa_tensor_t *out, fa_tensor_t *lse, float softmax_scale,
                                             int32_t causal, int32_t window, const fa_score_mod_t *score_mod,
                                             const fa_block_mask_t *block_mask, const fa_prologue_t *prologue,
                                             int32_t page_size, const fa_launch_t *launch, void *stream) {
  if (!launch || !q || !k_cache || !v_cache)
    return fa::set_host_error(FA_ERR_INVALID_ARG, "launch, q, k_cache and v_cache are required");
  if (q->ndim != 3 || k_cache->ndim < 3 || v_cache->ndim != k_cache->ndim)
    return fa::set_host_error(FA_ERR_INVALID_ARG, "q must be rank 3 and k/v caches rank 3 or 4");
  // Sizes come from q itself, so that every request too large for the static
  // scratch is refused here with that reason.
  if (q->shape[0] != launch->total_q)
    return fa::set_host_error(FA_ERR_INVALID_ARG, "q.shape[0] differs from launch->total_q");
  const int32_t hq = (int32_t)q->shape[1];
  const int32_t hkv = (int32_t)k_cache->shape[k_cache->ndim - 2];
  const int32_t dv = (int32_t)v_cache->shape[v_cache->ndim - 1];
  int32_t splits = launch->num_splits;
  if (splits <= 0)
    splits = fa_fwd_default_splits(launch->num_seqs, launch->max_seqlen_q, launch->max_seqlen_k, launch->total_k, hq,
                                   hkv, page_size);
  if (splits <= 1)
    return fa::set_host_error(FA_ERR_UNSUPPORTED,
                              "the allocation-free entry runs the split-KV decode only (needs 2 or more splits)");
  fa_launch_t L = *launch;
  L.num_splits = splits;
  const size_t need = fa_fwd_workspace_bytes(&L, hq, hkv, dv, prologue);
  if (need > (size_t)FA_NOALLOC_SCRATCH_BYTES) {
    char m[200];
    snprintf(m, sizeof m, "split-KV scratch of %zu bytes exceeds the static %zu-byte scratch; use fewer splits, fewer rows or fa_fwd_varlen",
             need, (size_t)FA_NOALLOC_SCRATCH_BYTES);
    return fa::set_host_error(FA_ERR_UNSUPPORTED, m);
  }
  void *scratch = nullptr;
  fa_status_t st = scratch_address(&scratch);
  if (st != FA_OK) return st;
  L.workspace = scratch;
  L.workspace_bytes = (size_t)FA_NOALLOC_SCRATCH_BYTES;
  return fa_fwd_varlen(q, k_cache, v_cache, block_table, cu_seqlens_q, cu_seqlens_k, k_scale, v_scale, out, lse,
                       softmax_scale, causal, window, score_mod, block_mask, prologue, page_size, &L, stream);
}
