// fa_api.cu -- the C ABI declared in include/fa_gb300.h: host-side validation,
// TMA descriptor encoding and variant dispatch.  Every check runs on the host
// before anything is enqueued; no device memory is read back or allocated.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "../../include/fa_gb300.h"
#include "fa_internal.h"

namespace fa {
// The per-device error word (one copy per device that loads the library).
__device__ int g_fa_error = 0;
}

namespace {

thread_local char g_msg[512] = "";

fa_status_t fail(fa_status_t st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return st;
}

fa_status_t cuda_fail(cudaError_t e, const char *where) {
  return fail(FA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Tiled map with 128-byte swizzle; strides in bytes for dims 1..rank-1.
fa_status_t make_map(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *base, const uint64_t *dims,
                     const uint64_t *strides, const uint32_t *box, const char *what,
                     CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, dt, rank, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
  return FA_OK;
}

int dtype_size(int dt) {
  switch (dt) {
    case FA_BF16: return 2;
    case FA_E4M3: return 1;
    case FA_I8: return 1;
    case FA_F32: return 4;
    case FA_I32: return 4;
    case FA_U8: return 1;
    default: return 0;
  }
}

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }
int ilog2(int64_t x) {
  int s = 0;
  while ((int64_t(1) << s) < x) ++s;
  return s;
}

// Basic shape/dtype check of a tensor descriptor.
fa_status_t check_tensor(const fa_tensor_t *t, const char *name, int dtype, int ndim) {
  if (!t) return fail(FA_ERR_INVALID_ARG, "%s is NULL", name);
  if (t->dtype != dtype) return fail(FA_ERR_INVALID_ARG, "%s has dtype %d, expected %d", name, t->dtype, dtype);
  if (t->ndim != ndim) return fail(FA_ERR_INVALID_ARG, "%s has %d dims, expected %d", name, t->ndim, ndim);
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0) return fail(FA_ERR_INVALID_ARG, "%s has a negative extent", name);
  return FA_OK;
}

bool contiguous(const fa_tensor_t *t) {
  int64_t s = 1;
  for (int i = t->ndim - 1; i >= 0; --i) {
    if (t->shape[i] != 1 && t->stride[i] != s) return false;
    s *= t->shape[i];
  }
  return true;
}

int64_t numel(const fa_tensor_t *t) {
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}

int64_t span_bytes(const fa_tensor_t *t) {
  int64_t hi = 0;
  for (int i = 0; i < t->ndim; ++i) hi += (t->shape[i] - 1) * t->stride[i];
  return (hi + 1) * dtype_size(t->dtype);
}

bool overlaps(const fa_tensor_t *a, const fa_tensor_t *b) {
  if (!a || !b || numel(a) == 0 || numel(b) == 0) return false;
  const char *a0 = (const char *)a->data, *b0 = (const char *)b->data;
  return a0 < b0 + span_bytes(b) && b0 < a0 + span_bytes(a);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Device address of the error word on the current device (looked up once per
// device; cudaGetSymbolAddress allocates nothing).
int *error_word() {
  static int *addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, fa::g_fa_error) == cudaSuccess) addr[dev] = (int *)p;
  }
  return addr[dev];
}

// Score mod (kind 0 none, 1 ALiBi, 2 soft-cap; NULL = none) and 128 x 128
// block mask checks shared by the forward and backward entry points.
fa_status_t check_mods(const fa_score_mod_t *score_mod, const fa_block_mask_t *block_mask, const fa_launch_t *launch,
                       int *mod, float *slope, float *cap) {
  *mod = 0;
  *slope = *cap = 0.f;
  if (score_mod) {
    *mod = score_mod->kind;
    if (*mod < 0 || *mod > 2) return fail(FA_ERR_INVALID_ARG, "score_mod.kind %d", *mod);
    *slope = score_mod->alibi_slope;
    *cap = score_mod->softcap;
    if (*mod == 1 && !std::isfinite(*slope)) return fail(FA_ERR_INVALID_ARG, "alibi_slope must be finite");
    if (*mod == 2 && !(*cap > 0.f && std::isfinite(*cap)))
      return fail(FA_ERR_INVALID_ARG, "softcap must be positive and finite");
  }
  if (block_mask) {
    if (!block_mask->data) return fail(FA_ERR_INVALID_ARG, "block_mask.data is NULL");
    if (block_mask->blk_q != 128 || block_mask->blk_k != 128)
      return fail(FA_ERR_UNSUPPORTED, "block masks use 128x128 blocks");
    if ((int64_t)block_mask->n_qblk * 128 < launch->max_seqlen_q || (int64_t)block_mask->n_kblk * 128 < launch->max_seqlen_k)
      return fail(FA_ERR_INVALID_ARG, "block_mask does not cover max_seqlen_q/k");
  }
  return FA_OK;
}

// The bf16 prefill runs its register-rebalanced one-pass softmax when the
// build's launch registers allow it, with two query tiles per CTA or one
// (two CTAs per SM) as tiles_per_cta() picks.  FA_GB300_PREFILL_VARIANT in
// the environment at the first forward call of the process overrides that
// (a diagnosis switch; results agree to rounding): 1 selects the 10-warp
// two-pass form, 2 one tile per CTA wherever it exists, 3 two tiles.
int prefill_variant() {
  static const int v = [] {
    const char *e = getenv("FA_GB300_PREFILL_VARIANT");
    return (e && e[0] >= '1' && e[0] <= '3') ? e[0] - '0' : 0;
  }();
  return v;
}

// Query tiles per CTA of the bf16 ping-pong prefill.  One tile per CTA lets
// two CTAs share an SM, so that each CTA's set-up, pipeline fill and
// epilogue overlap the other's main loop, and each CTA walks only its own
// tile's key tiles (a two-tile CTA walks the union of both tiles' lists).
// Measured on one GB300 (one tile against two): config-5 window run +25%,
// 50% block mask +26%, soft-cap +3-4%, ALiBi causal +2%, config-2 lengths
// +4% (+10% causal); long dense plain runs -3% and ALiBi non-causal -4%
// (one-tile CTAs reload K/V twice as often); a grid of a few CTAs is
// faster with two tiles.  With ALiBi's bias in the contraction (MOD 5,
// either form; fa_prefill2.cuh) config 5's causal run is faster with one
// tile (944 against 932 TFLOP/s) and the non-causal one with two (1070
// against 1034).
struct TileHints {
  double avg_key_tiles;   // key tiles a query tile visits, on average
  double n_tiles;         // query tiles x heads, about
  bool block_mask, causal, window;
  int mod;                // 0 plain, 1 ALiBi, 2 soft-cap
};
int tiles_per_cta(bool eligible, int variant, const TileHints &h) {
  if (!eligible || variant == 1 || variant == 3) return 2;
  if (variant == 2) return 1;
  if (h.n_tiles <= 64) return 2;
  if (h.block_mask || h.window || h.mod == 2 || h.avg_key_tiles <= 8.0 || (h.mod == 1 && h.causal)) return 1;
  return 2;
}

// Byte geometry of a paged cache [N_pg, P_s, Hkv, D] for the row gather.
fa::KvGather kv_gather(const fa_tensor_t *t, int esz) {
  fa::KvGather g;
  g.base = (const uint8_t *)t->data;
  g.page_stride = t->stride[0] * esz;
  g.slot_stride = t->stride[1] * esz;
  g.head_stride = t->stride[2] * esz;
  return g;
}

// Tensor maps over byte caches in the vectorized 5-D page layouts:
// K [N_pg, Hkv, Dk/16, P_s, 16] in boxes of {16 bytes, k_rows tokens,
// k_groups column groups}, V [N_pg, Hkv, P_s/16, Dv, 16] in boxes of
// {16 tokens, v_dims dims, v_groups token groups}; unswizzled uint8.
fa_status_t make_vec5_maps(CUtensorMap *tk, CUtensorMap *tv, const fa_tensor_t *k, const fa_tensor_t *v, int64_t dk,
                           int64_t dv, int64_t hkv, int64_t ps, int64_t n_pages, uint32_t k_rows, uint32_t k_groups,
                           uint32_t v_dims, uint32_t v_groups) {
  const uint64_t kd[5] = {16, (uint64_t)ps, (uint64_t)(dk / 16), (uint64_t)hkv, (uint64_t)n_pages};
  const uint64_t ks[4] = {(uint64_t)k->stride[3], (uint64_t)k->stride[2], (uint64_t)k->stride[1], (uint64_t)k->stride[0]};
  const uint32_t kb[5] = {16, k_rows, k_groups, 1, 1};
  const uint64_t vd[5] = {16, (uint64_t)dv, (uint64_t)(ps / 16), (uint64_t)hkv, (uint64_t)n_pages};
  const uint64_t vs[4] = {(uint64_t)v->stride[3], (uint64_t)v->stride[2], (uint64_t)v->stride[1], (uint64_t)v->stride[0]};
  const uint32_t vb[5] = {16, v_dims, v_groups, 1, 1};
  fa_status_t st = make_map(tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, k->data, kd, ks, kb, "k (5-D)", CU_TENSOR_MAP_SWIZZLE_NONE);
  if (st) return st;
  return make_map(tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, v->data, vd, vs, vb, "v (5-D)", CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool supported_dims(int64_t dk, int64_t dv) {
  return (dk == 64 && dv == 64) || (dk == 128 && dv == 128) || (dk == 192 && dv == 128);
}

// A prologue's op chains, each composed into one map x -> a * x + b.
struct Folded {
  double aq = 1, bq = 0, ak = 1, bk = 0, av = 1, bv = 0;
};

fa_status_t compose_chain(const fa_prologue_op_t *ops, int32_t n, const char *name, double *a, double *b) {
  *a = 1.0;
  *b = 0.0;
  if (n < 0 || n > FA_PROLOGUE_MAX_OPS)
    return fail(FA_ERR_INVALID_ARG, "prologue %s chain has %d ops (0 ... %d)", name, n, FA_PROLOGUE_MAX_OPS);
  for (int i = 0; i < n; ++i) {
    const double c = ops[i].value;
    if (!std::isfinite(ops[i].value)) return fail(FA_ERR_INVALID_ARG, "prologue values must be finite");
    switch (ops[i].op) {
      case FA_OP_MUL: *a *= c; *b *= c; break;
      case FA_OP_ADD: *b += c; break;
      case FA_OP_SUB: *b -= c; break;
      case FA_OP_DIV:
        if (c == 0.0) return fail(FA_ERR_INVALID_ARG, "prologue %s chain divides by 0", name);
        *a /= c;
        *b /= c;
        break;
      default: return fail(FA_ERR_INVALID_ARG, "prologue %s op %d: use FA_OP_MUL, ADD, SUB or DIV", name, ops[i].op);
    }
  }
  if (!std::isfinite(*a) || !std::isfinite(*b)) return fail(FA_ERR_INVALID_ARG, "prologue %s chain overflows", name);
  return FA_OK;
}

fa_status_t fold_prologue(const fa_prologue_t *pro, Folded *f) {
  *f = Folded();
  if (!pro) return FA_OK;
  fa_status_t st;
  if ((st = compose_chain(pro->q, pro->n_q, "q", &f->aq, &f->bq))) return st;
  if ((st = compose_chain(pro->k, pro->n_k, "k", &f->ak, &f->bk))) return st;
  return compose_chain(pro->v, pro->n_v, "v", &f->av, &f->bv);
}

// A Q add contributes scale * b_q * a_k * sum_d k_j[d] to score j.
bool needs_col_bias(const Folded &f) { return f.bq != 0.0 && f.ak != 0.0; }

int64_t col_bias_ld(int32_t max_seqlen_k) { return ((int64_t)max_seqlen_k + 127) / 128 * 128; }

size_t split_part_bytes(const fa_launch_t *L, int32_t hq, int32_t dv) {
  if (L->num_splits < 2 || L->total_q <= 0 || hq <= 0 || dv <= 0) return 0;
  const size_t o = (size_t)L->num_splits * L->total_q * hq * dv * sizeof(float);
  const size_t l = (size_t)L->num_splits * hq * L->total_q * sizeof(float);
  return align256(o) + align256(l);
}

size_t col_part_bytes(const fa_launch_t *L, int32_t hkv, const Folded &f) {
  if (!needs_col_bias(f) || L->num_seqs <= 0 || hkv <= 0 || L->max_seqlen_k <= 0) return 0;
  return align256((size_t)L->num_seqs * hkv * col_bias_ld(L->max_seqlen_k) * sizeof(float));
}

// e4m3 P * V: one fp32 per (sequence, kv head), the largest V scale.
size_t vmax_part_bytes(const fa_launch_t *L, int32_t hkv) {
  if (!(L->flags & FA_FLAG_PV_E4M3) || L->num_seqs <= 0 || hkv <= 0) return 0;
  return align256((size_t)L->num_seqs * hkv * sizeof(float));
}

}  // namespace

namespace fa {
fa_status_t set_host_error(fa_status_t st, const char *msg) { return fail(st, "%s", msg); }
}  // namespace fa

// A prepared forward call (fa_fwd_plan_create): the launch descriptors that
// fa_fwd_varlen would enqueue, kept for repeated launches.
struct fa_fwd_plan_s {
  int kind = 0;              // 0: nothing to launch, 1: split-KV decode (+ combine), 2: prefill
  int dk = 0, fp8 = 0;
  int has_cb = 0;            // the prologue's per-key term is computed first
  fa::ColBiasParams cb;
  int has_vm = 0;            // e4m3 P * V: the V-scale maxima are computed first
  fa::VmaxParams vm;
  fa::DecodeLaunch dl;
  int splits = 0, hq = 0, dv = 0;
  int64_t rows = 0;
  void *out = nullptr;
  fa::PrefillLaunch pl;
};

namespace {

fa_status_t run_col_bias(const fa_fwd_plan_s &P, cudaStream_t s) {
  if (P.has_vm) {
    cudaError_t e = fa::launch_vscale_max(P.vm, s);
    if (e != cudaSuccess) return cuda_fail(e, "V-scale pre-pass launch");
  }
  if (!P.has_cb) return FA_OK;
  cudaError_t e = fa::launch_col_bias(P.cb, s);
  if (e != cudaSuccess) return cuda_fail(e, "prologue key-term launch");
  return FA_OK;
}

fa_status_t run_decode(fa::DecodeLaunch L, const fa_fwd_plan_s &P, cudaStream_t s) {
  L.stream = s;
  fa_status_t st = run_col_bias(P, s);
  if (st != FA_OK) return st;
  cudaError_t e = fa::launch_decode(P.dk, L);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  if (P.splits > 1) {
    e = fa::launch_combine(L.p.o_part, L.p.lse_part, P.splits, P.rows, P.hq, P.dv, P.out, L.p.lse, s);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  }
  return FA_OK;
}

fa_status_t run_prefill(fa::PrefillLaunch L, const fa_fwd_plan_s &P, cudaStream_t s) {
  L.stream = s;
  fa_status_t st = run_col_bias(P, s);
  if (st != FA_OK) return st;
  cudaError_t e;
  if (P.dk == 64) e = fa::launch_prefill_64_64(L);
  else if (P.dk == 128) e = fa::launch_prefill_128_128(L);
  else e = fa::launch_prefill_192_128(L);
  if (e == cudaErrorNotSupported && P.fp8)
    return fail(FA_ERR_UNSUPPORTED, "the e4m3/int8 kernel's register split does not fit this build's launch registers");
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return FA_OK;
}

// Validates a forward call and builds its launch descriptors; launches them on
// `stream` unless `plan` is given, in which case they are stored there.
fa_status_t fwd_build(const fa_tensor_t *q, const fa_tensor_t *k_cache, const fa_tensor_t *v_cache,
                      const fa_tensor_t *block_table, const fa_tensor_t *cu_seqlens_q,
                      const fa_tensor_t *cu_seqlens_k, const fa_tensor_t *k_scale, const fa_tensor_t *v_scale,
                      fa_tensor_t *out, fa_tensor_t *lse, float softmax_scale, int32_t causal, int32_t window,
                      const fa_score_mod_t *score_mod, const fa_block_mask_t *block_mask,
                      const fa_prologue_t *prologue, int32_t page_size, const fa_launch_t *launch, void *stream,
                      fa_fwd_plan_s *plan);

}  // namespace

extern "C" {

const char *fa_last_error(void) { return g_msg; }

const char *fa_version(void) { return "fa_gb300 0.1 (sm_103a)"; }

size_t fa_fwd_workspace_bytes(const fa_launch_t *launch, int32_t hq, int32_t hkv, int32_t dv,
                              const fa_prologue_t *prologue) {
  if (!launch) return 0;
  Folded f;
  char saved[sizeof g_msg];
  memcpy(saved, g_msg, sizeof g_msg);
  if (fold_prologue(prologue, &f) != FA_OK) f = Folded();   // the call itself reports a malformed prologue
  memcpy(g_msg, saved, sizeof g_msg);
  return split_part_bytes(launch, hq, dv) + col_part_bytes(launch, hkv, f) + vmax_part_bytes(launch, hkv);
}

int32_t fa_fwd_default_splits(int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k, int64_t total_k,
                              int32_t hq, int32_t hkv, int32_t page_size) {
  (void)page_size;
  if (num_seqs <= 0 || hq <= 0 || hkv <= 0 || hq % hkv) return 0;
  const int64_t rows = (int64_t)max_seqlen_q * (hq / hkv);
  if (rows <= 0 || rows > fa::kDecRows) return 0;
  if (max_seqlen_k < 256) return 0;
  // Key ranges sized so that the non-empty (split, kv head, sequence) CTAs
  // make about three waves at two CTAs per SM: long ranges keep each CTA's
  // pipeline fill and partial-output traffic small, three waves bound the tail.
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 148;
  const double mean_k = total_k > 0 ? (double)total_k / num_seqs : 0.5 * max_seqlen_k;
  const double key_units = mean_k * num_seqs * hkv;
  const double target_ctas = 3.0 * 2.0 * sms;
  double keys_per_split = key_units / target_ctas;
  if (keys_per_split < 256) keys_per_split = 256;
  int64_t s = (int64_t)((max_seqlen_k + keys_per_split - 1) / keys_per_split);
  if (s > 64) s = 64;
  if (s < 1) s = 1;
  return (int32_t)s;
}

fa_status_t fa_get_device_error(void *stream, int32_t *code) {
  if (!code) return fail(FA_ERR_INVALID_ARG, "code is NULL");
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, fa::g_fa_error, sizeof v);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
  const int zero = 0;
  e = cudaMemcpyToSymbol(fa::g_fa_error, &zero, sizeof zero);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
  *code = v;
  return FA_OK;
}

fa_status_t fa_combine(const float *o_part, const float *lse_part, int32_t num_splits, int64_t n_rows, int32_t hq,
                       int32_t dv, void *out_bf16, float *lse, void *stream) {
  if (num_splits <= 0 || n_rows < 0 || hq <= 0) return fail(FA_ERR_INVALID_ARG, "bad combine sizes");
  if (dv != 64 && dv != 128) return fail(FA_ERR_UNSUPPORTED, "combine supports Dv 64 or 128, got %d", dv);
  if (n_rows == 0) return FA_OK;
  if (!o_part || !lse_part || !out_bf16) return fail(FA_ERR_INVALID_ARG, "combine pointer is NULL");
  if (((uintptr_t)o_part | (uintptr_t)out_bf16) & 15) return fail(FA_ERR_INVALID_ARG, "combine buffers must be 16-byte aligned");
  cudaError_t e = fa::launch_combine(o_part, lse_part, num_splits, n_rows, hq, dv, out_bf16, lse, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return FA_OK;
}

fa_status_t fa_fwd_varlen(const fa_tensor_t *q, const fa_tensor_t *k_cache, const fa_tensor_t *v_cache,
                          const fa_tensor_t *block_table, const fa_tensor_t *cu_seqlens_q,
                          const fa_tensor_t *cu_seqlens_k, const fa_tensor_t *k_scale, const fa_tensor_t *v_scale,
                          fa_tensor_t *out, fa_tensor_t *lse, float softmax_scale, int32_t causal, int32_t window,
                          const fa_score_mod_t *score_mod, const fa_block_mask_t *block_mask,
                          const fa_prologue_t *prologue, int32_t page_size, const fa_launch_t *launch, void *stream) {
  return fwd_build(q, k_cache, v_cache, block_table, cu_seqlens_q, cu_seqlens_k, k_scale, v_scale, out, lse,
                   softmax_scale, causal, window, score_mod, block_mask, prologue, page_size, launch, stream, nullptr);
}

fa_status_t fa_fwd_plan_create(const fa_tensor_t *q, const fa_tensor_t *k_cache, const fa_tensor_t *v_cache,
                               const fa_tensor_t *block_table, const fa_tensor_t *cu_seqlens_q,
                               const fa_tensor_t *cu_seqlens_k, const fa_tensor_t *k_scale,
                               const fa_tensor_t *v_scale, fa_tensor_t *out, fa_tensor_t *lse, float softmax_scale,
                               int32_t causal, int32_t window, const fa_score_mod_t *score_mod,
                               const fa_block_mask_t *block_mask, const fa_prologue_t *prologue, int32_t page_size,
                               const fa_launch_t *launch, fa_fwd_plan_t *plan) {
  if (!plan) return fail(FA_ERR_INVALID_ARG, "plan is NULL");
  *plan = nullptr;
  fa_fwd_plan_s *P = new (std::nothrow) fa_fwd_plan_s();
  if (!P) return fail(FA_ERR_INVALID_ARG, "out of host memory");
  const fa_status_t st = fwd_build(q, k_cache, v_cache, block_table, cu_seqlens_q, cu_seqlens_k, k_scale, v_scale,
                                   out, lse, softmax_scale, causal, window, score_mod, block_mask, prologue, page_size,
                                   launch, nullptr, P);
  if (st != FA_OK) {
    delete P;
    return st;
  }
  *plan = P;
  return FA_OK;
}

fa_status_t fa_fwd_plan_launch(fa_fwd_plan_t plan, void *stream) {
  g_msg[0] = 0;
  if (!plan) return fail(FA_ERR_INVALID_ARG, "plan is NULL");
  if (plan->kind == 1) return run_decode(plan->dl, *plan, (cudaStream_t)stream);
  if (plan->kind == 2) return run_prefill(plan->pl, *plan, (cudaStream_t)stream);
  return FA_OK;
}

void fa_fwd_plan_destroy(fa_fwd_plan_t plan) { delete plan; }

}  // extern "C"

namespace {

fa_status_t fwd_build(const fa_tensor_t *q, const fa_tensor_t *k_cache, const fa_tensor_t *v_cache,
                      const fa_tensor_t *block_table, const fa_tensor_t *cu_seqlens_q,
                      const fa_tensor_t *cu_seqlens_k, const fa_tensor_t *k_scale, const fa_tensor_t *v_scale,
                      fa_tensor_t *out, fa_tensor_t *lse, float softmax_scale, int32_t causal, int32_t window,
                      const fa_score_mod_t *score_mod, const fa_block_mask_t *block_mask,
                      const fa_prologue_t *prologue, int32_t page_size, const fa_launch_t *launch, void *stream,
                      fa_fwd_plan_s *plan) {
  fa_status_t st;
  g_msg[0] = 0;
  if (!launch) return fail(FA_ERR_INVALID_ARG, "launch is NULL");
  const int64_t B = launch->num_seqs;
  if (B < 0) return fail(FA_ERR_INVALID_ARG, "num_seqs < 0");
  // ---- q
  if (!q) return fail(FA_ERR_INVALID_ARG, "q is NULL");
  const int q_dt = q->dtype;
  if (q_dt != FA_BF16 && q_dt != FA_E4M3) return fail(FA_ERR_INVALID_ARG, "q dtype must be bf16 or e4m3");
  if ((st = check_tensor(q, "q", q_dt, 3))) return st;
  const int64_t Tq = q->shape[0], Hq = q->shape[1], Dk = q->shape[2];
  const int qsz = dtype_size(q_dt);
  if (Tq != launch->total_q) return fail(FA_ERR_INVALID_ARG, "q.shape[0]=%lld != launch.total_q=%lld", (long long)Tq, (long long)launch->total_q);
  if (q->stride[2] != 1 || (q->stride[1] * qsz) % 16 || (q->stride[0] * qsz) % 16)
    return fail(FA_ERR_INVALID_ARG, "q needs a contiguous last dim and strides that are multiples of 16 bytes");
  // ---- k/v: packed [T_k, Hkv, D], paged [N_pg, P_s, Hkv, D], or (byte
  // caches) the vectorized 5-D pages K [N_pg, Hkv, Dk/16, P_s, 16] and
  // V [N_pg, Hkv, P_s/16, Dv, 16]
  const bool paged = block_table != nullptr;
  if (!k_cache || !v_cache) return fail(FA_ERR_INVALID_ARG, "k_cache/v_cache is NULL");
  const bool vec5 = paged && k_cache->ndim == 5;
  const int kvnd = vec5 ? 5 : (paged ? 4 : 3);
  const int kv_dt = k_cache->dtype;
  if (kv_dt != FA_BF16 && kv_dt != FA_E4M3 && kv_dt != FA_I8)
    return fail(FA_ERR_INVALID_ARG, "k_cache dtype must be bf16, e4m3 or int8");
  if ((st = check_tensor(k_cache, "k_cache", kv_dt, kvnd))) return st;
  if ((st = check_tensor(v_cache, "v_cache", kv_dt, kvnd))) return st;
  int64_t Hkv, Dk2, Dv, cache_ps = 0;
  if (vec5) {
    if (kv_dt == FA_BF16) return fail(FA_ERR_UNSUPPORTED, "the vectorized 5-D layout is accepted for e4m3 and int8 caches");
    if (k_cache->shape[4] != 16 || v_cache->shape[4] != 16)
      return fail(FA_ERR_INVALID_ARG, "5-D k/v caches: the last dim holds 16 one-byte elements");
    Hkv = k_cache->shape[1];
    Dk2 = k_cache->shape[2] * 16;
    cache_ps = k_cache->shape[3];
    Dv = v_cache->shape[3];
    if (v_cache->shape[1] != Hkv || v_cache->shape[0] != k_cache->shape[0] || v_cache->shape[2] * 16 != cache_ps)
      return fail(FA_ERR_INVALID_ARG, "5-D k_cache [N_pg, Hkv, Dk/16, P_s, 16] and v_cache [N_pg, Hkv, P_s/16, Dv, 16] disagree");
  } else {
    Hkv = k_cache->shape[kvnd - 2];
    Dk2 = k_cache->shape[kvnd - 1];
    Dv = v_cache->shape[kvnd - 1];
    if (paged) cache_ps = k_cache->shape[1];
    if (v_cache->shape[kvnd - 2] != Hkv) return fail(FA_ERR_INVALID_ARG, "k_cache and v_cache disagree on Hkv");
    for (int i = 0; i < kvnd - 2; ++i)
      if (v_cache->shape[i] != k_cache->shape[i]) return fail(FA_ERR_INVALID_ARG, "k_cache and v_cache shapes disagree");
  }
  if (Dk2 != Dk) return fail(FA_ERR_INVALID_ARG, "k_cache head dim %lld != q head dim %lld", (long long)Dk2, (long long)Dk);
  if (Hkv <= 0 || Hq <= 0 || Hq % Hkv) return fail(FA_ERR_INVALID_ARG, "Hq=%lld must be a positive multiple of Hkv=%lld", (long long)Hq, (long long)Hkv);
  if (!supported_dims(Dk, Dv)) return fail(FA_ERR_UNSUPPORTED, "(Dk, Dv) = (%lld, %lld) is not compiled", (long long)Dk, (long long)Dv);
  // e4m3 Q: QK on the e4m3 bytes, which needs e4m3 keys; one head-dim pair.
  const bool q8 = q_dt == FA_E4M3;
  if (q8 && kv_dt != FA_E4M3) return fail(FA_ERR_UNSUPPORTED, "e4m3 q needs e4m3 k_cache/v_cache");
  if (q8 && !((Dk == 128 || Dk == 192) && Dv == 128))
    return fail(FA_ERR_UNSUPPORTED, "e4m3 q is compiled for (Dk, Dv) = (128, 128) and (192, 128)");
  if (q8 && launch->num_splits > 0) return fail(FA_ERR_UNSUPPORTED, "split-KV takes bf16 q; use num_splits = 0 with e4m3 q");
  const int esz = dtype_size(kv_dt);
  for (const fa_tensor_t *t : {k_cache, v_cache}) {
    if (t->stride[kvnd - 1] != 1) return fail(FA_ERR_INVALID_ARG, "k/v caches need a contiguous last dim");
    for (int i = 0; i < kvnd - 1; ++i)
      if ((t->stride[i] * esz) % 16) return fail(FA_ERR_INVALID_ARG, "k/v cache strides must be multiples of 16 bytes");
    if (((uintptr_t)t->data) & 15) return fail(FA_ERR_INVALID_ARG, "k/v cache base must be 16-byte aligned");
  }
  // ---- block table, lengths
  int64_t n_pages = 0, max_pages = 0;
  if (paged) {
    if ((st = check_tensor(block_table, "block_table", FA_I32, 2))) return st;
    if (block_table->shape[0] != B) return fail(FA_ERR_INVALID_ARG, "block_table has %lld rows, expected num_seqs=%lld", (long long)block_table->shape[0], (long long)B);
    if (block_table->stride[1] != 1 && block_table->shape[1] > 1) return fail(FA_ERR_INVALID_ARG, "block_table rows must be contiguous");
    max_pages = block_table->shape[1];
    n_pages = k_cache->shape[0];
    // Pages of >= 16 keys are landed by TMA boxes whose shared-memory
    // destinations stay 1024-byte aligned; pages of 1..8 keys take the row
    // gather (fa_gather.cuh), which e4m3 Q (keys straight into the MMA
    // operand with their scales) does not have.
    if (!is_pow2(page_size) || page_size < 1 || page_size > 1024)
      return fail(FA_ERR_UNSUPPORTED, "page_size %d: supported sizes are powers of two from 1 to 1024", page_size);
    if (q8 && page_size < 16) return fail(FA_ERR_UNSUPPORTED, "e4m3 q needs pages of at least 16 keys");
    if (cache_ps != page_size) return fail(FA_ERR_INVALID_ARG, "the k_cache page holds %lld keys, page_size=%d", (long long)cache_ps, page_size);
    if (vec5 && page_size < 16) return fail(FA_ERR_UNSUPPORTED, "the vectorized 5-D layout needs pages of at least 16 keys");
    if (vec5 && q8) return fail(FA_ERR_UNSUPPORTED, "e4m3 q reads keys in the token-major page layout only");
    if ((int64_t)launch->max_seqlen_k > max_pages * page_size) return fail(FA_ERR_INVALID_ARG, "max_seqlen_k exceeds block_table capacity");
    if (n_pages >= (int64_t(1) << 31)) return fail(FA_ERR_OVERFLOW, "num_pages must fit int32");
  }
  if ((st = check_tensor(cu_seqlens_q, "cu_seqlens_q", FA_I32, 1))) return st;
  if ((st = check_tensor(cu_seqlens_k, "cu_seqlens_k", FA_I32, 1))) return st;
  if (cu_seqlens_q->shape[0] != B + 1 || cu_seqlens_k->shape[0] != B + 1)
    return fail(FA_ERR_INVALID_ARG, "cu_seqlens must have num_seqs+1 = %lld entries", (long long)(B + 1));
  if (!contiguous(cu_seqlens_q) || !contiguous(cu_seqlens_k)) return fail(FA_ERR_INVALID_ARG, "cu_seqlens must be contiguous");
  if (launch->max_seqlen_q < 0 || launch->max_seqlen_k < 0 || launch->total_k < 0)
    return fail(FA_ERR_INVALID_ARG, "negative length in launch");
  if (Tq >= (int64_t(1) << 31) || launch->total_k >= (int64_t(1) << 31))
    return fail(FA_ERR_OVERFLOW, "total tokens must fit the int32 cu_seqlens");
  if (!paged && k_cache->shape[0] < launch->total_k) return fail(FA_ERR_INVALID_ARG, "packed k_cache has fewer rows than total_k");
  // ---- scales
  // e4m3 and int8 caches (byte values with per-token scales) share the
  // converter-warp kernel; `fp8` below means either.
  const bool fp8 = kv_dt == FA_E4M3 || kv_dt == FA_I8;
  if (fp8) {
    if (!k_scale || !v_scale) return fail(FA_ERR_INVALID_ARG, "e4m3 and int8 caches need k_scale and v_scale");
    // per token and kv head: [N_pg, P_s, Hkv] (paged, either page layout) or [T_k, Hkv]
    const int snd = paged ? 3 : 2;
    const int64_t want[3] = {k_cache->shape[0], paged ? cache_ps : Hkv, Hkv};
    for (const fa_tensor_t *s : {k_scale, v_scale}) {
      if ((st = check_tensor(s, "kv scale", FA_F32, snd))) return st;
      for (int i = 0; i < snd; ++i)
        if (s->shape[i] != want[i]) return fail(FA_ERR_INVALID_ARG, "kv scales must be [N_pg, P_s, Hkv] (paged) or [T_k, Hkv]");
      if (!contiguous(s)) return fail(FA_ERR_INVALID_ARG, "kv scales must be contiguous");
    }
  } else if (k_scale || v_scale) {
    return fail(FA_ERR_INVALID_ARG, "k_scale/v_scale are only valid with an e4m3 or int8 cache");
  }
  // ---- out, lse
  if ((st = check_tensor(out, "out", FA_BF16, 3))) return st;
  if (out->shape[0] != Tq || out->shape[1] != Hq || out->shape[2] != Dv)
    return fail(FA_ERR_INVALID_ARG, "out must be [%lld, %lld, %lld]", (long long)Tq, (long long)Hq, (long long)Dv);
  if (!contiguous(out)) return fail(FA_ERR_INVALID_ARG, "out must be contiguous");
  if (((uintptr_t)out->data) & 15) return fail(FA_ERR_INVALID_ARG, "out must be 16-byte aligned");
  if (lse) {
    if ((st = check_tensor(lse, "lse", FA_F32, 2))) return st;
    if (lse->shape[0] != Hq || lse->shape[1] != Tq) return fail(FA_ERR_INVALID_ARG, "lse must be [Hq=%lld, T_q=%lld]", (long long)Hq, (long long)Tq);
    if (!contiguous(lse)) return fail(FA_ERR_INVALID_ARG, "lse must be contiguous");
    if (overlaps(lse, out)) return fail(FA_ERR_INVALID_ARG, "lse must not alias out");
  }
  if (overlaps(out, q) || overlaps(out, k_cache) || overlaps(out, v_cache)) return fail(FA_ERR_INVALID_ARG, "out must not alias q/k/v");
  // ---- parameters
  if (!std::isfinite(softmax_scale)) return fail(FA_ERR_INVALID_ARG, "softmax_scale must be finite");
  int mod = 0;
  float slope = 0.f, cap = 0.f;
  if ((st = check_mods(score_mod, block_mask, launch, &mod, &slope, &cap))) return st;
  // ---- prologue: each chain composed to x -> a * x + b and folded (see
  // fa_prologue_t): a_q a_k into the score scale, the row term into the LSE
  // (or, under the soft-cap, into the capped score), the key term of a Q add
  // into a per-key array computed by a pre-pass, a_v and b_v into the output
  Folded fo;
  if ((st = fold_prologue(prologue, &fo))) return st;
  const bool col_bias = needs_col_bias(fo);
  if (q8 && (fo.bq != 0.0 || fo.bk != 0.0))
    return fail(FA_ERR_UNSUPPORTED, "prologue adds on q or k with e4m3 q");
  // ---- opt-in precision mode: P * V on e4m3 operands
  if (launch->flags & ~FA_FLAG_PV_E4M3) return fail(FA_ERR_INVALID_ARG, "unknown launch flags 0x%x", launch->flags);
  const bool pv8 = (launch->flags & FA_FLAG_PV_E4M3) != 0;
  if (pv8 && !q8) return fail(FA_ERR_UNSUPPORTED, "FA_FLAG_PV_E4M3 takes e4m3 q with e4m3 k/v caches");
  if (vec5 && col_bias) return fail(FA_ERR_UNSUPPORTED, "a prologue q add reads keys in the token-major page layout only");
  if (vec5 && mod == 2 && fo.bk != 0.0)
    return fail(FA_ERR_UNSUPPORTED, "a prologue k add under the soft-cap is not taken with the vectorized 5-D pages");
  float pro_vmul = (float)fo.av, pro_vadd = (float)fo.bv;
  float pro_lse_k = 0.f, pro_lse_c = 0.f, pro_row_k = 0.f, pro_row_c = 0.f, cb_factor = 0.f;
  {
    const double sc = softmax_scale;
    const double row_k = sc * fo.aq * fo.bk, row_c = sc * fo.bq * fo.bk * (double)Dk;
    // score units: log2 (the kernels' exponent), or 2u*log2(e) under the soft-cap
    const double unit = mod == 2 ? 2.0 * (double)fa::kLog2e / (double)cap : (double)fa::kLog2e;
    if (mod == 2) {
      pro_row_k = (float)(row_k * unit);
      pro_row_c = (float)(row_c * unit);
    } else {
      pro_lse_k = (float)row_k;
      pro_lse_c = (float)row_c;
    }
    cb_factor = (float)(sc * fo.bq * fo.ak * unit);
    softmax_scale = (float)(sc * fo.aq * fo.ak);
    if (!std::isfinite(softmax_scale) || !std::isfinite(cb_factor) || !std::isfinite(pro_row_k) ||
        !std::isfinite(pro_row_c) || !std::isfinite(pro_lse_k) || !std::isfinite(pro_lse_c))
      return fail(FA_ERR_INVALID_ARG, "prologue maps overflow the score scale");
  }
  if (window < 0) window = 0;
  if (B == 0 || Tq == 0) return FA_OK;
  if (launch->max_seqlen_q <= 0) return fail(FA_ERR_INVALID_ARG, "max_seqlen_q must be > 0 when total_q > 0");
  if (!q->data || !out->data || !cu_seqlens_q->data || !cu_seqlens_k->data)
    return fail(FA_ERR_INVALID_ARG, "a required data pointer is NULL");

  cudaStream_t s = (cudaStream_t)stream;
  const CUtensorMapDataType kv_tmdt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int group = (int)(Hq / Hkv);
  const bool have_keys = launch->total_k > 0 || (paged && n_pages > 0);
  // ---- workspace: [split-KV partials][prologue key terms][V-scale maxima]
  const size_t ws_split = split_part_bytes(launch, (int32_t)Hq, (int32_t)Dv);
  const size_t ws_cb = col_part_bytes(launch, (int32_t)Hkv, fo);
  const size_t ws_need = ws_split + ws_cb + vmax_part_bytes(launch, (int32_t)Hkv);
  // checked by each path after its own limits
  auto check_workspace = [&]() -> fa_status_t {
    if (ws_need == 0) return FA_OK;
    if (!launch->workspace || launch->workspace_bytes < ws_need)
      return fail(FA_ERR_INVALID_ARG, "this call needs a workspace of %zu bytes (fa_fwd_workspace_bytes)", ws_need);
    if ((uintptr_t)launch->workspace & 255) return fail(FA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    return FA_OK;
  };
  fa::ColBiasParams cbp;
  memset(&cbp, 0, sizeof cbp);
  float *col_bias_ptr = nullptr;
  const int64_t cb_ld = col_bias_ld(launch->max_seqlen_k);
  if (col_bias && launch->max_seqlen_k > 0 && have_keys) {
    if (B > 65535 || Hkv > 65535) return fail(FA_ERR_UNSUPPORTED, "a Q add needs num_seqs and Hkv <= 65535");
    col_bias_ptr = (float *)((char *)launch->workspace + ws_split);
    cbp.k = (const uint8_t *)k_cache->data;
    cbp.kv = kv_dt == FA_E4M3 ? 1 : (kv_dt == FA_I8 ? 2 : 0);
    cbp.s_page = k_cache->stride[0] * esz;
    cbp.s_slot = paged ? k_cache->stride[1] * esz : 0;
    cbp.s_head = k_cache->stride[kvnd - 2] * esz;
    cbp.block_table = paged ? (const int32_t *)block_table->data : nullptr;
    cbp.bt_stride = paged ? block_table->stride[0] : 0;
    cbp.max_pages = max_pages;
    cbp.page_size = paged ? page_size : 1;
    cbp.page_shift = paged ? ilog2(page_size) : 0;
    cbp.n_pages = paged ? n_pages : k_cache->shape[0];
    cbp.cu_k = (const int32_t *)cu_seqlens_k->data;
    cbp.k_scale = fp8 ? (const float *)k_scale->data : nullptr;
    cbp.dk = (int32_t)Dk;
    cbp.hkv = (int32_t)Hkv;
    cbp.num_seqs = (int32_t)B;
    cbp.ld = cb_ld;
    cbp.factor = cb_factor;
    cbp.out = col_bias_ptr;
    cbp.err = error_word();
  }

  // ------------------------------------------------------------ split-KV --
  if (launch->num_splits > 0) {
    const int S = launch->num_splits;
    if ((int64_t)launch->max_seqlen_q * group > fa::kDecRows)
      return fail(FA_ERR_UNSUPPORTED, "split-KV needs max_seqlen_q * Hq/Hkv <= %d", fa::kDecRows);
    if (Dk != Dv || (Dk != 64 && Dk != 128)) return fail(FA_ERR_UNSUPPORTED, "split-KV supports Dk = Dv in {64, 128}");
    if (B > 65535 || Hkv > 65535) return fail(FA_ERR_UNSUPPORTED, "too many sequences or kv heads for split-KV");
    if ((st = check_workspace())) return st;
    fa::DecodeLaunch L;
    memset(&L, 0, sizeof L);
    L.kv = kv_dt == FA_E4M3 ? 1 : (kv_dt == FA_I8 ? 2 : 0);
    L.rows8 = (int64_t)launch->max_seqlen_q * group <= 8;
    const int rows_box = paged ? (page_size < fa::kDecStageKeys ? page_size : fa::kDecStageKeys) : fa::kDecStageKeys;
    if (have_keys && fp8) {
      // byte caches: one box per page piece, all D bytes of a key; at D = 128
      // 128-byte swizzled (the kernel reads the bytes into MMA fragments)
      const CUtensorMapSwizzle kv8_swz = Dk == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
      if (vec5) {
        if ((st = make_vec5_maps(&L.tm_k, &L.tm_v, k_cache, v_cache, Dk, Dv, Hkv, page_size, n_pages,
                                 (uint32_t)rows_box, (uint32_t)(Dk / 16), (uint32_t)Dv, (uint32_t)(rows_box / 16))))
          return st;
      } else if (paged) {
        const uint64_t dk[4] = {(uint64_t)Dk, (uint64_t)Hkv, (uint64_t)page_size, (uint64_t)n_pages};
        const uint64_t sk[3] = {(uint64_t)(k_cache->stride[2]), (uint64_t)(k_cache->stride[1]), (uint64_t)(k_cache->stride[0])};
        const uint64_t sv[3] = {(uint64_t)(v_cache->stride[2]), (uint64_t)(v_cache->stride[1]), (uint64_t)(v_cache->stride[0])};
        const uint32_t box[4] = {(uint32_t)Dk, 1, (uint32_t)rows_box, 1};
        if ((st = make_map(&L.tm_k, kv_tmdt, 4, k_cache->data, dk, sk, box, "k8", kv8_swz))) return st;
        if ((st = make_map(&L.tm_v, kv_tmdt, 4, v_cache->data, dk, sv, box, "v8", kv8_swz))) return st;
      } else {
        const uint64_t dk[3] = {(uint64_t)Dk, (uint64_t)Hkv, (uint64_t)k_cache->shape[0]};
        const uint64_t sk[2] = {(uint64_t)(k_cache->stride[1]), (uint64_t)(k_cache->stride[0])};
        const uint64_t sv[2] = {(uint64_t)(v_cache->stride[1]), (uint64_t)(v_cache->stride[0])};
        const uint32_t box[3] = {(uint32_t)Dk, 1, (uint32_t)rows_box};
        if ((st = make_map(&L.tm_k, kv_tmdt, 3, k_cache->data, dk, sk, box, "k8", kv8_swz))) return st;
        if ((st = make_map(&L.tm_v, kv_tmdt, 3, v_cache->data, dk, sv, box, "v8", kv8_swz))) return st;
      }
    } else if (have_keys) {
      if (paged) {
        const uint64_t dk[4] = {(uint64_t)Dk, (uint64_t)Hkv, (uint64_t)page_size, (uint64_t)n_pages};
        const uint64_t sk[3] = {(uint64_t)(k_cache->stride[2] * esz), (uint64_t)(k_cache->stride[1] * esz), (uint64_t)(k_cache->stride[0] * esz)};
        const uint64_t sv[3] = {(uint64_t)(v_cache->stride[2] * esz), (uint64_t)(v_cache->stride[1] * esz), (uint64_t)(v_cache->stride[0] * esz)};
        const uint32_t box[4] = {64, 1, (uint32_t)rows_box, 1};
        if ((st = make_map(&L.tm_k, kv_tmdt, 4, k_cache->data, dk, sk, box, "k"))) return st;
        if ((st = make_map(&L.tm_v, kv_tmdt, 4, v_cache->data, dk, sv, box, "v"))) return st;
      } else {
        const uint64_t dk[3] = {(uint64_t)Dk, (uint64_t)Hkv, (uint64_t)k_cache->shape[0]};
        const uint64_t sk[2] = {(uint64_t)(k_cache->stride[1] * esz), (uint64_t)(k_cache->stride[0] * esz)};
        const uint64_t sv[2] = {(uint64_t)(v_cache->stride[1] * esz), (uint64_t)(v_cache->stride[0] * esz)};
        const uint32_t box[3] = {64, 1, (uint32_t)rows_box};
        if ((st = make_map(&L.tm_k, kv_tmdt, 3, k_cache->data, dk, sk, box, "k"))) return st;
        if ((st = make_map(&L.tm_v, kv_tmdt, 3, v_cache->data, dk, sv, box, "v"))) return st;
      }
    }
    fa::DecodeParams &p = L.p;
    p.q = (const __nv_bfloat16 *)q->data;
    p.q_stride_t = q->stride[0];
    p.q_stride_h = q->stride[1];
    p.cu_q = (const int32_t *)cu_seqlens_q->data;
    p.cu_k = (const int32_t *)cu_seqlens_k->data;
    p.block_table = paged ? (const int32_t *)block_table->data : nullptr;
    p.bt_stride = paged ? block_table->stride[0] : 0;
    p.page_size = paged ? page_size : fa::kDecStageKeys;
    p.page_shift = ilog2(p.page_size);
    p.rows_per_box = rows_box;
    p.boxes_per_stage = fa::kDecStageKeys / rows_box;
    p.gather = paged && page_size < 16;
    if (p.gather) {
      p.gk = kv_gather(k_cache, esz);
      p.gv = kv_gather(v_cache, esz);
    }
    p.pro_vmul = pro_vmul;
    p.pro_vadd = pro_vadd;
    p.pro_lse_k = pro_lse_k;
    p.pro_lse_c = pro_lse_c;
    p.pro_row_k = pro_row_k;
    p.pro_row_c = pro_row_c;
    p.col_bias = col_bias_ptr;
    p.cb_ld = cb_ld;
    p.vec5 = vec5;
    // the plain score loop has no per-key term: a Q add takes the general
    // path (ALiBi with slope 0)
    p.mod = (mod == 0 && col_bias_ptr) ? 1 : mod;
    p.alibi_log2 = mod == 1 ? slope * fa::kLog2e : 0.f;
    p.softcap_arg = mod == 2 ? softmax_scale / cap : 0.f;
    p.softcap_log2 = mod == 2 ? cap * fa::kLog2e : 0.f;
    p.block_mask = block_mask ? (const uint8_t *)block_mask->data : nullptr;
    p.n_qblk = block_mask ? block_mask->n_qblk : 0;
    p.n_kblk = block_mask ? block_mask->n_kblk : 0;
    p.hq = (int)Hq;
    p.hkv = (int)Hkv;
    p.group = group;
    int64_t split_keys = (launch->max_seqlen_k + S - 1) / S;
    split_keys = ((split_keys + fa::kDecStageKeys - 1) / fa::kDecStageKeys) * fa::kDecStageKeys;
    if (split_keys <= 0) split_keys = fa::kDecStageKeys;
    p.split_keys = (int)split_keys;
    p.num_splits = S;
    p.causal = causal != 0;
    p.window = window;
    p.total_q = Tq;
    p.scale_log2 = softmax_scale * fa::kLog2e;
    p.out = (__nv_bfloat16 *)out->data;
    p.out_stride_t = out->stride[0];
    p.out_stride_h = out->stride[1];
    p.lse = lse ? (float *)lse->data : nullptr;
    p.err = error_word();
    p.k_scale = fp8 ? (const float *)k_scale->data : nullptr;
    p.v_scale = fp8 ? (const float *)v_scale->data : nullptr;
    if (S > 1) {
      p.o_part = (float *)launch->workspace;
      p.lse_part = (float *)((char *)launch->workspace + align256((size_t)S * Tq * Hq * Dv * sizeof(float)));
    }
    L.grid = dim3((unsigned)S, (unsigned)Hkv, (unsigned)B);
    fa_fwd_plan_s local;
    fa_fwd_plan_s &P = plan ? *plan : local;
    P.kind = 1;
    P.dk = (int)Dk;
    P.has_cb = col_bias_ptr != nullptr;
    P.cb = cbp;
    P.splits = S;
    P.rows = Tq;
    P.hq = (int)Hq;
    P.dv = (int)Dv;
    P.out = out->data;
    P.dl = L;
    return plan ? FA_OK : run_decode(L, P, s);
  }

  // ------------------------------------------------------------ prefill --
  // Prefill kernels compute two 128-row query tiles per CTA, except the bf16
  // ping-pong kernel's one-tile form (tiles_per_cta): Dk = Dv in {64, 128},
  // no prologue score terms, pages of >= 16 keys.
  const bool terms = col_bias_ptr || pro_row_k != 0.f || pro_row_c != 0.f;
  int ntiles;
  {
    const bool eligible = !fp8 && !q8 && Dk == Dv && (Dk == 64 || Dk == 128) && !(paged && page_size < 16) && !terms;
    // average key tiles a query tile visits: keys per sequence, halved by a
    // causal mask, bounded by a window
    TileHints h;
    h.avg_key_tiles = (double)launch->total_k / (double)B / (double)fa::kBlockN;
    if (paged) h.avg_key_tiles = (double)launch->max_seqlen_k / (double)fa::kBlockN;
    if (causal) h.avg_key_tiles *= 0.5;
    if (window > 0)
      h.avg_key_tiles = std::min(h.avg_key_tiles, (double)(causal ? window : 2 * window) / fa::kBlockN + 1.0);
    h.n_tiles = ((double)Tq / (double)fa::kBlockM + (double)B) * (double)Hq;
    h.block_mask = block_mask != nullptr;
    h.causal = causal != 0;
    h.window = window > 0;
    h.mod = mod;
    ntiles = tiles_per_cta(eligible, prefill_variant(), h);
  }
  const int64_t rows_per_cta = ntiles * fa::kBlockM;
  const int64_t n_qtiles = (launch->max_seqlen_q + rows_per_cta - 1) / rows_per_cta;
  const int64_t head_group = Hq < 8 ? Hq : 8;
  const int64_t n_hgroups = (Hq + head_group - 1) / head_group;
  const int64_t n_blocks = B * n_hgroups * n_qtiles * head_group;
  if (n_blocks >= (int64_t(1) << 31)) return fail(FA_ERR_UNSUPPORTED, "grid too large");
  if ((st = check_workspace())) return st;
  fa::PrefillLaunch L;
  memset(&L, 0, sizeof L);
  {
    // bf16 Q: boxes of 64 columns (128 bytes); e4m3 Q: 128 columns.
    const uint64_t dq[3] = {(uint64_t)Dk, (uint64_t)Hq, (uint64_t)Tq};
    const uint64_t sq[2] = {(uint64_t)(q->stride[1] * qsz), (uint64_t)(q->stride[0] * qsz)};
    const uint32_t box[3] = {q8 ? 128u : 64u, 1, (uint32_t)fa::kBlockM};
    if (((uintptr_t)q->data) & 15) return fail(FA_ERR_INVALID_ARG, "q must be 16-byte aligned");
    if ((st = make_map(&L.tm_q, q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q->data,
                       dq, sq, box, "q")))
      return st;
  }
  const int rows_box = paged ? (page_size < fa::kBlockN ? page_size : fa::kBlockN) : fa::kBlockN;
  // e4m3: 64-byte row pieces (one 64-column block) in boxes of at most 32
  // rows, unswizzled; the converter warps turn each 32-row slice into the
  // swizzled f16 operand in place.  With e4m3 Q the keys are the MMA operand
  // as stored: whole 128-byte rows, 128-byte swizzled, in the same boxes.
  const int rows_box8 = paged ? (page_size < 32 ? page_size : 32) : 32;
  const uint32_t k8_cols = q8 ? 128u : 64u;
  const CUtensorMapSwizzle k8_swz = q8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
  if (have_keys && fp8) {
    if (vec5) {
      // staged byte rows for the converters: K boxes of 64 columns (4 groups
      // of 16), V boxes of 64 dims
      if ((st = make_vec5_maps(&L.tm_k, &L.tm_v, k_cache, v_cache, Dk, Dv, Hkv, page_size, n_pages,
                               (uint32_t)rows_box8, 4, 64, (uint32_t)(rows_box8 / 16))))
        return st;
    } else if (paged) {
      const uint64_t dk[4] = {(uint64_t)Dk, (uint64_t)Hkv, (uint64_t)page_size, (uint64_t)n_pages};
      const uint64_t dv[4] = {(uint64_t)Dv, (uint64_t)Hkv, (uint64_t)page_size, (uint64_t)n_pages};
      const uint64_t sk[3] = {(uint64_t)(k_cache->stride[2]), (uint64_t)(k_cache->stride[1]), (uint64_t)(k_cache->stride[0])};
      const uint64_t sv[3] = {(uint64_t)(v_cache->stride[2]), (uint64_t)(v_cache->stride[1]), (uint64_t)(v_cache->stride[0])};
      const uint32_t bk[4] = {k8_cols, 1, (uint32_t)rows_box8, 1};
      const uint32_t bv[4] = {64, 1, (uint32_t)rows_box8, 1};
      if ((st = make_map(&L.tm_k, kv_tmdt, 4, k_cache->data, dk, sk, bk, "k8", k8_swz))) return st;
      if ((st = make_map(&L.tm_v, kv_tmdt, 4, v_cache->data, dv, sv, bv, "v8", CU_TENSOR_MAP_SWIZZLE_NONE))) return st;
    } else {
      const uint64_t dk[3] = {(uint64_t)Dk, (uint64_t)Hkv, (uint64_t)k_cache->shape[0]};
      const uint64_t dv[3] = {(uint64_t)Dv, (uint64_t)Hkv, (uint64_t)v_cache->shape[0]};
      const uint64_t sk[2] = {(uint64_t)(k_cache->stride[1]), (uint64_t)(k_cache->stride[0])};
      const uint64_t sv[2] = {(uint64_t)(v_cache->stride[1]), (uint64_t)(v_cache->stride[0])};
      const uint32_t bk[3] = {k8_cols, 1, (uint32_t)rows_box8};
      const uint32_t bv[3] = {64, 1, (uint32_t)rows_box8};
      if ((st = make_map(&L.tm_k, kv_tmdt, 3, k_cache->data, dk, sk, bk, "k8", k8_swz))) return st;
      if ((st = make_map(&L.tm_v, kv_tmdt, 3, v_cache->data, dv, sv, bv, "v8", CU_TENSOR_MAP_SWIZZLE_NONE))) return st;
    }
  } else if (have_keys) {
    if (paged) {
      const uint64_t dk[4] = {(uint64_t)Dk, (uint64_t)Hkv, (uint64_t)page_size, (uint64_t)n_pages};
      const uint64_t dv[4] = {(uint64_t)Dv, (uint64_t)Hkv, (uint64_t)page_size, (uint64_t)n_pages};
      const uint64_t sk[3] = {(uint64_t)(k_cache->stride[2] * esz), (uint64_t)(k_cache->stride[1] * esz), (uint64_t)(k_cache->stride[0] * esz)};
      const uint64_t sv[3] = {(uint64_t)(v_cache->stride[2] * esz), (uint64_t)(v_cache->stride[1] * esz), (uint64_t)(v_cache->stride[0] * esz)};
      const uint32_t box[4] = {64, 1, (uint32_t)rows_box, 1};
      if ((st = make_map(&L.tm_k, kv_tmdt, 4, k_cache->data, dk, sk, box, "k"))) return st;
      if ((st = make_map(&L.tm_v, kv_tmdt, 4, v_cache->data, dv, sv, box, "v"))) return st;
    } else {
      const uint64_t dk[3] = {(uint64_t)Dk, (uint64_t)Hkv, (uint64_t)k_cache->shape[0]};
      const uint64_t dv[3] = {(uint64_t)Dv, (uint64_t)Hkv, (uint64_t)v_cache->shape[0]};
      const uint64_t sk[2] = {(uint64_t)(k_cache->stride[1] * esz), (uint64_t)(k_cache->stride[0] * esz)};
      const uint64_t sv[2] = {(uint64_t)(v_cache->stride[1] * esz), (uint64_t)(v_cache->stride[0] * esz)};
      const uint32_t box[3] = {64, 1, (uint32_t)fa::kBlockN};
      if ((st = make_map(&L.tm_k, kv_tmdt, 3, k_cache->data, dk, sk, box, "k"))) return st;
      if ((st = make_map(&L.tm_v, kv_tmdt, 3, v_cache->data, dv, sv, box, "v"))) return st;
    }
  }
  fa::PrefillParams &p = L.p;
  p.cu_q = (const int32_t *)cu_seqlens_q->data;
  p.cu_k = (const int32_t *)cu_seqlens_k->data;
  p.block_table = paged ? (const int32_t *)block_table->data : nullptr;
  p.bt_stride = paged ? block_table->stride[0] : 0;
  p.k_scale = fp8 ? (const float *)k_scale->data : nullptr;
  p.v_scale = fp8 ? (const float *)v_scale->data : nullptr;
  p.out = (__nv_bfloat16 *)out->data;
  p.out_stride_t = out->stride[0];
  p.out_stride_h = out->stride[1];
  p.lse = lse ? (float *)lse->data : nullptr;
  p.total_q = Tq;
  p.block_mask = block_mask ? block_mask->data : nullptr;
  p.n_qblk = block_mask ? block_mask->n_qblk : 0;
  p.n_kblk = block_mask ? block_mask->n_kblk : 0;
  p.num_seqs = (int)B;
  p.hq = (int)Hq;
  p.hkv = (int)Hkv;
  p.group = group;
  p.page_size = paged ? page_size : fa::kBlockN;
  p.page_shift = ilog2(p.page_size);
  p.rows_per_box = fp8 ? rows_box8 : rows_box;
  p.gather = paged && page_size < 16;
  if (p.gather) {
    p.gk = kv_gather(k_cache, esz);
    p.gv = kv_gather(v_cache, esz);
  }
  p.pro_vmul = pro_vmul;
  p.pro_vadd = pro_vadd;
  p.pro_lse_k = pro_lse_k;
  p.pro_lse_c = pro_lse_c;
  p.pro_row_k = pro_row_k;
  p.pro_row_c = pro_row_c;
  p.col_bias = col_bias_ptr;
  p.cb_ld = cb_ld;
  p.vec5 = vec5;
  // e4m3 P * V: the V-scale maxima, written by a pre-pass into the workspace
  fa::VmaxParams vmp;
  memset(&vmp, 0, sizeof vmp);
  if (pv8) {
    float *vmax_ptr = (float *)((char *)launch->workspace + ws_split + ws_cb);
    vmp.v_scale = (const float *)v_scale->data;
    vmp.block_table = paged ? (const int32_t *)block_table->data : nullptr;
    vmp.bt_stride = paged ? block_table->stride[0] : 0;
    vmp.max_pages = max_pages;
    vmp.page_size = paged ? page_size : 1;
    vmp.page_shift = paged ? ilog2(page_size) : 0;
    vmp.n_pages = paged ? n_pages : v_cache->shape[0];
    vmp.cu_k = (const int32_t *)cu_seqlens_k->data;
    vmp.hkv = (int32_t)Hkv;
    vmp.num_seqs = (int32_t)B;
    vmp.out = vmax_ptr;
    vmp.err = error_word();
    p.pv_vmax = vmax_ptr;
  }
  L.pv8 = pv8;
  p.q = (const __nv_bfloat16 *)q->data;
  p.q_stride_t = q->stride[0];
  p.q_stride_h = q->stride[1];
  p.pages_per_tile = fa::kBlockN / p.rows_per_box;
  p.n_qtiles = (int)n_qtiles;
  p.causal = causal != 0;
  p.window = window;
  p.scale_log2 = softmax_scale * fa::kLog2e;
  p.softcap_arg = mod == 2 ? softmax_scale / cap : 0.f;
  p.softcap_log2 = mod == 2 ? cap * fa::kLog2e : 0.f;
  p.alibi_log2 = mod == 1 ? slope * fa::kLog2e : 0.f;
  p.err = error_word();
  L.paged = paged;
  L.fp8 = fp8;
  L.int8 = kv_dt == FA_I8;
  L.q8 = q8;
  L.variant = prefill_variant();
  L.tiles_per_cta = ntiles;
  // The plain-softmax kernels fold a positive scale into the exponent and
  // have no per-key term; any other scale, and a Q add, take the general
  // score path (ALiBi with slope 0).  The prologue's score terms select the
  // kernels that carry them (mod 3: general score, 4: soft-cap).
  // The row term enters the kernels only under the soft-cap (as pro_row_*),
  // where it selects them too.
  int kmod = mod;
  if (mod == 0 && (!(softmax_scale > 0.f) || col_bias_ptr)) {
    kmod = 1;
    p.alibi_log2 = 0.f;
  }
  L.mod = terms ? kmod + 2 : kmod;
  // ALiBi with a positive scale on the ping-pong kernel (register-split
  // variants): the bias's linear part goes into the QK contraction (MOD 5)
  const bool alibi_mma_ok = !fp8 && !q8 && Dk == Dv && (Dk == 64 || Dk == 128);
  if (L.mod == 1 && mod == 1 && alibi_mma_ok && softmax_scale > 0.f && prefill_variant() != 1) L.mod = 5;
  p.head_group = (int)head_group;
  p.n_hgroups = (int)n_hgroups;
  p.n_items = (int)n_blocks;
  // One CTA per work item: the hardware hands items to SMs as they free up,
  // which balances ragged batches.
  L.grid = dim3((unsigned)n_blocks, 1, 1);
  fa_fwd_plan_s local;
  fa_fwd_plan_s &P = plan ? *plan : local;
  P.kind = 2;
  P.dk = (int)Dk;
  P.fp8 = fp8;
  P.has_cb = col_bias_ptr != nullptr;
  P.cb = cbp;
  P.has_vm = pv8 && B > 0;
  P.vm = vmp;
  P.pl = L;
  return plan ? FA_OK : run_prefill(L, P, s);
}

}  // namespace

// ------------------------------------------------------------- backward --
namespace {

// A bf16 [rows, heads, D] operand with a contiguous last dim and 16-byte
// aligned rows, as the TMA maps and the 16-byte stores need.
fa_status_t check_rows(const fa_tensor_t *t, const char *name, int64_t rows, int64_t heads, int64_t d) {
  fa_status_t st = check_tensor(t, name, FA_BF16, 3);
  if (st) return st;
  if (t->shape[0] != rows || t->shape[1] != heads || t->shape[2] != d)
    return fail(FA_ERR_INVALID_ARG, "%s has shape [%lld, %lld, %lld], expected [%lld, %lld, %lld]", name,
                (long long)t->shape[0], (long long)t->shape[1], (long long)t->shape[2], (long long)rows,
                (long long)heads, (long long)d);
  if (t->stride[2] != 1) return fail(FA_ERR_INVALID_ARG, "%s: last dim must be contiguous", name);
  if ((t->stride[0] % 8) || (t->stride[1] % 8) || (((uintptr_t)t->data) & 15))
    return fail(FA_ERR_INVALID_ARG, "%s: strides must be multiples of 8 elements and the base 16-byte aligned", name);
  if (!t->data && rows > 0) return fail(FA_ERR_INVALID_ARG, "%s data is NULL", name);
  return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_bwd_workspace_bytes(int64_t total_q, int32_t hq) {
  if (total_q <= 0 || hq <= 0) return 0;
  return align256((size_t)total_q * hq * sizeof(float));
}

fa_status_t fa_bwd_varlen(const fa_tensor_t *q, const fa_tensor_t *k, const fa_tensor_t *v, const fa_tensor_t *out,
                          const fa_tensor_t *dout, const fa_tensor_t *lse, const fa_tensor_t *cu_seqlens_q,
                          const fa_tensor_t *cu_seqlens_k, fa_tensor_t *dq, fa_tensor_t *dk, fa_tensor_t *dv,
                          float softmax_scale, int32_t causal, int32_t window, const fa_score_mod_t *score_mod,
                          const fa_block_mask_t *block_mask, const fa_launch_t *launch, void *stream) {
  g_msg[0] = 0;
  fa_status_t st;
  if (!launch) return fail(FA_ERR_INVALID_ARG, "launch is NULL");
  if (!q || !k || !v) return fail(FA_ERR_INVALID_ARG, "q, k and v are required");
  if ((st = check_tensor(q, "q", FA_BF16, 3))) return st;
  const int64_t B = launch->num_seqs, Tq = q->shape[0], Hq = q->shape[1], D = q->shape[2];
  if (k->ndim != 3) return fail(FA_ERR_INVALID_ARG, "k must be packed [T_k, Hkv, D] (no paged backward)");
  const int64_t Tk = k->shape[0], Hkv = k->shape[1];
  if (D != 64 && D != 128) return fail(FA_ERR_UNSUPPORTED, "backward supports Dk = Dv in {64, 128}, got %lld", (long long)D);
  if (Hkv <= 0 || Hq % Hkv) return fail(FA_ERR_INVALID_ARG, "Hq (%lld) must be a multiple of Hkv (%lld)", (long long)Hq, (long long)Hkv);
  if ((st = check_rows(q, "q", Tq, Hq, D)) || (st = check_rows(k, "k", Tk, Hkv, D)) ||
      (st = check_rows(v, "v", Tk, Hkv, D)) || (st = check_rows(out, "out", Tq, Hq, D)) ||
      (st = check_rows(dout, "dout", Tq, Hq, D)) || (st = check_rows(dq, "dq", Tq, Hq, D)) ||
      (st = check_rows(dk, "dk", Tk, Hkv, D)) || (st = check_rows(dv, "dv", Tk, Hkv, D)))
    return st;
  if ((st = check_tensor(lse, "lse", FA_F32, 2))) return st;
  if (lse->shape[0] != Hq || lse->shape[1] != Tq || !contiguous(lse))
    return fail(FA_ERR_INVALID_ARG, "lse must be contiguous fp32 [Hq, T_q] (the forward's LSE)");
  if ((st = check_tensor(cu_seqlens_q, "cu_seqlens_q", FA_I32, 1)) || (st = check_tensor(cu_seqlens_k, "cu_seqlens_k", FA_I32, 1)))
    return st;
  if (cu_seqlens_q->shape[0] != B + 1 || cu_seqlens_k->shape[0] != B + 1)
    return fail(FA_ERR_INVALID_ARG, "cu_seqlens must have num_seqs + 1 entries");
  if (launch->total_q != Tq) return fail(FA_ERR_INVALID_ARG, "launch->total_q != q.shape[0]");
  if (Tq >= (int64_t(1) << 31) || Tk >= (int64_t(1) << 31)) return fail(FA_ERR_OVERFLOW, "token counts must fit int32");
  const fa_tensor_t *outs[3] = {dq, dk, dv};
  const fa_tensor_t *ins[8] = {q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_k};
  for (const fa_tensor_t *o : outs)
    for (const fa_tensor_t *i : ins)
      if (overlaps(o, i)) return fail(FA_ERR_INVALID_ARG, "gradient buffers must not overlap the inputs");
  if (overlaps(dq, dk) || overlaps(dq, dv) || overlaps(dk, dv)) return fail(FA_ERR_INVALID_ARG, "dq, dk, dv overlap");
  if (window < 0) window = 0;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return fail(FA_ERR_INVALID_ARG, "softmax_scale must be positive and finite");
  int mod = 0;
  float slope = 0.f, cap = 0.f;
  if ((st = check_mods(score_mod, block_mask, launch, &mod, &slope, &cap))) return st;
  if (B == 0 || Tq == 0) return FA_OK;
  if (launch->max_seqlen_q <= 0 || launch->max_seqlen_k < 0) return fail(FA_ERR_INVALID_ARG, "bad max_seqlen");
  if (B > 65535 || Hq > 65535) return fail(FA_ERR_UNSUPPORTED, "num_seqs and Hq must be at most 65535");
  const size_t need = fa_bwd_workspace_bytes(Tq, (int)Hq);
  if (!launch->workspace || launch->workspace_bytes < need)
    return fail(FA_ERR_INVALID_ARG, "the backward needs a workspace of %zu bytes (fa_bwd_workspace_bytes)", need);
  if ((uintptr_t)launch->workspace & 255) return fail(FA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");

  fa::BwdLaunch L;
  memset(&L, 0, sizeof L);
  {
    const uint32_t box[3] = {64, 1, 128};
    const fa_tensor_t *ts[4] = {q, k, v, dout};
    CUtensorMap *ms[4] = {&L.tm_q, &L.tm_k, &L.tm_v, &L.tm_do};
    const char *names[4] = {"q", "k", "v", "dout"};
    for (int x = 0; x < 4; ++x) {
      const fa_tensor_t *t = ts[x];
      const uint64_t dims[3] = {(uint64_t)D, (uint64_t)t->shape[1], (uint64_t)t->shape[0]};
      const uint64_t strides[2] = {(uint64_t)(t->stride[1] * 2), (uint64_t)(t->stride[0] * 2)};
      if (t->shape[0] == 0) continue;
      if ((st = make_map(ms[x], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, t->data, dims, strides, box, names[x]))) return st;
    }
  }
  float *delta = (float *)launch->workspace;
  fa::BwdParams &p = L.p;
  p.cu_q = (const int32_t *)cu_seqlens_q->data;
  p.cu_k = (const int32_t *)cu_seqlens_k->data;
  p.lse = (const float *)lse->data;
  p.delta = delta;
  p.dq = (__nv_bfloat16 *)dq->data;
  p.dq_stride_t = dq->stride[0];
  p.dq_stride_h = dq->stride[1];
  p.dk = (__nv_bfloat16 *)dk->data;
  p.dk_stride_t = dk->stride[0];
  p.dk_stride_h = dk->stride[1];
  p.dv = (__nv_bfloat16 *)dv->data;
  p.dv_stride_t = dv->stride[0];
  p.dv_stride_h = dv->stride[1];
  p.total_q = Tq;
  p.num_seqs = (int)B;
  p.hq = (int)Hq;
  p.hkv = (int)Hkv;
  p.group = (int)(Hq / Hkv);
  p.n_qtiles = (launch->max_seqlen_q + 127) / 128;
  p.n_ktiles = (launch->max_seqlen_k + 127) / 128;
  p.causal = causal != 0;
  p.window = window;
  p.scale = softmax_scale;
  p.scale_log2 = softmax_scale * fa::kLog2e;
  p.err = error_word();
  p.softcap_arg = mod == 2 ? softmax_scale / cap : 0.f;
  p.softcap_log2 = mod == 2 ? cap * fa::kLog2e : 0.f;
  p.alibi_log2 = mod == 1 ? slope * fa::kLog2e : 0.f;
  p.block_mask = block_mask ? (const uint8_t *)block_mask->data : nullptr;
  p.n_qblk = block_mask ? block_mask->n_qblk : 0;
  p.n_kblk = block_mask ? block_mask->n_kblk : 0;
  L.mod = mod;
  fa::BwdDeltaParams &dp = L.dp;
  dp.out = (const __nv_bfloat16 *)out->data;
  dp.dout = (const __nv_bfloat16 *)dout->data;
  dp.o_stride_t = out->stride[0];
  dp.o_stride_h = out->stride[1];
  dp.do_stride_t = dout->stride[0];
  dp.do_stride_h = dout->stride[1];
  dp.delta = delta;
  dp.total_q = Tq;
  dp.hq = (int)Hq;
  dp.d = (int)D;
  L.delta_blocks = (unsigned)((Tq * Hq + 31) / 32);   // 32 rows per 256-thread block
  L.grid_q = dim3((unsigned)p.n_qtiles, (unsigned)Hq, (unsigned)B);
  L.grid_kv = dim3((unsigned)(p.n_ktiles > 0 ? p.n_ktiles : 1), (unsigned)Hkv, (unsigned)B);
  L.stream = (cudaStream_t)stream;
  cudaError_t e = fa::launch_bwd((int)D, L);
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  return FA_OK;
}

}  // extern "C"
