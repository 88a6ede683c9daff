/*
 * fa_gb300.h -- C ABI of the GB300 (sm_103a) attention forward library.
 *
 * One operation, in several entry points: the FlashAttention forward pass
 * over packed variable-length sequences and a paged KV cache, with per-row
 * log-sum-exp output.  For query row i of sequence b and head h:
 *
 *   out[i]  = sum_j softmax_j(s_ij) * v_j        over the keys j the mask allows
 *   lse[i]  = log sum_j exp(s_ij)                (natural log)
 *   s_ij    = scale * <q_i, k_j>, then soft-cap, then ALiBi
 *
 * The passages that define it:
 *  - tiled QK^T, online (running max / running sum) softmax, PV and the
 *    attention-domain LSE = M + log(L) over packed cu_seqlens tensors
 *    [total_tokens, H, D]: RL-Kernel PR #237 "SM90 TMA + mma.sync
 *    FlashAttention", commit texts and summary;
 *  - the LSE written also for fully masked rows, and the split-K combine
 *    m_max*ln2 + ln(den): FlyDSL PR #844 "Add forward LSE output", Changes;
 *  - paged KV addressed through block_table, FP8 e4m3 KV with scales,
 *    Q/K head dim 192 with V/O 128 at native BF16 width, bottom-right causal
 *    mask, offsets above 4 GiB: FlyDSL PR #1066 "Support paged FP8 Flash
 *    attention with asymmetric K/V head dim", overview, review and PR
 *    description;
 *  - per-token fp8 scale max|row|/448, ALiBi, SoftCap, SlidingWindow and
 *    128x128 block sparsity: fkl_python PR #7 "flash_attention: prologue
 *    fusion, mma tensor cores, fp8 KV cache, flex attention + block
 *    sparsity", commits and summary.
 *
 * Conventions for every entry point:
 *  - Pointers inside fa_tensor_t are DEVICE pointers on the current CUDA
 *    device, owned by the caller.  The library never frees them and keeps no
 *    reference after the call returns.
 *  - Calls are asynchronous: work is enqueued on `stream` (a cudaStream_t
 *    passed as void*, NULL = legacy default stream) and the call returns.
 *    The library performs no host<->device copy, no device synchronisation
 *    and no memory allocation inside fa_fwd_varlen / fa_combine.
 *  - All validation happens on the host before any launch, using the shapes
 *    in fa_tensor_t and the host scalars in fa_launch_t.  On any non-OK
 *    status nothing has been enqueued; fa_last_error() describes the cause.
 *  - Device-side waits are bounded.  A wait that runs out, or an index that
 *    the kernel finds out of range, records a code in a per-device error word
 *    read by fa_get_device_error(); the kernel then returns early.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

/* Every entry point below is exported; the library is built with hidden
 * visibility for everything else (kernels, templates, helpers), so that two
 * copies loaded into one process do not bind to each other's internals. */
#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,    /* malformed shape, dtype, stride or pointer */
    FA_ERR_UNSUPPORTED = 2,    /* valid request outside the compiled variant set */
    FA_ERR_OVERFLOW = 3,       /* a size that does not fit the index types */
    FA_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed */
    FA_ERR_DEVICE_TIMEOUT = 5, /* (device word) a bounded wait ran out */
    FA_ERR_DEVICE_BOUNDS = 6   /* (device word) an index was out of range */
} fa_status_t;

typedef enum { FA_BF16 = 0, FA_E4M3 = 1, FA_F32 = 2, FA_I32 = 3, FA_U8 = 4, FA_I8 = 5 } fa_dtype_t;

/* A strided device tensor.  Strides are in ELEMENTS; shape[ndim..4] unused. */
typedef struct {
    void *data;
    int32_t dtype;       /* fa_dtype_t */
    int32_t ndim;
    int64_t shape[5];
    int64_t stride[5];
} fa_tensor_t;

/* Score modifier (fkl_python PR #7, flex commit): kind 0 none, 1 ALiBi
 * (s -= alibi_slope * |i' - j|, i' = i + Sk - Sq), 2 soft-cap
 * (s = softcap * tanh(s / softcap), on the scaled score, before ALiBi). */
typedef struct {
    int32_t kind;
    float alibi_slope;
    float softcap;
} fa_score_mod_t;

/* Prologue (fkl_python PR #7, prologue-fusion commit: op chains fused onto
 * the Q/K/V reads, values passed at run time).  Each tensor has a chain of
 * up to FA_PROLOGUE_MAX_OPS scalar ops, applied in order to every element as
 * it is read: FA_OP_MUL (x * value), FA_OP_ADD (x + value), FA_OP_SUB
 * (x - value), FA_OP_DIV (x / value).  n_q, n_k, n_v give the chain lengths
 * (0 = no op on that tensor).
 *
 * The library composes each chain into one map x -> a * x + b (in double
 * precision, on the host) and folds the maps instead of rewriting the
 * operands, which is exact in real arithmetic.  With q' = a_q q + b_q and
 * k' = a_k k + b_k the score scale * <q'_i, k'_j> is
 *   scale a_q a_k <q_i, k_j>                 (the scale is multiplied)
 *   + scale (a_q b_k sum_d q_i[d] + b_q b_k Dk)   (one term per query row)
 *   + scale b_q a_k sum_d k_j[d]             (one term per key),
 * and with v' = a_v v + b_v the output is a_v out + b_v (softmax weights sum
 * to 1).  The row term cancels in the softmax and is added to the LSE, or,
 * under the soft-cap (not shift-invariant), enters the capped score.  The key
 * term (a Q add) is computed by a pre-pass over the keys into the caller's
 * workspace (fa_fwd_workspace_bytes() includes it) and added to each score.
 * Rows that see no key keep out = 0 and LSE = -inf.
 * Limits: FA_ERR_INVALID_ARG for an unknown op, a chain longer than
 * FA_PROLOGUE_MAX_OPS, a value that is not finite or a division by 0;
 * FA_ERR_UNSUPPORTED for b_q or b_k != 0 with e4m3 q.  NULL, or empty chains,
 * is no prologue. */
enum { FA_OP_MUL = 1, FA_OP_ADD = 2, FA_OP_SUB = 3, FA_OP_DIV = 4 };
#define FA_PROLOGUE_MAX_OPS 8
typedef struct {
    int32_t op;          /* FA_OP_* */
    float value;
} fa_prologue_op_t;
typedef struct {
    int32_t n_q, n_k, n_v;
    fa_prologue_op_t q[FA_PROLOGUE_MAX_OPS];
    fa_prologue_op_t k[FA_PROLOGUE_MAX_OPS];
    fa_prologue_op_t v[FA_PROLOGUE_MAX_OPS];
} fa_prologue_t;

/* 128x128 block-sparsity mask, uint8 [num_seqs * Hq][n_qblk][n_kblk],
 * contiguous; block (qb, kb) of sequence b, head h is active when
 * data[((b*Hq + h)*n_qblk + qb)*n_kblk + kb] != 0, with qb = i/128 and
 * kb = j/128 in sequence-local indices.  blk_q = blk_k = 128 only. */
typedef struct {
    const uint8_t *data;
    int32_t n_qblk, n_kblk, blk_q, blk_k;
} fa_block_mask_t;

/* Opt-in precision mode (fa_launch_t.flags): P * V on e4m3 operands
 * (FlyDSL PR #1066, Technical Details and Test Result: direct FP8 P x V at V
 * head dim 128, with its larger error).  Taken with e4m3 q and e4m3 K/V,
 * (Dk, Dv) in {(128, 128), (192, 128)}, token-major pages or packed K/V, no
 * prologue and a single pass (num_splits 0); FA_ERR_UNSUPPORTED otherwise.
 * The attention weights go to e4m3 as p * v_scale / 2^e, with 2^e above the
 * largest V scale of the sequence (a pre-pass over the V scales, writing one
 * fp32 per (sequence, kv head) into the workspace), and P * V runs on the
 * tensor core's e4m3 path with fp32 accumulation; the row sums and the LSE
 * stay fp32.  Each weight carries up to 2^-4 relative rounding, so outputs
 * differ from the exact attention by more than in the default mode (the
 * tests hold them to 4e-2; the LSE keeps its 1e-3). */
#define FA_FLAG_PV_E4M3 1

/* Host-side scalars, so that no length is read back from the device.
 * num_splits: 0 = single pass; > 0 = split-KV over that many key ranges
 * followed by the combine.  workspace: fa_fwd_workspace_bytes() bytes, needed
 * by split-KV with 2 or more splits, by a prologue with a Q add and by
 * FA_FLAG_PV_E4M3.  flags: 0, or FA_FLAG_PV_E4M3. */
typedef struct {
    int32_t num_seqs;
    int32_t max_seqlen_q;
    int32_t max_seqlen_k;
    int32_t num_splits;
    int64_t total_q;
    int64_t total_k;
    void *workspace;         /* device, 256-byte aligned, caller-owned */
    size_t workspace_bytes;
    int32_t flags;
} fa_launch_t;

/*
 * fa_fwd_varlen -- the attention forward pass.
 *
 *  q            bf16 [T_q, Hq, Dk], or e4m3 [T_q, Hq, Dk] with e4m3 caches,
 *               Dk 128 or 192 and Dv 128 (FlyDSL PR #1066 description: E4M3
 *               Q/K/V with scalar descales; the caller folds the Q descale
 *               into softmax_scale, and QK runs on the e4m3 bytes with the
 *               per-key scale applied to each score).  Last dim contiguous, the other
 *               strides multiples of 16 bytes.  Split-KV takes bf16 q only
 *               (Dk = Dv in {64, 128}); score mods, block masks and
 *               prologues apply to it as to the single pass.
 *  k_cache      paged: [N_pg, P_s, Hkv, Dk]; packed (block_table NULL):
 *               [T_k, Hkv, Dk].  bf16, e4m3 or int8.  Last three dims contiguous.
 *  v_cache      same layout and dtype with Dv (Dv may differ from Dk).
 *               Paged e4m3 and int8 caches may instead come in the
 *               vectorized 5-D layouts (FlyDSL PR #1066, Technical Details
 *               and review): K [N_pg, Hkv, Dk/16, P_s, 16] and V [N_pg, Hkv,
 *               P_s/16, Dv, 16], contiguous, 16 one-byte elements in the last
 *               dim, with pages of >= 16 keys and k_scale/v_scale
 *               [N_pg, P_s, Hkv]; results are bit-identical to the
 *               token-major pages.  Not with e4m3 q, a prologue add on q, or
 *               an add on k under the soft-cap (FA_ERR_UNSUPPORTED).
 *  block_table  int32 [num_seqs, max_pages], or NULL for packed K/V.  Entries
 *               for pages past a sequence's length are never read.
 *  cu_seqlens_q int32 [num_seqs + 1], prefix sums of query lengths.
 *  cu_seqlens_k int32 [num_seqs + 1], prefix sums of key lengths (row offsets
 *               into packed K/V; with a block table only their differences,
 *               the lengths, are used).
 *  k_scale      fp32 per token and kv head, [N_pg, P_s, Hkv] (paged) or
 *  v_scale      [T_k, Hkv] (packed); required for e4m3, must be NULL for bf16.
 *               The dequantised key is e4m3(k) * k_scale (same for v).
 *  out          bf16 [T_q, Hq, Dv], contiguous, caller-allocated; rows whose
 *               allowed key set is empty are written as 0.
 *  lse          fp32 [Hq, T_q] contiguous, or NULL to skip; -inf for rows
 *               with no allowed key.
 *  softmax_scale  multiplies <q, k>.
 *  causal       non-zero: key j visible iff j <= i + Sk - Sq (bottom-right).
 *  window       > 0: sliding window of `window` keys including the diagonal
 *               (causal: i' - j < window; otherwise |i' - j| < window).
 *  score_mod    NULL or fa_score_mod_t.
 *  block_mask   NULL or fa_block_mask_t.
 *  prologue     NULL or fa_prologue_t.
 *  page_size    tokens per page when paged: a power of two, 1 ... 1024.
 *               Pages of 16 or more keys are landed by TMA boxes; pages of
 *               1 ... 8 keys are gathered key row by key row (same results,
 *               bit for bit; slower).  e4m3 q needs pages of >= 16 keys.
 *  launch       host scalars (required).
 *  stream       cudaStream_t.
 *
 * e4m3 caches: K and V become f16 operands RN(e4m3 * scale) inside the
 * kernel, so |e4m3 value * scale| must stay below 65504 (scales below 146).
 *
 * Supported head dims: (Dk, Dv) in {(64,64), (128,128), (192,128)}.  Hq must
 * be a multiple of Hkv (query head h reads kv head h / (Hq/Hkv)).
 * Returns FA_OK or an error status; see fa_last_error().
 */
FA_API fa_status_t fa_fwd_varlen(const fa_tensor_t *q, const fa_tensor_t *k_cache,
                          const fa_tensor_t *v_cache, const fa_tensor_t *block_table,
                          const fa_tensor_t *cu_seqlens_q, const fa_tensor_t *cu_seqlens_k,
                          const fa_tensor_t *k_scale, const fa_tensor_t *v_scale,
                          fa_tensor_t *out, fa_tensor_t *lse, float softmax_scale,
                          int32_t causal, int32_t window, const fa_score_mod_t *score_mod,
                          const fa_block_mask_t *block_mask, const fa_prologue_t *prologue,
                          int32_t page_size, const fa_launch_t *launch, void *stream);

/*
 * Prepared calls.  fa_fwd_plan_create validates a forward call exactly like
 * fa_fwd_varlen (same arguments except the stream) and records the launches
 * it would make -- tensor maps, kernel parameters, grid -- without enqueuing
 * anything.  fa_fwd_plan_launch enqueues them on `stream`: the host work of a
 * call drops to the kernel launches, which matters for small problems issued
 * repeatedly (decode loops, serving).  The plan keeps the device addresses of
 * every tensor and of the workspace: they must stay allocated, unmoved and of
 * the same shape while the plan is used, and their contents are read at each
 * launch.  A plan runs on the device that was current at creation.  Launching
 * a plan on two streams at once is allowed only without a workspace (split-KV
 * partials would race).  fa_fwd_plan_destroy frees the host-side plan (NULL is
 * a no-op).  Status and error reporting as for fa_fwd_varlen.
 */
typedef struct fa_fwd_plan_s *fa_fwd_plan_t;

FA_API fa_status_t fa_fwd_plan_create(const fa_tensor_t *q, const fa_tensor_t *k_cache, const fa_tensor_t *v_cache,
                               const fa_tensor_t *block_table, const fa_tensor_t *cu_seqlens_q,
                               const fa_tensor_t *cu_seqlens_k, const fa_tensor_t *k_scale,
                               const fa_tensor_t *v_scale, fa_tensor_t *out, fa_tensor_t *lse,
                               float softmax_scale, int32_t causal, int32_t window,
                               const fa_score_mod_t *score_mod, const fa_block_mask_t *block_mask,
                               const fa_prologue_t *prologue, int32_t page_size, const fa_launch_t *launch,
                               fa_fwd_plan_t *plan);
FA_API fa_status_t fa_fwd_plan_launch(fa_fwd_plan_t plan, void *stream);
FA_API void fa_fwd_plan_destroy(fa_fwd_plan_t plan);

/*
 * Workspace size in bytes of a forward call with these host scalars, head
 * counts and prologue (NULL = none): for split-KV with launch->num_splits >= 2,
 * partial outputs fp32 [num_splits, T_q, Hq, Dv] and partial LSEs fp32
 * [num_splits, Hq, T_q]; for a prologue whose Q chain adds a constant (see
 * fa_prologue_t), the per-key score terms fp32 [num_seqs, Hkv,
 * ceil(max_seqlen_k / 128) * 128].  Each part is 256-byte aligned.  0 when
 * neither applies or launch is NULL.
 */
FA_API size_t fa_fwd_workspace_bytes(const fa_launch_t *launch, int32_t hq, int32_t hkv, int32_t dv,
                              const fa_prologue_t *prologue);

/*
 * Recommended split count for a problem (0 = single pass).  Split-KV applies
 * when few query rows share each kv head (decode: max_seqlen_q * Hq/Hkv <= 16)
 * and keys are long.  The key ranges are sized so that the non-empty CTAs make
 * about three waves at two CTAs per SM of the current device; total_k (the
 * sum of key lengths, 0 if unknown) refines the estimate of non-empty ranges.
 */
FA_API int32_t fa_fwd_default_splits(int32_t num_seqs, int32_t max_seqlen_q, int32_t max_seqlen_k,
                              int64_t total_k, int32_t hq, int32_t hkv, int32_t page_size);

/*
 * fa_combine -- merge of partial results over disjoint key ranges (the
 * split-KV combine; FlyDSL PR #844, Changes: m_max*ln2 + ln(den)):
 *   LSE = ln sum_s exp(LSE_s),  out = sum_s exp(LSE_s - LSE) * O_s,
 * partials with LSE_s = -inf are skipped; all -inf gives out 0, LSE -inf.
 *  o_part   fp32 [num_splits, n_rows, Hq, Dv] contiguous (n_rows = T_q)
 *  lse_part fp32 [num_splits, Hq, n_rows] contiguous
 *  out      bf16 [n_rows, Hq, Dv] contiguous;  lse fp32 [Hq, n_rows] or NULL.
 */
FA_API fa_status_t fa_combine(const float *o_part, const float *lse_part, int32_t num_splits,
                       int64_t n_rows, int32_t hq, int32_t dv, void *out_bf16, float *lse,
                       void *stream);

/*
 * fa_bwd_varlen -- the backward pass: gradients of L = sum(dout * out) with
 * respect to q, k and v, recomputed from the forward's saved LSE
 * (RL-Kernel PR #237, backward commit: a Delta preprocess, then dQ/dK/dV from
 * the saved LSE):
 *   Delta_i = <dout_i, out_i>,   P_ij = exp(softmax_scale * <q_i, k_j> - LSE_i)
 *   dP_ij = <dout_i, v_j>,   dS_ij = P_ij * (dP_ij - Delta_i)
 *   dv_j = sum_i P_ij dout_i,  dk_j = softmax_scale * sum_i dS_ij q_i,
 *   dq_i = softmax_scale * sum_j dS_ij k_j      (allowed (i, j) only)
 * With a score mod, P uses the modified score s_ij.  ALiBi leaves dS as
 * written; the soft-cap s = cap * tanh(u / cap), u = softmax_scale <q, k>,
 * multiplies dS_ij by ds/du = 1 - tanh^2(u_ij / cap).
 *
 *  q, out, dout, dq   bf16 [T_q, Hq, D];  k, v, dk, dv   bf16 [T_k, Hkv, D],
 *                     packed varlen (no block table).  D = 64 or 128 (Dk = Dv).
 *                     Last dim contiguous, other strides multiples of 8
 *                     elements, bases 16-byte aligned.  GQA: Hq % Hkv == 0;
 *                     dk, dv sum over the q heads of each kv head's group.
 *  lse                fp32 [Hq, T_q] contiguous, the forward's LSE for the
 *                     same (q, k, v, masks).
 *  cu_seqlens_q/k     int32 [num_seqs + 1] (row offsets of q and of k/v).
 *  softmax_scale      > 0;  causal, window, score_mod (NULL or kind 0, 1, 2)
 *                     and block_mask (NULL or 128 x 128 blocks) as in
 *                     fa_fwd_varlen: a skipped block adds nothing to any
 *                     gradient.
 *  launch             num_seqs, max_seqlen_q/k, total_q (= T_q) and a
 *                     workspace of fa_bwd_workspace_bytes(T_q, Hq) bytes,
 *                     256-byte aligned, for Delta (fp32 [Hq, T_q]).
 * Outputs are overwritten (rows of keys or queries that see nothing get 0)
 * and must not overlap any input or each other.  Three kernels are enqueued
 * on `stream` (Delta, dK/dV, dQ); no allocation, copy or synchronisation.
 * Errors as for fa_fwd_varlen: FA_ERR_INVALID_ARG for shapes, dtypes,
 * strides, alignment or a missing workspace, FA_ERR_UNSUPPORTED for other
 * head dims, FA_ERR_CUDA for launch failures.
 */
FA_API fa_status_t fa_bwd_varlen(const fa_tensor_t *q, const fa_tensor_t *k, const fa_tensor_t *v,
                          const fa_tensor_t *out, const fa_tensor_t *dout, const fa_tensor_t *lse,
                          const fa_tensor_t *cu_seqlens_q, const fa_tensor_t *cu_seqlens_k,
                          fa_tensor_t *dq, fa_tensor_t *dk, fa_tensor_t *dv, float softmax_scale,
                          int32_t causal, int32_t window, const fa_score_mod_t *score_mod,
                          const fa_block_mask_t *block_mask, const fa_launch_t *launch, void *stream);

/* Workspace bytes of fa_bwd_varlen: Delta, fp32 [Hq, T_q], rounded up to 256. */
FA_API size_t fa_bwd_workspace_bytes(int64_t total_q, int32_t hq);

/*
 * fa_fwd_varlen_noalloc -- the split-KV decode of fa_fwd_varlen for callers
 * that cannot allocate device memory.  (The pages have no counterpart: this
 * entry exists for deployment, not for the method.)
 *
 * Who needs it: custom ops and plugins that are handed only their input and
 * output buffers, serving loops whose device memory is fixed at start-up, and
 * request paths that must not call cudaMalloc because it may synchronise the
 * device or fail under memory pressure.  Instead of launch->workspace, the
 * per-split partials go to a static device array of FA_NOALLOC_SCRATCH_BYTES
 * owned by the library.  The array is part of the library's device code:
 * CUDA reserves it on a device when it loads the library's code there, which
 * under lazy module loading (the default since CUDA 12) happens at the first
 * use on that device -- possibly this entry's first call -- and it stays
 * reserved until the process exits.  Callers with no spare device memory
 * should therefore make one call per device at start-up.  The call itself
 * asks for no memory: no cudaMalloc, no allocating library routine.
 *
 * Arguments and layouts are those of fa_fwd_varlen; launch->workspace and
 * launch->workspace_bytes are ignored.  launch->num_splits <= 0 picks
 * fa_fwd_default_splits(); the problem must be a split-KV decode shape with
 * at least 2 splits, and fa_fwd_workspace_bytes() for it (with q.shape[0]
 * rows, which must equal launch->total_q) must not exceed
 * FA_NOALLOC_SCRATCH_BYTES, else FA_ERR_UNSUPPORTED is returned with nothing
 * enqueued.
 *
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * Every call shares the one array and leaves its partials there: calls whose
 * work overlaps on the GPU (different streams, or the same stream from several
 * host threads without ordering) race on it.  No part of the array needs to
 * start at zero.
 */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
FA_API fa_status_t fa_fwd_varlen_noalloc(const fa_tensor_t *q, const fa_tensor_t *k_cache,
                                  const fa_tensor_t *v_cache, const fa_tensor_t *block_table,
                                  const fa_tensor_t *cu_seqlens_q, const fa_tensor_t *cu_seqlens_k,
                                  const fa_tensor_t *k_scale, const fa_tensor_t *v_scale,
                                  fa_tensor_t *out, fa_tensor_t *lse, float softmax_scale,
                                  int32_t causal, int32_t window, const fa_score_mod_t *score_mod,
                                  const fa_block_mask_t *block_mask, const fa_prologue_t *prologue,
                                  int32_t page_size, const fa_launch_t *launch, void *stream);

/* Message for the last non-OK status returned on this thread ("" if none). */
FA_API const char *fa_last_error(void);

/* Synchronises `stream`, then reads and clears the current device's error
 * word into *code (FA_OK when no kernel recorded a problem). */
FA_API fa_status_t fa_get_device_error(void *stream, int32_t *code);

/* Library version string. */
FA_API const char *fa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FA_GB300_H */
