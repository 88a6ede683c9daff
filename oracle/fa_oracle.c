/*
 * fa_oracle.c -- plain fp64 CPU oracle for the attention forward and backward passes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * What it computes is the plain definition of masked softmax attention with a
 * per-row log-sum-exp, one (query token, query head) row at a time:
 *
 *   s_j   = scale * <q_i, k_j>                     (all keys j of the sequence)
 *   s_j   = cap * tanh(s_j / cap)                  (soft-cap score mod)
 *   s_j   = s_j - slope * |i' - j|                 (ALiBi score mod)
 *   A_i   = { j : causal, window, block mask and j < Sk allow (i, j) }
 *   m     = max_{j in A_i} s_j
 *   l     = sum_{j in A_i} exp(s_j - m)
 *   out_i = sum_{j in A_i} exp(s_j - m) v_j / l
 *   LSE_i = m + ln(l)
 *
 * with out_i = 0 and LSE_i = -inf when A_i is empty.  Sources:
 *  - online softmax and LSE = M + log(L): RL-Kernel PR #237 "SM90 TMA +
 *    mma.sync FlashAttention", first commit (attention-domain LSE) and the
 *    summary (independent per-sequence masked-softmax + logsumexp reference);
 *  - LSE stored on fully masked tiles: FlyDSL PR #844 "Add forward LSE output",
 *    Changes list;
 *  - packed varlen cu_seqlens tensors [total_tokens, H, D]: RL-Kernel PR #237,
 *    first commit;
 *  - paged KV through block_table, FP8 e4m3 KV with per-token scales, Q/K 192
 *    and V/O 128: FlyDSL PR #1066 overview and PR description; fkl_python PR #7,
 *    fp8 KV commit (scale = max|row|/448);
 *  - e4m3 Q with a scalar descale (folded into softmax_scale): FlyDSL PR #1066
 *    description (OCP E4M3 Q/K/V with scalar descales);
 *  - int8 KV with per-token dequantisation (value = int8 * scale): fkl_python
 *    PR #7, prologue-fusion commit (int8 token dequant read) and fp8 KV commit
 *    (int8's 127 uniform levels);
 *  - bottom-right causal alignment: FlyDSL PR #1066 review (COMMENT, "What I
 *    verified": bottom-right causal mask, cross_seqlen=True);
 *  - ALiBi, SoftCap, SlidingWindow and 128x128 block masks: fkl_python PR #7,
 *    flex attention commit;
 *  - prologue: every element of Q, K and V is put through its tensor's op
 *    chain (Mul, Add, Sub or Div by a scalar, one op after the other, in the
 *    order given) as it is read, before anything else: fkl_python PR #7,
 *    prologue-fusion commit (op chains fused onto the Q/K/V reads, values at
 *    run time).  The ops are applied literally, one by one; nothing is
 *    composed here.
 *
 * Readings taken where the pages are silent:
 * i' = i + Sk - Sq; window W>0 keeps 0 <= i'-j < W when causal, |i'-j| < W
 * otherwise; ALiBi bias -slope*|i'-j| for every head; soft-cap acts on the
 * scaled score before ALiBi; block-mask index (b*Hq + h, i/128, j/128) with
 * sequence-local i, j; GQA head hk = h / (Hq/Hkv); per-token scales are one
 * fp32 per (page, slot, kv head).
 *
 * All arithmetic is double precision; bf16, e4m3 and int8 inputs are widened exactly.
 * Threads (pthreads) only split the independent rows between cores.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { KV_BF16 = 0, KV_E4M3 = 1, KV_F64 = 2, KV_I8 = 3 };
enum { MOD_NONE = 0, MOD_ALIBI = 1, MOD_SOFTCAP = 2 };

/* One prologue op chain: x -> op_{n-1}(... op_1(op_0(x, c_0), c_1) ..., c_{n-1}). */
enum { ORACLE_OP_MUL = 1, ORACLE_OP_ADD = 2, ORACLE_OP_SUB = 3, ORACLE_OP_DIV = 4 };
#define ORACLE_MAX_OPS 8
typedef struct {
    int32_t n;
    int32_t op[ORACLE_MAX_OPS];
    double c[ORACLE_MAX_OPS];
} fa_oracle_chain;

typedef struct {
    const void *q;                /* [T_q][Hq][Dk]: bf16 bits, or e4m3 bytes (q_dtype) */
    const void *k, *v;            /* packed [T_k][Hkv][D] or paged [N_pg][P_s][Hkv][D] */
    int32_t kv_dtype;             /* KV_BF16 | KV_E4M3 | KV_F64 | KV_I8 */
    const int32_t *block_table;   /* [B][bt_stride] or NULL (packed K/V) */
    int64_t bt_stride;
    const int32_t *cu_q, *cu_k;   /* [B+1] */
    int32_t num_seqs;
    const float *k_scale, *v_scale; /* per token and kv head; NULL unless e4m3 / int8 */
    int32_t hq, hkv, dk, dv, page_size;
    double softmax_scale;
    int32_t causal, window, mod_kind;
    double alibi_slope, softcap;
    const uint8_t *block_mask;    /* [B*Hq][n_qblk][n_kblk] or NULL */
    int32_t n_qblk, n_kblk, blk_q, blk_k;
    int64_t kv_lo, kv_hi;         /* restrict keys to [kv_lo, kv_hi) when kv_hi >= 0 */
    int32_t q_dtype;              /* Q_BF16 | Q_E4M3 (a per-tensor Q scale is folded into softmax_scale) | Q_F64 */
    fa_oracle_chain pro_q, pro_k, pro_v;   /* prologue op chains (n = 0: none) */
} fa_oracle_problem;

enum { Q_BF16 = 0, Q_E4M3 = 1, Q_F64 = 2 };

/* bf16 -> double: the bf16 bits are the upper half of an IEEE binary32. */
double fa_oracle_bf16_decode(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 (the "OCP E4M3" of FlyDSL PR #1066): 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN. */
/* A stored int8 byte (two's complement) as its integer value. */
double fa_oracle_i8_decode(uint8_t x) {
    return (double)(x < 128 ? (int)x : (int)x - 256);
}

double fa_oracle_e4m3_decode(uint8_t x) {
    int s = (x >> 7) & 1, e = (x >> 3) & 0xF, m = x & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) mag = ldexp((double)m / 8.0, -6);          /* subnormal */
    else mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* The op chain applied to one element, op after op. */
static double apply_chain(const fa_oracle_chain *ch, double x) {
    for (int i = 0; i < ch->n; i++) {
        const double c = ch->c[i];
        switch (ch->op[i]) {
            case ORACLE_OP_MUL: x = x * c; break;
            case ORACLE_OP_ADD: x = x + c; break;
            case ORACLE_OP_SUB: x = x - c; break;
            case ORACLE_OP_DIV: x = x / c; break;
            default: x = NAN; break;
        }
    }
    return x;
}

static int chain_is_empty(const fa_oracle_chain *ch) { return ch->n == 0; }

static int chain_valid(const fa_oracle_chain *ch) {
    if (ch->n < 0 || ch->n > ORACLE_MAX_OPS) return 0;
    for (int i = 0; i < ch->n; i++)
        if (ch->op[i] < ORACLE_OP_MUL || ch->op[i] > ORACLE_OP_DIV) return 0;
    return 1;
}

/* Row j of the sequence's keys (or values) for kv head hk, widened to double
 * (dequantised with the token's scale for byte caches) and put through the
 * tensor's prologue op chain. */
static void fetch_row(const fa_oracle_problem *p, const void *base, const float *scale, const fa_oracle_chain *ch,
                      int b, int64_t j, int hk, int d, double *dst) {
    int64_t tok;       /* flat token index in the [*, Hkv] view of the pool */
    if (p->block_table) {
        int64_t page = p->block_table[(int64_t)b * p->bt_stride + j / p->page_size];
        tok = page * p->page_size + j % p->page_size;
    } else {
        tok = (int64_t)p->cu_k[b] + j;
    }
    int64_t off = (tok * p->hkv + hk) * (int64_t)d;
    double sc = 1.0;
    if (p->kv_dtype == KV_E4M3 || p->kv_dtype == KV_I8) sc = (double)scale[tok * p->hkv + hk];
    for (int x = 0; x < d; x++) {
        double val;
        if (p->kv_dtype == KV_BF16) val = fa_oracle_bf16_decode(((const uint16_t *)base)[off + x]);
        else if (p->kv_dtype == KV_E4M3) val = fa_oracle_e4m3_decode(((const uint8_t *)base)[off + x]);
        else if (p->kv_dtype == KV_I8) val = fa_oracle_i8_decode(((const uint8_t *)base)[off + x]);
        else val = ((const double *)base)[off + x];
        dst[x] = apply_chain(ch, val * sc);
    }
}

/* Query row (token t, head h) widened to double and put through q's
 * prologue op chain. */
static void fetch_q(const fa_oracle_problem *p, int64_t t, int h, double *qrow) {
    for (int x = 0; x < p->dk; x++) {
        const int64_t at = (t * p->hq + h) * (int64_t)p->dk + x;
        double val;
        if (p->q_dtype == Q_E4M3) val = fa_oracle_e4m3_decode(((const uint8_t *)p->q)[at]);
        else if (p->q_dtype == Q_F64) val = ((const double *)p->q)[at];
        else val = fa_oracle_bf16_decode(((const uint16_t *)p->q)[at]);
        qrow[x] = apply_chain(&p->pro_q, val);
    }
}

/* Is key j visible from query row i of sequence b, head h? */
static int allowed(const fa_oracle_problem *p, int b, int h, int64_t i, int64_t j,
                   int64_t sq, int64_t sk) {
    int64_t ip = i + sk - sq;                      /* bottom-right aligned query position */
    if (j < 0 || j >= sk) return 0;
    if (p->kv_hi >= 0 && (j < p->kv_lo || j >= p->kv_hi)) return 0;
    if (p->causal && j > ip) return 0;
    if (p->window > 0) {
        if (p->causal) {
            if (ip - j >= p->window) return 0;
        } else {
            int64_t dist = ip > j ? ip - j : j - ip;
            if (dist >= p->window) return 0;
        }
    }
    if (p->block_mask) {
        int64_t qb = i / p->blk_q, kb = j / p->blk_k;
        if (qb >= p->n_qblk || kb >= p->n_kblk) return 0;
        int64_t idx = (((int64_t)b * p->hq + h) * p->n_qblk + qb) * p->n_kblk + kb;
        if (!p->block_mask[idx]) return 0;
    }
    return 1;
}

/* One row: query token t (global), head h.  Writes out[dv] and *lse. */
static void one_row(const fa_oracle_problem *p, int64_t t, int h, double *out, double *lse,
                    double *qrow, double *krow, double *vrow, double *s, unsigned char *ok) {
    int b = 0;
    while (b < p->num_seqs && !(t >= p->cu_q[b] && t < p->cu_q[b + 1])) b++;
    int64_t sq = p->cu_q[b + 1] - p->cu_q[b];
    int64_t sk = p->cu_k[b + 1] - p->cu_k[b];
    int64_t i = t - p->cu_q[b];
    int64_t ip = i + sk - sq;
    int hk = h / (p->hq / p->hkv);

    fetch_q(p, t, h, qrow);

    int any = 0;
    double m = -INFINITY;
    for (int64_t j = 0; j < sk; j++) {
        ok[j] = (unsigned char)allowed(p, b, h, i, j, sq, sk);
        if (!ok[j]) continue;
        fetch_row(p, p->k, p->k_scale, &p->pro_k, b, j, hk, p->dk, krow);
        double dot = 0.0;
        for (int x = 0; x < p->dk; x++) dot += qrow[x] * krow[x];
        double sj = p->softmax_scale * dot;
        if (p->mod_kind == MOD_SOFTCAP) sj = p->softcap * tanh(sj / p->softcap);
        if (p->mod_kind == MOD_ALIBI) sj -= p->alibi_slope * (double)(ip > j ? ip - j : j - ip);
        s[j] = sj;
        if (sj > m) m = sj;
        any = 1;
    }
    for (int x = 0; x < p->dv; x++) out[x] = 0.0;
    if (!any) {
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < sk; j++) {
        if (!ok[j]) continue;
        double w = exp(s[j] - m);
        l += w;
        fetch_row(p, p->v, p->v_scale, &p->pro_v, b, j, hk, p->dv, vrow);
        for (int x = 0; x < p->dv; x++) out[x] += w * vrow[x];
    }
    for (int x = 0; x < p->dv; x++) out[x] /= l;
    *lse = m + log(l);
}

typedef struct {
    const fa_oracle_problem *p;
    const int64_t *units;     /* pairs (t, h), or NULL for all rows */
    int64_t n_units;
    double *out, *lse;
    int tid, nthreads;
    int64_t max_sk;
} worker_arg;

static void *worker(void *argp) {
    worker_arg *a = (worker_arg *)argp;
    const fa_oracle_problem *p = a->p;
    int64_t cap_k = a->max_sk > 0 ? a->max_sk : 1;
    double *qrow = (double *)malloc(sizeof(double) * p->dk);
    double *krow = (double *)malloc(sizeof(double) * p->dk);
    double *vrow = (double *)malloc(sizeof(double) * p->dv);
    double *s = (double *)malloc(sizeof(double) * cap_k);
    unsigned char *ok = (unsigned char *)malloc(cap_k);
    for (int64_t u = a->tid; u < a->n_units; u += a->nthreads) {
        int64_t t, h;
        if (a->units) { t = a->units[2 * u]; h = a->units[2 * u + 1]; }
        else { t = u / p->hq; h = u % p->hq; }
        one_row(p, t, (int)h, a->out + u * p->dv, a->lse + u, qrow, krow, vrow, s, ok);
    }
    free(qrow); free(krow); free(vrow); free(s); free(ok);
    return NULL;
}

/*
 * Compute rows of the forward pass.
 *   units   : NULL for every (t, h) in t-major order, else n_units pairs (t, h)
 *   out     : [n_units][Dv] doubles;  lse: [n_units] doubles
 * Returns 0, or -1 on a malformed problem.
 */
int fa_oracle_fwd(const fa_oracle_problem *p, const int64_t *units, int64_t n_units,
                  double *out, double *lse, int nthreads) {
    if (!p || p->hq <= 0 || p->hkv <= 0 || p->hq % p->hkv || p->num_seqs < 0) return -1;
    if (p->block_table && p->page_size <= 0) return -1;
    if (!chain_valid(&p->pro_q) || !chain_valid(&p->pro_k) || !chain_valid(&p->pro_v)) return -1;
    if (!units) n_units = (int64_t)p->cu_q[p->num_seqs] * p->hq;
    int64_t max_sk = 0;
    for (int b = 0; b < p->num_seqs; b++) {
        int64_t sk = p->cu_k[b + 1] - p->cu_k[b];
        if (sk > max_sk) max_sk = sk;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    pthread_t th[1024];
    worker_arg args[1024];
    for (int i = 0; i < nthreads; i++) {
        args[i] = (worker_arg){p, units, n_units, out, lse, i, nthreads, max_sk};
        if (nthreads > 1) pthread_create(&th[i], NULL, worker, &args[i]);
    }
    if (nthreads == 1) worker(&args[0]);
    else for (int i = 0; i < nthreads; i++) pthread_join(th[i], NULL);
    return 0;
}

/*
 * Merge of partial results over disjoint key sets (split-KV combine).
 * Softmax over a union of disjoint key sets S_1..S_n: with L_s the LSE and
 * O_s the normalised output over S_s,
 *   LSE = ln sum_s exp(L_s),   out = sum_s exp(L_s - LSE) * O_s.
 * Sets with L_s = -inf contribute nothing; all -inf gives out 0, LSE -inf.
 * The pages' split-K combine finalises m_max*ln2 + ln(den) from per-split
 * (m, l) (FlyDSL PR #844, Changes list); this is the same merge in the
 * natural-log domain.
 *   o_part: [n_split][n][Dv], lse_part: [n_split][n]
 */
void fa_oracle_combine(const double *o_part, const double *lse_part, int n_split, int64_t n,
                       int dv, double *out, double *lse) {
    for (int64_t r = 0; r < n; r++) {
        double mx = -INFINITY;
        for (int s = 0; s < n_split; s++) {
            double v = lse_part[(int64_t)s * n + r];
            if (v > mx) mx = v;
        }
        for (int x = 0; x < dv; x++) out[r * dv + x] = 0.0;
        if (mx == -INFINITY) { lse[r] = -INFINITY; continue; }
        double den = 0.0;
        for (int s = 0; s < n_split; s++) den += exp(lse_part[(int64_t)s * n + r] - mx);
        double L = mx + log(den);
        lse[r] = L;
        for (int s = 0; s < n_split; s++) {
            double w = exp(lse_part[(int64_t)s * n + r] - L);
            if (w == 0.0) continue;
            for (int x = 0; x < dv; x++) out[r * dv + x] += w * o_part[((int64_t)s * n + r) * dv + x];
        }
    }
}

/*
 * Backward pass: the gradients of L = sum_{i,x} dO[i][x] * out[i][x] with
 * respect to q, k and v, by the chain rule through the definition above
 * (RL-Kernel PR #237, backward commit: recompute the probabilities from the
 * forward's saved statistics, then dQ, dK, dV).  For one row i with allowed
 * set A_i and probabilities P_j = exp(s_j - LSE_i):
 *
 *   dV_j  += P_j * dO_i                        (out_i = sum_j P_j v_j)
 *   dP_j   = <dO_i, v_j>
 *   dS_j   = P_j * (dP_j - sum_{l in A_i} P_l dP_l)    (softmax Jacobian)
 *   dU_j   = dS_j * d s_j / d u_j              (u_j = scale <q_i, k_j>;
 *            1 - tanh^2(u_j / cap) under the soft-cap, 1 otherwise; ALiBi
 *            adds a constant, so its derivative is 1)
 *   dQ_i  += scale * dU_j * k_j,   dK_j += scale * dU_j * q_i
 *
 * Rows with an empty A_i contribute nothing.  GQA: the q heads of a kv head's
 * group all add into its dK, dV.  Packed K/V only (block_table NULL), K/V
 * bf16 or f64.  Work is split by (sequence, kv head), so each thread owns the
 * rows it accumulates.
 *   dout: [T_q][Hq][Dv] doubles
 *   dq: [T_q][Hq][Dk], dk: [T_k][Hkv][Dk], dv: [T_k][Hkv][Dv] doubles (overwritten)
 */
typedef struct {
    const fa_oracle_problem *p;
    const double *dout;
    double *dq, *dk, *dv;
    int tid, nthreads;
    int64_t max_sk;
} bwd_arg;

static void *bwd_worker(void *argp) {
    bwd_arg *a = (bwd_arg *)argp;
    const fa_oracle_problem *p = a->p;
    const int g = p->hq / p->hkv;
    int64_t cap_k = a->max_sk > 0 ? a->max_sk : 1;
    double *qrow = (double *)malloc(sizeof(double) * p->dk);
    double *krow = (double *)malloc(sizeof(double) * p->dk);
    double *vrow = (double *)malloc(sizeof(double) * p->dv);
    double *s = (double *)malloc(sizeof(double) * cap_k);
    double *u = (double *)malloc(sizeof(double) * cap_k);
    double *dp = (double *)malloc(sizeof(double) * cap_k);
    unsigned char *ok = (unsigned char *)malloc(cap_k);
    for (int64_t unit = a->tid; unit < (int64_t)p->num_seqs * p->hkv; unit += a->nthreads) {
        const int b = (int)(unit / p->hkv), hk = (int)(unit % p->hkv);
        const int64_t sq = p->cu_q[b + 1] - p->cu_q[b], sk = p->cu_k[b + 1] - p->cu_k[b];
        for (int h = hk * g; h < (hk + 1) * g; h++) {
            for (int64_t i = 0; i < sq; i++) {
                const int64_t t = p->cu_q[b] + i, ip = i + sk - sq;
                fetch_q(p, t, h, qrow);
                const double *dorow = a->dout + (t * p->hq + h) * (int64_t)p->dv;
                double m = -INFINITY;
                int any = 0;
                for (int64_t j = 0; j < sk; j++) {
                    ok[j] = (unsigned char)allowed(p, b, h, i, j, sq, sk);
                    if (!ok[j]) continue;
                    fetch_row(p, p->k, p->k_scale, &p->pro_k, b, j, hk, p->dk, krow);
                    double dot = 0.0;
                    for (int x = 0; x < p->dk; x++) dot += qrow[x] * krow[x];
                    double sj = p->softmax_scale * dot;
                    u[j] = sj;
                    if (p->mod_kind == MOD_SOFTCAP) sj = p->softcap * tanh(sj / p->softcap);
                    if (p->mod_kind == MOD_ALIBI) sj -= p->alibi_slope * (double)(ip > j ? ip - j : j - ip);
                    s[j] = sj;
                    if (sj > m) m = sj;
                    any = 1;
                }
                if (!any) continue;
                double l = 0.0;
                for (int64_t j = 0; j < sk; j++)
                    if (ok[j]) l += exp(s[j] - m);
                const double lse = m + log(l);
                double dsum = 0.0;
                for (int64_t j = 0; j < sk; j++) {
                    if (!ok[j]) continue;
                    fetch_row(p, p->v, p->v_scale, &p->pro_v, b, j, hk, p->dv, vrow);
                    double d = 0.0;
                    for (int x = 0; x < p->dv; x++) d += dorow[x] * vrow[x];
                    dp[j] = d;
                    const double pj = exp(s[j] - lse);
                    dsum += pj * d;
                    double *dvrow = a->dv + ((p->cu_k[b] + j) * p->hkv + hk) * (int64_t)p->dv;
                    for (int x = 0; x < p->dv; x++) dvrow[x] += pj * dorow[x];
                }
                double *dqrow = a->dq + (t * p->hq + h) * (int64_t)p->dk;
                for (int64_t j = 0; j < sk; j++) {
                    if (!ok[j]) continue;
                    const double pj = exp(s[j] - lse);
                    double du = pj * (dp[j] - dsum);
                    if (p->mod_kind == MOD_SOFTCAP) {
                        const double th = tanh(u[j] / p->softcap);
                        du *= 1.0 - th * th;
                    }
                    fetch_row(p, p->k, p->k_scale, &p->pro_k, b, j, hk, p->dk, krow);
                    double *dkrow = a->dk + ((p->cu_k[b] + j) * p->hkv + hk) * (int64_t)p->dk;
                    for (int x = 0; x < p->dk; x++) {
                        dqrow[x] += p->softmax_scale * du * krow[x];
                        dkrow[x] += p->softmax_scale * du * qrow[x];
                    }
                }
            }
        }
    }
    free(qrow); free(krow); free(vrow); free(s); free(u); free(dp); free(ok);
    return NULL;
}

int fa_oracle_bwd(const fa_oracle_problem *p, const double *dout, double *dq, double *dk, double *dv,
                  int nthreads) {
    if (!p || p->hq <= 0 || p->hkv <= 0 || p->hq % p->hkv || p->num_seqs < 0) return -1;
    if (p->block_table || (p->kv_dtype != KV_BF16 && p->kv_dtype != KV_F64)) return -1;
    /* gradients with respect to the stored tensors: no prologue */
    if (!chain_is_empty(&p->pro_q) || !chain_is_empty(&p->pro_k) || !chain_is_empty(&p->pro_v)) return -1;
    const int64_t tq = p->cu_q[p->num_seqs], tk = p->cu_k[p->num_seqs];
    memset(dq, 0, sizeof(double) * tq * p->hq * p->dk);
    memset(dk, 0, sizeof(double) * tk * p->hkv * p->dk);
    memset(dv, 0, sizeof(double) * tk * p->hkv * p->dv);
    int64_t max_sk = 0;
    for (int b = 0; b < p->num_seqs; b++) {
        int64_t sk = p->cu_k[b + 1] - p->cu_k[b];
        if (sk > max_sk) max_sk = sk;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    pthread_t th[1024];
    bwd_arg args[1024];
    for (int i = 0; i < nthreads; i++) {
        args[i] = (bwd_arg){p, dout, dq, dk, dv, i, nthreads, max_sk};
        if (nthreads > 1) pthread_create(&th[i], NULL, bwd_worker, &args[i]);
    }
    if (nthreads == 1) bwd_worker(&args[0]);
    else for (int i = 0; i < nthreads; i++) pthread_join(th[i], NULL);
    return 0;
}
