// fa_decode.cuh -- split-KV decode kernel and the LSE combine kernel.
//
// Decode (few query rows per kv head, long keys) is bound by streaming the KV
// cache from HBM: about 4 flops per byte for bf16 K/V with a GQA group of 4.
// The kernel therefore spends its effort on the memory side -- TMA page
// gathers into a 3-stage shared-memory ring, many CTAs in flight -- and uses
// warp-level mma.sync only as a dense FMA engine for the tiny contractions.
//
// Split-KV: CTA (split s, kv head hk, sequence b) reduces the keys
// [s*split_keys, (s+1)*split_keys) of that sequence for the rows that share kv
// head hk: (query token tq, head hk*g + x) with row index tq*g + x < 16.  It
// writes the normalised partial output O_s (fp32) and its LSE_s; the combine
// kernel merges the splits:  LSE = ln sum_s exp(LSE_s),
// out = sum_s exp(LSE_s - LSE) * O_s  (FlyDSL PR #844, Changes: split-K combine
// finalising m_max*ln2 + ln(den); FlyDSL PR #1066 lists split-K/combine as
// the long-KV decode form).  With a single split the kernel writes the final
// bf16 output and LSE itself.
//
// Byte caches (KV = 1: e4m3, KV = 2: int8; per-token scales, fkl_python PR #7:
// fp8 KV decode from the raw quantised bytes, half the traffic of bf16).  TMA
// lands the bytes, the producer lanes copy the stage's per-token k/v scales
// with cp.async beside them, and each consumer warp turns its own 16 keys into
// f16 exactly (e4m3 and int8 values are f16 numbers): at D = 128 in registers,
// straight from the 128-byte-swizzled stage into its MMA fragments (DIRECT
// below), at D = 64 through a private swizzled f16 buffer.  Q is brought to
// f16 with a per-row power-of-two factor.  The scales
// stay in fp32: k_scale multiplies each score column, v_scale each P column
// before the f16 P V product, so the cached values are never rounded.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_gather.cuh"
#include "sm103_ptx.cuh"

namespace fa {

constexpr int kDecRows = 16;          // MMA M: query rows per CTA
constexpr int kDecStageKeys = 64;     // keys per pipeline stage
constexpr int kDecStages = 3;
constexpr int kDecWarps = 4;          // consumer warps (16 keys each per stage)
constexpr int kDecThreads = (kDecWarps + 1) * 32;

struct DecodeParams {
  const __nv_bfloat16 *q;
  int64_t q_stride_t, q_stride_h;     // elements
  const int32_t *cu_q;
  const int32_t *cu_k;
  const int32_t *block_table;
  int64_t bt_stride;
  int32_t page_size, page_shift, rows_per_box, boxes_per_stage;
  int32_t hq, hkv, group;
  int32_t split_keys, num_splits;
  int32_t causal, window;
  int64_t total_q;
  float scale_log2;
  // outputs: partials when o_part != null, else final out/lse
  float *o_part;                      // [S, T_q, Hq, Dv]
  float *lse_part;                    // [S, Hq, T_q]
  __nv_bfloat16 *out;
  int64_t out_stride_t, out_stride_h;
  float *lse;                         // [Hq, T_q] or null
  int *err;                           // device error word
  const float *k_scale, *v_scale;     // byte caches: per (token, kv head), in the cache's token order
  int32_t gather;                     // pages of < 16 keys: K/V rows by cp.async (fa_gather.cuh)
  KvGather gk, gv;
  // folded prologue: partial or final out = pro_vmul * o + pro_vadd on rows
  // that see keys; the row term pro_lse_k * sum_d q[d] + pro_lse_c is added
  // to the LSE, or under the soft-cap enters the capped score as
  // pro_row_k * sum_d q[d] + pro_row_c (2u*log2(e) units); col_bias holds the
  // per-key term of a Q add, [B][Hkv][cb_ld] in the score's units, or null
  float pro_vmul, pro_vadd, pro_lse_k, pro_lse_c, pro_row_k, pro_row_c;
  const float *col_bias;
  int64_t cb_ld;
  // byte caches in the vectorized 5-D layouts (paged, pages of >= 16 keys):
  // K [N_pg, Hkv, D/16, P_s, 16], V [N_pg, Hkv, P_s/16, D, 16]
  int32_t vec5;
  // score mods (0 none, 1 ALiBi, 2 soft-cap) and 128 x 128 block masks, as
  // in the prefill kernels
  int32_t mod;
  float alibi_log2;                   // slope * log2(e)
  float softcap_arg, softcap_log2;    // softmax_scale / cap, cap * log2(e)
  const uint8_t *block_mask;          // [B*Hq, n_qblk, n_kblk] or null
  int32_t n_qblk, n_kblk;
};

// DIRECT (byte caches at D = 128, token-major pages): the stage's K and V
// bytes land 128-byte swizzled and go from shared memory straight into the
// MMA fragments (see the consumer), with no f16 copy in between.  OT (with
// DIRECT, at most 8 query rows): P V is computed transposed, half the MMAs
// and accumulators, which lets three CTAs share an SM.
template <int D, int KV = 0, bool DIRECT = false, bool OT = false>
struct DecodeCfg {
  static_assert(!DIRECT || (KV && D == 128), "fragment-direct bytes: byte caches at D = 128");
  static_assert(!OT || DIRECT, "the transposed P V runs on the fragment-direct path");
  static constexpr int kElt = KV ? 1 : 2;                  // cache bytes per element
  static constexpr int kKBytes = kDecStageKeys * D * kElt;   // per stage
  static constexpr int kVBytes = kDecStageKeys * D * kElt;
  static constexpr int kScaleBytes = KV ? 2 * kDecStageKeys * 4 : 0;   // k then v scales of the stage
  // DIRECT: stages start on 1024-byte boundaries (the swizzle pattern's period)
  static constexpr int kStageBytes = DIRECT ? (kKBytes + kVBytes + kScaleBytes + 1023) / 1024 * 1024
                                            : kKBytes + kVBytes + kScaleBytes;
  // byte caches: a deeper ring of half-size stages keeps as many bytes in
  // flight as the bf16 ring does (DIRECT: one more, in the conversion
  // buffers' room)
  static constexpr int NST = KV ? (DIRECT ? (OT ? 4 : 6) : 5) : kDecStages;
  static constexpr int kOffStages = 0;
  // byte caches: per consumer warp, its 16 keys of K, then of V, as swizzled f16
  static constexpr int kConvWarpBytes = (KV && !DIRECT) ? 16 * D * 2 : 0;
  static constexpr int kOffConv = ((NST * kStageBytes + 1023) / 1024) * 1024;
  static constexpr int kOffQ = kOffConv + kDecWarps * kConvWarpBytes;   // 16 x D bf16 (f16 for byte caches)
  static constexpr int kOffQInv = kOffQ + kDecRows * D * 2;            // byte caches: 2^-e per Q row
  static constexpr int kOffBar = kOffQInv + kDecRows * 4;
  static constexpr int kOffMisc = kOffBar + 2 * NST * 8;
  static constexpr int kSmemBytes = kOffMisc + 64 + 1024;
  static_assert(NST * kStageBytes >= kDecWarps * kDecRows * D * 4 + kDecWarps * kDecRows * 8,
                "the stage ring doubles as the cross-warp reduction buffer");
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <int KV>
__device__ __forceinline__ void dec_mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (KV) mma_f16_16816(c, a, b0, b1);
  else mma_bf16_16816(c, a, b0, b1);
}

// 4-byte global -> shared copy; `bytes` 0 writes zeros and reads nothing.
__device__ __forceinline__ void dec_cp_async_4(uint32_t dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
// One arrival on `bar` once this thread's earlier cp.async copies have landed.
__device__ __forceinline__ void dec_cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
// Four cache bytes -> four f16 values (two packed pairs), exactly: e4m3 by the
// hardware conversion of each 16-bit half; int8 byte x as the f16 whose bits
// are 0x6400 | (x + 128), i.e. 1024 + (x + 128) (f16 spacing is 1 on
// [1024, 2048)), minus 1152 in f16 (exact; checked for all 256 bytes).
template <int KV>
__device__ __forceinline__ void dec_bytes4_to_f16(uint32_t w, uint32_t &o0, uint32_t &o1) {
  if constexpr (KV == 1) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(o0), "=r"(o1)
        : "r"(w));
  } else {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t lo = __byte_perm(u, 0x64646464u, 0x4140), hi = __byte_perm(u, 0x64646464u, 0x4342);
    asm("sub.f16x2 %0, %1, %2;" : "=r"(o0) : "r"(lo), "r"(0x64806480u));   // 0x6480 = 1152 in f16
    asm("sub.f16x2 %0, %1, %2;" : "=r"(o1) : "r"(hi), "r"(0x64806480u));
  }
}

// Byte offset of (row, 16-byte chunk) in a 128-byte-swizzled [rows x 64] bf16 block.
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// V5: byte caches in the vectorized 5-D pages (a kernel of its own, so that
// the token-major kernels keep their register allocation).
template <int D, int KV, bool V5>
constexpr bool dec_direct() { return KV != 0 && D == 128 && !V5; }

// R8: every CTA has at most 8 query rows (max_seqlen_q * Hq/Hkv <= 8).
template <int D, int KV = 0, bool V5 = false, bool R8 = false>
__global__ void __launch_bounds__(kDecThreads, (dec_direct<D, KV, V5>() && R8) ? 3 : 2)
    fa_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const DecodeParams p) {
  constexpr bool DIRECT = dec_direct<D, KV, V5>();
  constexpr bool OT = R8 && DIRECT;
  // KDIR (byte caches at D = 128, token-major or 5-D pages): the QK product
  // reads the raw K bytes into its fragments, with the permuted contraction
  // order below, so that both page layouts sum the scores alike
  constexpr bool KDIR = KV != 0 && D == 128;
  // QT (with KDIR, at most 8 query rows): QK computed transposed as well,
  // S^T = K Q^T with N = 8 rows (half the QK MMAs); the thread then owns rows
  // 2t and 2t+1, and P reaches the P V operand layout by shuffles
  static_assert(!R8 || KDIR, "the 8-row forms read the key bytes directly");
  constexpr bool QT = R8;
  using Cfg = DecodeCfg<D, KV, DIRECT, OT>;
  constexpr int NCB = D / 64;          // 64-dim column blocks
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int qa = __ldg(p.cu_q + b), sq = __ldg(p.cu_q + b + 1) - qa;
  const int sk = __ldg(p.cu_k + b + 1) - __ldg(p.cu_k + b);
  const int rows = sq * p.group;       // <= 16, checked on the host
  if (rows == 0) return;
  const int key_lo = split * p.split_keys;
  const int key_hi = min(sk, key_lo + p.split_keys);
  // Largest key any row of this CTA may see (causal: the last row's i').
  int vis_hi = key_hi;
  if (p.causal) vis_hi = min(vis_hi, sk);   // last row i' = sk - 1
  int vis_lo = key_lo;
  if (p.window > 0) vis_lo = max(vis_lo, (0 + sk - sq) - p.window + 1);
  const int n_stages = vis_hi > vis_lo ? (vis_hi - key_lo + kDecStageKeys - 1) / kDecStageKeys : 0;
  const int first_stage = vis_hi > vis_lo ? max(0, (vis_lo - key_lo) / kDecStageKeys) : 0;

  if (n_stages <= first_stage) {
    // Empty key range for every row: LSE -inf (the combine skips it).
    for (int r = threadIdx.x; r < rows; r += blockDim.x) {
      const int tq = r / p.group, h = hk * p.group + r % p.group;
      const int64_t t = (int64_t)qa + tq;
      if (p.o_part) {
        p.lse_part[((int64_t)split * p.hq + h) * p.total_q + t] = -INFINITY;
      } else {
        __nv_bfloat16 *o = p.out + t * p.out_stride_t + (int64_t)h * p.out_stride_h;
        for (int d = 0; d < D; ++d) o[d] = __float2bfloat16(0.f);
        if (p.lse) p.lse[(int64_t)h * p.total_q + t] = -INFINITY;
      }
    }
    return;
  }

  uint8_t *stages = smem + Cfg::kOffStages;
  __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(smem + Cfg::kOffQ);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
  constexpr int NST = Cfg::NST;
  uint64_t *empty = full + NST;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc);

  float *sQinv = reinterpret_cast<float *>(smem + Cfg::kOffQInv);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      // byte caches: the producer's arrival plus one cp.async arrival per lane
      // (scales); gathered rows (pages of < 16 keys): one arrival per lane
      // in place of the producer's
      const uint32_t n_fill = p.gather ? 32u : 1u;
      mbar_init(smem_u32(full + s), KV ? n_fill + 32 : n_fill);
      mbar_init(smem_u32(empty + s), kDecWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if constexpr (KV == 0) {
    // Q rows -> shared memory (zero rows past `rows`), plain layout [16][D].
    for (int e = threadIdx.x; e < kDecRows * D / 8; e += blockDim.x) {
      const int r = e / (D / 8), c8 = e % (D / 8);
      uint4 val = make_uint4(0, 0, 0, 0);
      if (r < rows) {
        const int tq = r / p.group, h = hk * p.group + r % p.group;
        const __nv_bfloat16 *src = p.q + (int64_t)(qa + tq) * p.q_stride_t + (int64_t)h * p.q_stride_h + c8 * 8;
        val = *reinterpret_cast<const uint4 *>(src);
      }
      *reinterpret_cast<uint4 *>(sQ + r * D + c8 * 8) = val;
    }
  } else {
    // Q rows as f16 with a per-row factor 2^e, max|q| * 2^e in [2^14, 2^15):
    // every bf16 element within 2^-24 of the row maximum is exact in f16.
    // One warp per row, D/32 elements per lane; 2^-e is kept for the scores.
    for (int r = warp; r < kDecRows; r += kDecWarps + 1) {
      constexpr int kPer = D / 32;
      float v[kPer];
      float mx = 0.f;
#pragma unroll
      for (int e = 0; e < kPer; ++e) v[e] = 0.f;
      if (r < rows) {
        const int tq = r / p.group, h = hk * p.group + r % p.group;
        const __nv_bfloat16 *src = p.q + (int64_t)(qa + tq) * p.q_stride_t + (int64_t)h * p.q_stride_h + lane * kPer;
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          v[e] = __bfloat162float(src[e]);
          mx = fmaxf(mx, fabsf(v[e]));
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      int ex = 0;
      if (mx > 0.f) ex = 14 - ilogbf(mx);        // mx * 2^ex in [2^14, 2^15)
      const float f = ldexpf(1.f, ex);
      __half *dst = reinterpret_cast<__half *>(sQ) + r * D + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; ++e) dst[e] = __float2half_rn(v[e] * f);
      if (lane == 0) sQinv[r] = ldexpf(1.f, -ex);
    }
  }
  __syncthreads();

  if (warp == kDecWarps) {
    // ------------------------------------------------------- producer --
    // Lane 0 waits for the stage and arms its barrier; the stage's boxes (up
    // to 64 with page size 1, one page-table read each) are issued by all
    // lanes in parallel.
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    const int32_t *bt = p.block_table ? p.block_table + (int64_t)b * p.bt_stride : nullptr;
    const int krow0 = __ldg(p.cu_k + b);
    // Page ids are read one stage ahead, so that the block-table latency
    // overlaps the wait for a free stage.  Lane bx < boxes_per_stage (<= 4,
    // pages of 16 keys or more) owns box bx; with byte caches lane l also
    // copies the scales of keys l and l + 32.
    auto box_page = [&](int st) -> int {
      if (!bt || lane >= p.boxes_per_stage || st >= n_stages) return -1;
      const int key0 = key_lo + st * kDecStageKeys + lane * p.rows_per_box;
      return key0 < sk ? __ldg(bt + (key0 >> p.page_shift)) : -1;
    };
    auto scale_page = [&](int st, int u) -> int {
      if (!KV || !bt || st >= n_stages) return 0;
      const int key = key_lo + st * kDecStageKeys + lane + 32 * u;
      return key < sk ? __ldg(bt + (key >> p.page_shift)) : 0;
    };
    bool ok = true;
    if (p.gather && bt) {
      // Pages of < 16 keys: every key row by its own page-table read and
      // 16-byte copies (fa_gather.cuh): swizzled bf16 blocks or plain byte
      // rows, the layouts the boxes fill.  pg[u] is the page of key
      // lane + 32u of a stage; byte caches take their scales through it too.
      auto pages_of = [&](int st, int (&pg)[2]) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int key = key_lo + st * kDecStageKeys + lane + 32 * u;
          pg[u] = (st < n_stages && key < sk) ? __ldg(bt + (key >> p.page_shift)) : -1;
        }
      };
      // one stage in flight: the stage the producer waits for frees once
      // the consumers are done with stage it - NST (NST >= 3), older than
      // the newest (two in flight would also be safe, but measured slower)
      GatherPipe<1> gp;
      int pg[2], pgn[2];
      pages_of(first_stage, pg);
      for (int st = first_stage; st < n_stages; ++st) {
        const int it = st - first_stage;
        const int slot_i = it % NST;
        pages_of(st + 1, pgn);
        if (lane == 0 && it >= NST) ok = mbar_wait(smem_u32(empty + slot_i), ((it / NST) - 1) & 1, abort_flag, p.err);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        uint8_t *kd = stages + slot_i * Cfg::kStageBytes;
        uint8_t *vd = kd + Cfg::kKBytes;
        const int key0 = key_lo + st * kDecStageKeys;
        if constexpr (KV) {
          const uint32_t sdst = smem_u32(vd + Cfg::kVBytes);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int kk = lane + 32 * u;
            const bool live = pg[u] >= 0;
            const int64_t at = ((int64_t)pg[u] * p.page_size + ((key0 + kk) & (p.page_size - 1))) * p.hkv + hk;
            dec_cp_async_4(sdst + 4 * kk, live ? p.k_scale + at : p.k_scale, live ? 4u : 0u);
            dec_cp_async_4(sdst + 4 * (kDecStageKeys + kk), live ? p.v_scale + at : p.v_scale, live ? 4u : 0u);
          }
          dec_cp_async_arrive_noinc(smem_u32(full + slot_i));
          if constexpr (DIRECT) {
            gather_block<kDecStageKeys, 128, kGatherSw128, 4>(kd, p.gk, hk, key0, p.page_size - 1, 0, pg, lane);
            gather_block<kDecStageKeys, 128, kGatherSw128, 4>(vd, p.gv, hk, key0, p.page_size - 1, 0, pg, lane);
          } else {
            gather_block<kDecStageKeys, D, kGatherPlain, 4>(kd, p.gk, hk, key0, p.page_size - 1, 0, pg, lane);
            gather_block<kDecStageKeys, D, kGatherPlain, 4>(vd, p.gv, hk, key0, p.page_size - 1, 0, pg, lane);
          }
        } else {
#pragma unroll
          for (int cb = 0; cb < NCB; ++cb) {
            const uint32_t off = cb * kDecStageKeys * 128;
            gather_block<kDecStageKeys, 128, kGatherSw128, 4>(kd + off, p.gk, hk, key0, p.page_size - 1, cb * 128, pg, lane);
            gather_block<kDecStageKeys, 128, kGatherSw128, 4>(vd + off, p.gv, hk, key0, p.page_size - 1, cb * 128, pg, lane);
          }
        }
        gp.commit(smem_u32(full + slot_i));
#pragma unroll
        for (int u = 0; u < 2; ++u) pg[u] = pgn[u];
      }
      gp.drain();
    }
    int pg_next = ok && !(p.gather && bt) ? box_page(first_stage) : -1;
    int sp_next[2] = {scale_page(first_stage, 0), scale_page(first_stage, 1)};
    for (int st = first_stage; ok && !(p.gather && bt) && st < n_stages; ++st) {
      const int it = st - first_stage;
      const int slot_i = it % NST;
      const int pg = pg_next, sp[2] = {sp_next[0], sp_next[1]};
      pg_next = box_page(st + 1);
      sp_next[0] = scale_page(st + 1, 0);
      sp_next[1] = scale_page(st + 1, 1);
      if (lane == 0) {
        if (it >= NST) ok = mbar_wait(smem_u32(empty + slot_i), ((it / NST) - 1) & 1, abort_flag, p.err);
        if (ok) mbar_expect_tx(smem_u32(full + slot_i), Cfg::kKBytes + Cfg::kVBytes);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      uint8_t *kd = stages + slot_i * Cfg::kStageBytes;
      uint8_t *vd = kd + Cfg::kKBytes;
      if constexpr (KV) {
        // the stage's k and v scales (keys lane and lane + 32) beside the bytes
        const uint32_t sdst = smem_u32(vd + Cfg::kVBytes);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int kk = lane + 32 * u;
          const int key = key_lo + st * kDecStageKeys + kk;
          const bool live = key < sk;
          const int64_t tok = bt ? (int64_t)sp[u] * p.page_size + (key & (p.page_size - 1)) : (int64_t)krow0 + key;
          const int64_t at = tok * p.hkv + hk;
          dec_cp_async_4(sdst + 4 * kk, live ? p.k_scale + at : p.k_scale, live ? 4u : 0u);
          dec_cp_async_4(sdst + 4 * (kDecStageKeys + kk), live ? p.v_scale + at : p.v_scale, live ? 4u : 0u);
        }
        dec_cp_async_arrive_noinc(smem_u32(full + slot_i));
      }
      if (lane < p.boxes_per_stage) {
        const int bx = lane;
        const int key0 = key_lo + st * kDecStageKeys + bx * p.rows_per_box;
        const int slot = key0 & (p.page_size - 1);
        if constexpr (KV) {
          // one box per page piece: rows_per_box keys x D bytes, unswizzled
          // (DIRECT: 128-byte swizzled; 5-D: K as [D/16][rows][16], V as
          // [rows/16][D][16 tokens])
          const uint32_t off = bx * p.rows_per_box * D;
          if (V5) {
            tma_load_5d(smem_u32(kd + off), &tm_k, smem_u32(full + slot_i), 0, slot, 0, hk, pg);
            tma_load_5d(smem_u32(vd + off), &tm_v, smem_u32(full + slot_i), 0, 0, slot >> 4, hk, pg);
          } else if (bt) {
            tma_load_4d(smem_u32(kd + off), &tm_k, smem_u32(full + slot_i), 0, hk, slot, pg);
            tma_load_4d(smem_u32(vd + off), &tm_v, smem_u32(full + slot_i), 0, hk, slot, pg);
          } else {
            tma_load_3d(smem_u32(kd + off), &tm_k, smem_u32(full + slot_i), 0, hk, krow0 + key0);
            tma_load_3d(smem_u32(vd + off), &tm_v, smem_u32(full + slot_i), 0, hk, krow0 + key0);
          }
        } else {
#pragma unroll
          for (int cb = 0; cb < NCB; ++cb) {
            const uint32_t off = cb * kDecStageKeys * 128 + bx * p.rows_per_box * 128;
            if (bt) {
              tma_load_4d(smem_u32(kd + off), &tm_k, smem_u32(full + slot_i), cb * 64, hk, slot, pg);
              tma_load_4d(smem_u32(vd + off), &tm_v, smem_u32(full + slot_i), cb * 64, hk, slot, pg);
            } else {
              tma_load_3d(smem_u32(kd + off), &tm_k, smem_u32(full + slot_i), cb * 64, hk, krow0 + key0);
              tma_load_3d(smem_u32(vd + off), &tm_v, smem_u32(full + slot_i), cb * 64, hk, krow0 + key0);
            }
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------- consumers --
    // Q fragments (A operand, 16 rows x D) for all D/16 k-steps.
    uint32_t qf[D / 16][4];
    if constexpr (KDIR) {
      // The contraction index is permuted so that a lane's K bytes are
      // contiguous: in k-step ks, lane (g, t) holds the MMA's k positions
      // 2t, 2t+1, 2t+8, 2t+9, which stand for the dims 32t + 4ks + 0..3 --
      // four consecutive bytes of a key row.  Q takes the same order: a0/a2
      // of row r are its f16 pairs at dims 32t + 4ks and 32t + 4ks + 2.
      const int g = lane >> 2, t = lane & 3;
      const __half *q16 = reinterpret_cast<const __half *>(sQ);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint2 lo = *reinterpret_cast<const uint2 *>(q16 + g * D + 32 * t + 4 * ks);
        const uint2 hi = *reinterpret_cast<const uint2 *>(q16 + (g + 8) * D + 32 * t + 4 * ks);
        qf[ks][0] = lo.x;
        qf[ks][1] = hi.x;
        qf[ks][2] = lo.y;
        qf[ks][3] = hi.y;
      }
    } else {
      const uint32_t qbase = smem_u32(sQ);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        // matrices: (rows 0-7, k 0-7), (rows 8-15, k 0-7), (rows 0-7, k 8-15), (rows 8-15, k 8-15)
        const int mrow = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int mcol = ks * 16 + (lane >> 4) * 8;
        ldsm_x4(qbase + (mrow * D + mcol) * 2, qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
      }
    }
    // Rows this thread holds in the C fragments: g0 = lane/4, g1 = lane/4 + 8.
    // (QT: rows 2t and 2t+1, the columns of the S^T fragment)
    const int r0 = QT ? 2 * (lane & 3) : lane >> 2, r1 = QT ? r0 + 1 : r0 + 8;
    const int ip0 = (r0 / p.group) + sk - sq;   // bottom-right aligned positions
    const int ip1 = (r1 / p.group) + sk - sq;
    // byte caches: Q rows carry a factor 2^e that the score scale removes
    const float sc0 = KV ? p.scale_log2 * sQinv[r0] : p.scale_log2;
    const float sc1 = KV ? p.scale_log2 * sQinv[r1] : p.scale_log2;
    // score mods: the raw product <q, k> of row r is s * kf * qf_r
    const float qf0 = KV ? sQinv[r0] : 1.f, qf1 = KV ? sQinv[r1] : 1.f;
    const float c2u = 2.f * kLog2e * p.softcap_arg;   // soft-cap: raw product -> 2u log2(e)
    // block masks: the heads and query blocks of rows r0 and r1
    const int h0 = hk * p.group + r0 % p.group, h1 = hk * p.group + r1 % p.group;
    const int qb0 = (r0 / p.group) / 128, qb1 = (r1 / p.group) / 128;
    auto block_live = [&](int h, int qb, int kb) -> bool {
      if (p.block_mask == nullptr) return true;
      if (qb >= p.n_qblk || kb >= p.n_kblk) return false;
      return p.block_mask[((int64_t)(b * p.hq + h) * p.n_qblk + qb) * p.n_kblk + kb] != 0;
    };
    // Prologue terms: under the soft-cap, each row's term (pro_row_k *
    // sum_d q + pro_row_c) enters the capped score; a Q add's per-key term
    // comes from col_bias (already in the score's units).
    float rt0 = 0.f, rt1 = 0.f;
    if (p.mod == 2 && (p.pro_row_k != 0.f || p.pro_row_c != 0.f)) {
      auto row_sum = [&](int r) -> float {
        if (r >= rows || p.pro_row_k == 0.f) return 0.f;
        const __nv_bfloat16 *qrow =
            p.q + ((int64_t)qa + r / p.group) * p.q_stride_t + (int64_t)(hk * p.group + r % p.group) * p.q_stride_h;
        float qs = 0.f;
        for (int d = 0; d < D; ++d) qs += __bfloat162float(qrow[d]);
        return qs;
      };
      rt0 = fmaf(p.pro_row_k, row_sum(r0), p.pro_row_c);
      rt1 = fmaf(p.pro_row_k, row_sum(r1), p.pro_row_c);
    }
    const float *cb_row = p.col_bias ? p.col_bias + ((int64_t)b * p.hkv + hk) * p.cb_ld : nullptr;
    // one modified score in log2 units from the raw product x of row (ip, .),
    // with the row's and the key's prologue terms rt and cb
    auto mod_score = [&](float x, int ip, int j, float rt, float cb) -> float {
      if (p.mod == 2) {
        float r;
        return softcap_log2_score(ex2(fmaf(x, c2u, rt + cb)), p.softcap_log2, r);
      }
      return fmaf(x, p.scale_log2, cb - p.alibi_log2 * fabsf((float)(ip - j)));
    };
    uint8_t *conv = smem + Cfg::kOffConv + warp * Cfg::kConvWarpBytes;   // byte caches only
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    // O accumulators: D/8 n-tiles of 8 dims (rows r0, r1), or (OT) O^T as
    // D/16 m-tiles of 16 dims for the rows 2t, 2t+1 (see the P V product)
    constexpr int NO = OT ? D / 16 : D / 8;
    float o[NO][4];
#pragma unroll
    for (int n = 0; n < NO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    // Byte caches: stage offsets of the lane's 16-byte pieces, one per pass
    // (see convert below) -- token rows of D bytes, and K in the vectorized
    // 5-D pages, where key kk's bytes from column c0 sit at (kk / R) R D +
    // (c0 / 16) 16 R + (kk % R) 16, R = rows_per_box (a power of two).
    // 5-D V: the warp's 16 keys are one token group, [D][16 bytes] at
    // (kw / R) R D + ((kw % R) / 16) 16 D of the stage (kw = the warp's first key).
    int koff[D / 32], voff[D / 32], v5off;
    {
      const int R = p.rows_per_box, lg = __ffs(R) - 1, kw = warp * 16;
      v5off = ((kw >> lg) << lg) * D + ((kw & (R - 1)) >> 4) * 16 * D;
#pragma unroll
      for (int ps_ = 0; ps_ < D / 32; ++ps_) {
        const int off = ps_ * 512 + lane * 16;
        const int kk = kw + off / D, c0 = off % D;
        voff[ps_] = kw * D + off;
        koff[ps_] = V5 ? ((kk >> lg) << lg) * D + ((c0 >> 4) << (4 + lg)) + ((kk & (R - 1)) << 4) : voff[ps_];
      }
    }
    // KDIR: stage offsets of the 16-byte pieces (keys kw + g and kw + 8 + g,
    // dims 32t .. +15 and 32t+16 .. +31) the lane's QK fragments come from:
    // token-major rows 128-byte swizzled (kw is a multiple of 16, so both rows
    // swizzle by g, and a quarter warp covers all eight chunk positions: no
    // bank conflicts), or the 5-D pieces at (kk / R) R D + (c / 16) 16 R + (kk % R) 16
    int kdo[4];
    {
      const int g = lane >> 2, t = lane & 3, kw = warp * 16;
      const int R = p.rows_per_box, lg = __ffs(R) - 1;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int kk = kw + g + 8 * (i >> 1), cg = 2 * t + (i & 1);
        kdo[i] = V5 ? ((kk >> lg) << lg) * D + (cg << (4 + lg)) + ((kk & (R - 1)) << 4) : kk * 128 + ((cg ^ g) << 4);
      }
    }
    bool ok = true;
    for (int st = first_stage; st < n_stages; ++st) {
      const int it = st - first_stage;
      const int slot_i = it % NST;
      ok = mbar_wait(smem_u32(full + slot_i), (it / NST) & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      uint8_t *kd = stages + slot_i * Cfg::kStageBytes;
      uint8_t *vd = kd + Cfg::kKBytes;
      const int kw0 = warp * 16;                               // this warp's 16 keys in the stage
      const int key_base = key_lo + st * kDecStageKeys + kw0;  // sequence-local key of row kw0
      float ksc[2][2], vsc[2][2];                              // byte caches: scales of the lane's 4 keys
      // byte caches: this warp's 16 keys (16 x D bytes) -> f16 in its private
      // swizzled buffer, K first and V after the QK product.  Each pass, the
      // 32 lanes read 512 consecutive bytes (16 per lane, no bank conflicts);
      // keys at or past key_hi become zeros (their bytes may be anything).
      auto convert = [&](const uint8_t *src, const int (&offs)[D / 32]) {
#pragma unroll
        for (int ps_ = 0; ps_ < D / 32; ++ps_) {
          const int off = ps_ * 512 + lane * 16;
          const int lr = off / D, c0 = off % D;             // key within the 16, first element
          const bool live = key_base + lr < key_hi;
          const uint4 raw = live ? *reinterpret_cast<const uint4 *>(src + offs[ps_]) : make_uint4(0, 0, 0, 0);
          uint32_t h[8];
          dec_bytes4_to_f16<KV>(raw.x, h[0], h[1]);
          dec_bytes4_to_f16<KV>(raw.y, h[2], h[3]);
          dec_bytes4_to_f16<KV>(raw.z, h[4], h[5]);
          dec_bytes4_to_f16<KV>(raw.w, h[6], h[7]);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int c = c0 + half * 8;
            const int cb = c >> 6, ch = (c & 63) >> 3;
            *reinterpret_cast<uint4 *>(conv + cb * 16 * 128 + sw128(lr, ch)) =
                make_uint4(h[4 * half], h[4 * half + 1], h[4 * half + 2], h[4 * half + 3]);
          }
        }
        __syncwarp();
      };
      if constexpr (KV) {
        if constexpr (!KDIR) convert(kd, koff);
        const float *sct = reinterpret_cast<const float *>(vd + Cfg::kVBytes);
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int col = kw0 + n * 8 + (lane & 3) * 2 + e;
            ksc[n][e] = sct[col];
            vsc[n][e] = sct[kDecStageKeys + col];
          }
      }
      // Clear V rows of keys outside [key_lo, key_hi) (0 * NaN would be NaN).
      if (KV == 0 && key_base + 16 > key_hi) {
        for (int e = lane; e < 16 * NCB * 8; e += 32) {
          const int rr = e / (NCB * 8), rest = e % (NCB * 8);
          const int cb = rest / 8, ch = rest % 8;
          if (key_base + rr >= key_hi)
            *reinterpret_cast<uint4 *>(vd + cb * kDecStageKeys * 128 + (kw0 + rr) * 128 + ch * 16) =
                make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      float a0, a1;     // the rows' rescale factors (rows r0, r1)
      uint32_t pa[4];   // P as the A fragment of O = P V (rows g, g+8; keys 2t, 2t+1 / 2t+8, 2t+9)
      if constexpr (QT) {
        // S^T = K Q^T for the warp's 16 keys: M = 16 keys (g, g+8), N = 8
        // rows, the contraction order of the KDIR fragments.  C: keys g and
        // g+8 (c0/c1 and c2/c3) of rows 2t and 2t+1.  Two partial
        // accumulators (even and odd k-steps) halve the dependent chain.
        const uint4 ka0 = *reinterpret_cast<const uint4 *>(kd + kdo[0]);
        const uint4 ka1 = *reinterpret_cast<const uint4 *>(kd + kdo[1]);
        const uint4 kc0 = *reinterpret_cast<const uint4 *>(kd + kdo[2]);
        const uint4 kc1 = *reinterpret_cast<const uint4 *>(kd + kdo[3]);
        const uint32_t w0[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
        const uint32_t w1[8] = {kc0.x, kc0.y, kc0.z, kc0.w, kc1.x, kc1.y, kc1.z, kc1.w};
        float st[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t ak[4];
          dec_bytes4_to_f16<KV>(w0[ks], ak[0], ak[2]);
          dec_bytes4_to_f16<KV>(w1[ks], ak[1], ak[3]);
          dec_mma<KV>(st[ks & 1], ak, qf[ks][0], qf[ks][2]);
        }
        float sv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sv[e] = st[0][e] + st[1][e];
        const float *sct = reinterpret_cast<const float *>(vd + Cfg::kVBytes);
        const int g = lane >> 2, t = lane & 3;
        const bool blk0 = block_live(h0, qb0, key_base / 128), blk1 = block_live(h1, qb1, key_base / 128);
        float mx0 = -INFINITY, mx1 = -INFINITY;
        float vk[2];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          const int jj = kw0 + g + 8 * n;   // key within the stage
          const int j = key_base + g + 8 * n;
          const bool in = j < key_hi;
          bool ok0 = in && r0 < rows && blk0, ok1 = in && r1 < rows && blk1;
          if (p.causal) { ok0 = ok0 && j <= ip0; ok1 = ok1 && j <= ip1; }
          if (p.window > 0) {
            if (p.causal) { ok0 = ok0 && ip0 - j < p.window; ok1 = ok1 && ip1 - j < p.window; }
            else { ok0 = ok0 && abs(ip0 - j) < p.window; ok1 = ok1 && abs(ip1 - j) < p.window; }
          }
          const float kf = sct[jj];
          vk[n] = sct[kDecStageKeys + jj];
          float x0 = sv[2 * n], x1 = sv[2 * n + 1];
          if (p.mod == 0) {
            x0 = ok0 ? x0 * kf * sc0 : -INFINITY;
            x1 = ok1 ? x1 * kf * sc1 : -INFINITY;
          } else {
            const float cb = (cb_row && in && j < p.cb_ld) ? cb_row[j] : 0.f;
            x0 = ok0 ? mod_score(x0 * kf * qf0, ip0, j, rt0, cb) : -INFINITY;
            x1 = ok1 ? mod_score(x1 * kf * qf1, ip1, j, rt1, cb) : -INFINITY;
          }
          sv[2 * n] = x0;
          sv[2 * n + 1] = x1;
          mx0 = fmaxf(mx0, x0);
          mx1 = fmaxf(mx1, x1);
        }
        // the rows' maxima over the 16 keys: the 8 lanes of each t
#pragma unroll
        for (int o_ = 4; o_ < 32; o_ <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o_));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o_));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
        a0 = ex2(m0 - mu0);
        a1 = ex2(m1 - mu1);
        m0 = mn0;
        m1 = mn1;
        float pp[4];
        pp[0] = ex2(sv[0] - mu0);
        pp[1] = ex2(sv[1] - mu1);
        pp[2] = ex2(sv[2] - mu0);
        pp[3] = ex2(sv[3] - mu1);
        l0 = l0 * a0 + (pp[0] + pp[2]);   // per-thread partial sums; reduced over g at the end
        l1 = l1 * a1 + (pp[1] + pp[3]);
        // P (times the keys' v scales) to the A layout: lane (g, t) needs
        // row g at keys 2t, 2t+1 (and + 8), held by lanes (2t, g/2) and
        // (2t+1, g/2) as the half g mod 2 of their (row 2t', 2t'+1) pairs.
        const uint32_t pk0 = pack_f16x2(pp[0] * vk[0], pp[1] * vk[0]);
        const uint32_t pk1 = pack_f16x2(pp[2] * vk[1], pp[3] * vk[1]);
        const int src0 = ((2 * t) << 2) | (g >> 1), src1 = ((2 * t + 1) << 2) | (g >> 1);
        const uint32_t u0 = __shfl_sync(0xffffffffu, pk0, src0), u1 = __shfl_sync(0xffffffffu, pk0, src1);
        const uint32_t v0 = __shfl_sync(0xffffffffu, pk1, src0), v1 = __shfl_sync(0xffffffffu, pk1, src1);
        const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;
        pa[0] = __byte_perm(u0, u1, sel);
        pa[1] = 0u;
        pa[2] = __byte_perm(v0, v1, sel);
        pa[3] = 0u;
      } else {
      // S = Q K^T for 16 keys: two n-tiles of 8 keys.
      float s[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
      if constexpr (KDIR) {
        // Lane (g, t) reads 32 bytes (dims 32t .. 32t+31) of keys g and 8+g
        // of the warp's 16 (offsets kdo, fixed per lane).
        const uint4 a0 = *reinterpret_cast<const uint4 *>(kd + kdo[0]);
        const uint4 a1 = *reinterpret_cast<const uint4 *>(kd + kdo[1]);
        const uint4 c0 = *reinterpret_cast<const uint4 *>(kd + kdo[2]);
        const uint4 c1 = *reinterpret_cast<const uint4 *>(kd + kdo[3]);
        const uint32_t w0[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t w1[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t b0, b1;
          dec_bytes4_to_f16<KV>(w0[ks], b0, b1);
          dec_mma<KV>(s[0], qf[ks], b0, b1);
          dec_bytes4_to_f16<KV>(w1[ks], b0, b1);
          dec_mma<KV>(s[1], qf[ks], b0, b1);
        }
      }
#pragma unroll
      for (int ks = 0; ks < (KDIR ? 0 : D / 16); ++ks) {
        // matrices: (keys 0-7, dims 0-7), (keys 0-7, dims 8-15), (keys 8-15, dims 0-7), (keys 8-15, dims 8-15)
        const int krow = (lane & 7) + (lane >> 4) * 8;   // key within the warp's 16
        const int dim = ks * 16 + ((lane >> 3) & 1) * 8;
        const int cb = dim >> 6, ch = (dim & 63) >> 3;
        uint32_t b0, b1, b2, b3;
        const uint32_t kaddr = KV ? smem_u32(conv + cb * 16 * 128) + sw128(krow, ch)
                                  : smem_u32(kd + cb * kDecStageKeys * 128) + sw128(kw0 + krow, ch);
        ldsm_x4(kaddr, b0, b1, b2, b3);
        dec_mma<KV>(s[0], qf[ks], b0, b1);
        dec_mma<KV>(s[1], qf[ks], b2, b3);
      }
      // Scale, mask, online softmax for rows r0 and r1.  The warp's 16 keys
      // lie in one 128-key block.
      const bool blk0 = block_live(h0, qb0, key_base / 128), blk1 = block_live(h1, qb1, key_base / 128);
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < 2; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = key_base + n * 8 + (lane & 3) * 2 + e;
          const bool in = j < key_hi;
          bool ok0 = in && r0 < rows && blk0, ok1 = in && r1 < rows && blk1;
          if (p.causal) { ok0 = ok0 && j <= ip0; ok1 = ok1 && j <= ip1; }
          if (p.window > 0) {
            if (p.causal) { ok0 = ok0 && ip0 - j < p.window; ok1 = ok1 && ip1 - j < p.window; }
            else { ok0 = ok0 && abs(ip0 - j) < p.window; ok1 = ok1 && abs(ip1 - j) < p.window; }
          }
          const float kf = KV ? ksc[n][e] : 1.f;   // per-key scale of a byte cache
          if (p.mod == 0) {
            s[n][e] = ok0 ? s[n][e] * kf * sc0 : -INFINITY;
            s[n][2 + e] = ok1 ? s[n][2 + e] * kf * sc1 : -INFINITY;
          } else {
            const float cb = (cb_row && in && j < p.cb_ld) ? cb_row[j] : 0.f;
            s[n][e] = ok0 ? mod_score(s[n][e] * kf * qf0, ip0, j, rt0, cb) : -INFINITY;
            s[n][2 + e] = ok1 ? mod_score(s[n][2 + e] * kf * qf1, ip1, j, rt1, cb) : -INFINITY;
          }
          mx0 = fmaxf(mx0, s[n][e]);
          mx1 = fmaxf(mx1, s[n][2 + e]);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
      a0 = ex2(m0 - mu0);   // 0 when the old max is -inf
      a1 = ex2(m1 - mu1);
      m0 = mn0;
      m1 = mn1;
      float ps[2][4];
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        ps[n][0] = ex2(s[n][0] - mu0);
        ps[n][1] = ex2(s[n][1] - mu0);
        ps[n][2] = ex2(s[n][2] - mu1);
        ps[n][3] = ex2(s[n][3] - mu1);
        sum0 += ps[n][0] + ps[n][1];
        sum1 += ps[n][2] + ps[n][3];
      }
      l0 = l0 * a0 + sum0;   // per-thread partial sums; reduced across the quad at the end
      l1 = l1 * a1 + sum1;
      if constexpr (KV) {
        // P times the keys' v scales (f16; the row sums above use P itself)
        pa[0] = pack_f16x2(ps[0][0] * vsc[0][0], ps[0][1] * vsc[0][1]);
        pa[1] = pack_f16x2(ps[0][2] * vsc[0][0], ps[0][3] * vsc[0][1]);
        pa[2] = pack_f16x2(ps[1][0] * vsc[1][0], ps[1][1] * vsc[1][1]);
        pa[3] = pack_f16x2(ps[1][2] * vsc[1][0], ps[1][3] * vsc[1][1]);
      } else {
        pa[0] = pack_bf16x2(ps[0][0], ps[0][1]);
        pa[1] = pack_bf16x2(ps[0][2], ps[0][3]);
        pa[2] = pack_bf16x2(ps[1][0], ps[1][1]);
        pa[3] = pack_bf16x2(ps[1][2], ps[1][3]);
      }
      }
      // O is rescaled only when a row maximum moved somewhere in the warp
      // (after the first stages it rarely does); the factors are exactly 1
      // otherwise, so skipping changes nothing.
      if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
        if constexpr (OT) {
          // rows 2t and 2t+1: the thread's own (QT), or from lanes 8t and
          // 8t + 4 (g = row)
          const int t = lane & 3;
          const float at0 = QT ? a0 : __shfl_sync(0xffffffffu, a0, 8 * t);
          const float at1 = QT ? a1 : __shfl_sync(0xffffffffu, a0, 8 * t + 4);
#pragma unroll
          for (int n = 0; n < NO; ++n) {
            o[n][0] *= at0;
            o[n][1] *= at1;
            o[n][2] *= at0;
            o[n][3] *= at1;
          }
        } else if constexpr (QT) {
          // O rows g (and g+8, all zero): row g's factor from lane g/2 (t = g/2)
          const int g = lane >> 2;
          const float x0 = __shfl_sync(0xffffffffu, a0, g >> 1), x1 = __shfl_sync(0xffffffffu, a1, g >> 1);
          const float ag = (g & 1) ? x1 : x0;
#pragma unroll
          for (int n = 0; n < NO; ++n) {
            o[n][0] *= ag;
            o[n][1] *= ag;
          }
        } else {
#pragma unroll
          for (int n = 0; n < NO; ++n) {
            o[n][0] *= a0;
            o[n][1] *= a0;
            o[n][2] *= a1;
            o[n][3] *= a1;
          }
        }
      }
      if constexpr (DIRECT) {
        // O += P V with the bytes in registers.  Lane (g, t) reads the 16
        // bytes of dims 16g .. 16g+15 of keys 2t, 2t+1, 2t+8 and 2t+9 (the
        // k positions its B fragments hold; chunk g swizzled by the row:
        // conflict-free per quarter warp), zeroes keys past key_hi (their
        // bytes may be anything, and 0 * NaN would be NaN), and pairs the
        // keys' bytes per dim with byte permutes.  The output dims are
        // permuted too: n-tile j, column n stands for dim 16n + j.
        const int g = lane >> 2, t = lane & 3;
        const int rk[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
        uint4 vr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = kw0 + rk[i];
          vr[i] = *reinterpret_cast<const uint4 *>(vd + row * 128 + ((g ^ (row & 7)) << 4));
          if (key_base + rk[i] >= key_hi) vr[i] = make_uint4(0, 0, 0, 0);
        }
        const uint32_t r0w[4] = {vr[0].x, vr[0].y, vr[0].z, vr[0].w}, r1w[4] = {vr[1].x, vr[1].y, vr[1].z, vr[1].w};
        const uint32_t r2w[4] = {vr[2].x, vr[2].y, vr[2].z, vr[2].w}, r3w[4] = {vr[3].x, vr[3].y, vr[3].z, vr[3].w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t b0[4], b1[4];   // per dim 16g + 4w + i: keys (2t, 2t+1) and (2t+8, 2t+9)
          dec_bytes4_to_f16<KV>(__byte_perm(r0w[w], r1w[w], 0x5140), b0[0], b0[1]);
          dec_bytes4_to_f16<KV>(__byte_perm(r0w[w], r1w[w], 0x7362), b0[2], b0[3]);
          dec_bytes4_to_f16<KV>(__byte_perm(r2w[w], r3w[w], 0x5140), b1[0], b1[1]);
          dec_bytes4_to_f16<KV>(__byte_perm(r2w[w], r3w[w], 0x7362), b1[2], b1[3]);
          if constexpr (OT) {
            // O^T += V^T P^T: m-tile j's rows g and g+8 stand for the dims
            // 16g + 2j and 16g + 2j + 1, so the pairs above are its A
            // fragments as they come; B = P^T is pa[0] / pa[2] (row g of P,
            // keys 2t, 2t+1 and 2t+8, 2t+9).  C: rows 2t, 2t+1 of O.
            const uint32_t e0[4] = {b0[0], b0[1], b1[0], b1[1]}, e1[4] = {b0[2], b0[3], b1[2], b1[3]};
            dec_mma<KV>(o[2 * w], e0, pa[0], pa[2]);
            dec_mma<KV>(o[2 * w + 1], e1, pa[0], pa[2]);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) dec_mma<KV>(o[4 * w + i], pa, b0[i], b1[i]);
          }
        }
        // every lane has used its K and V bytes and the stage's scales
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(empty + slot_i));
      } else if constexpr (KV) {
        __syncwarp();                 // the QK product has read K from the buffer
        if constexpr (V5) {
          // 5-D V (the token group at v5off): lane (octet oc, half th)
          // transposes 8 tokens x 8 dims and writes 8 key rows.
          const uint8_t *gsrc = vd + v5off;
          const int oc = lane >> 1, th = lane & 1;
          if (oc < D / 8) {
            uint2 in[8], tr[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) in[k] = *reinterpret_cast<const uint2 *>(gsrc + (8 * oc + k) * 16 + 8 * th);
            transpose_8x8_bytes(in, tr);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const int lr = 8 * th + t;
              uint32_t h[4];
              dec_bytes4_to_f16<KV>(tr[t].x, h[0], h[1]);
              dec_bytes4_to_f16<KV>(tr[t].y, h[2], h[3]);
              if (key_base + lr >= key_hi) h[0] = h[1] = h[2] = h[3] = 0u;
              const int c = 8 * oc, cb = c >> 6, ch = (c & 63) >> 3;
              *reinterpret_cast<uint4 *>(conv + cb * 16 * 128 + sw128(lr, ch)) = make_uint4(h[0], h[1], h[2], h[3]);
            }
          }
          __syncwarp();
        } else {
          convert(vd, voff);
        }
        // the stage's bytes and scales are no longer needed by this warp
        if (lane == 0) mbar_arrive(smem_u32(empty + slot_i));
      }
      // O += P V : D/8 n-tiles of 8 dims, one k-step of 16 keys.
#pragma unroll
      for (int nd = 0; nd < (DIRECT ? 0 : D / 16); ++nd) {
        // matrices: (keys 0-7, dims 0-7), (keys 8-15, dims 0-7), (keys 0-7, dims 8-15), (keys 8-15, dims 8-15)
        const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;   // key within the warp's 16
        const int dim = nd * 16 + (lane >> 4) * 8;
        const int cb = dim >> 6, ch = (dim & 63) >> 3;
        uint32_t b0, b1, b2, b3;
        const uint32_t vaddr = KV ? smem_u32(conv + cb * 16 * 128) + sw128(krow, ch)
                                  : smem_u32(vd + cb * kDecStageKeys * 128) + sw128(kw0 + krow, ch);
        ldsm_x4_t(vaddr, b0, b1, b2, b3);
        dec_mma<KV>(o[2 * nd], pa, b0, b1);
        dec_mma<KV>(o[2 * nd + 1], pa, b2, b3);
      }
      __syncwarp();
      if (KV == 0 && lane == 0) mbar_arrive(smem_u32(empty + slot_i));
    }

    // Reduce l over the lanes sharing a row: the quad, or (QT) the 8 lanes of a t.
#pragma unroll
    for (int o_ = QT ? 4 : 1; o_ < (QT ? 32 : 4); o_ <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o_);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o_);
    }

    // Merge the four warps' (m, l, O) through shared memory (stage buffers are
    // free once every warp has passed its last stage).
    float *red_o = reinterpret_cast<float *>(stages);                     // [4][16][D]
    float *red_ml = reinterpret_cast<float *>(stages + kDecWarps * kDecRows * D * 4);  // [4][16][2]
    asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32));
    if (ok && OT) {
      // O^T m-tile j of lane (g, t): rows 2t, 2t+1 at the dims 16g + 2j, +1
      const int g = lane >> 2, t = lane & 3;
#pragma unroll
      for (int j = 0; j < NO; ++j) {
        const int c = 16 * g + 2 * j;
        *reinterpret_cast<float2 *>(red_o + (warp * kDecRows + 2 * t) * D + c) = make_float2(o[j][0], o[j][2]);
        *reinterpret_cast<float2 *>(red_o + (warp * kDecRows + 2 * t + 1) * D + c) = make_float2(o[j][1], o[j][3]);
      }
    } else if (ok) {
#pragma unroll
      for (int n = 0; n < NO; ++n) {
        // O rows g and g+8; DIRECT: n-tile n, column 2t + e is dim 16 (2t + e) + n
        const int og = lane >> 2;
        const int c = DIRECT ? 32 * (lane & 3) + n : n * 8 + (lane & 3) * 2;
        const int c1 = DIRECT ? c + 16 : c + 1;
        red_o[(warp * kDecRows + og) * D + c] = o[n][0];
        red_o[(warp * kDecRows + og) * D + c1] = o[n][1];
        red_o[(warp * kDecRows + og + 8) * D + c] = o[n][2];
        red_o[(warp * kDecRows + og + 8) * D + c1] = o[n][3];
      }
    }
    // m and l of rows r0, r1: one lane per row pair (QT: the lanes with g = 0)
    if (ok && (QT ? (lane >> 2) == 0 : (lane & 3) == 0)) {
      red_ml[(warp * kDecRows + r0) * 2] = m0;
      red_ml[(warp * kDecRows + r0) * 2 + 1] = l0;
      red_ml[(warp * kDecRows + r1) * 2] = m1;
      red_ml[(warp * kDecRows + r1) * 2 + 1] = l1;
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32));
    if (ok) {
      // 128 threads: thread -> (row = tid / 8, 16-dim slice = tid % 8 ... for D=128)
      constexpr int kPerRow = kDecWarps * 32 / kDecRows;   // 8 threads per row
      constexpr int kSlice = D / kPerRow;
      const int row = threadIdx.x / kPerRow, sl = threadIdx.x % kPerRow;
      if (row < rows) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, red_ml[(w * kDecRows + row) * 2]);
        float wgt[kDecWarps], L = 0.f;
        const float Mu = M == -INFINITY ? 0.f : M;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
          wgt[w] = ex2(red_ml[(w * kDecRows + row) * 2] - Mu);
          L += wgt[w] * red_ml[(w * kDecRows + row) * 2 + 1];
        }
        const bool has = L > 0.f;
        const float inv = has ? 1.f / L : 0.f;
        const float sc = inv * p.pro_vmul;   // prologue's V map folded into the normalisation
        const int tq = row / p.group, h = hk * p.group + row % p.group;
        const int64_t t = (int64_t)qa + tq;
        float lse_v = has ? (M + __log2f(L)) * kLn2 : -INFINITY;
        if (has) lse_v += p.pro_lse_c;     // the prologue's row term, carried by the LSE
        if (has && p.pro_lse_k != 0.f) {
          const __nv_bfloat16 *qrow = p.q + t * p.q_stride_t + (int64_t)h * p.q_stride_h;
          float qs = 0.f;
          for (int d = 0; d < D; ++d) qs += __bfloat162float(qrow[d]);
          lse_v += p.pro_lse_k * qs;
        }
        if (p.o_part) {
          float *dst = p.o_part + (((int64_t)split * p.total_q + t) * p.hq + h) * D + sl * kSlice;
#pragma unroll
          for (int d = 0; d < kSlice; d += 4) {
            float4 v;
            float *vv = reinterpret_cast<float *>(&v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float acc = 0.f;
#pragma unroll
              for (int w = 0; w < kDecWarps; ++w) acc += wgt[w] * red_o[(w * kDecRows + row) * D + sl * kSlice + d + e];
              vv[e] = has ? fmaf(acc, sc, p.pro_vadd) : 0.f;
            }
            *reinterpret_cast<float4 *>(dst + d) = v;
          }
          if (sl == 0) p.lse_part[((int64_t)split * p.hq + h) * p.total_q + t] = lse_v;
        } else {
          __nv_bfloat16 *dst = p.out + t * p.out_stride_t + (int64_t)h * p.out_stride_h + sl * kSlice;
#pragma unroll
          for (int d = 0; d < kSlice; d += 2) {
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) {
              acc0 += wgt[w] * red_o[(w * kDecRows + row) * D + sl * kSlice + d];
              acc1 += wgt[w] * red_o[(w * kDecRows + row) * D + sl * kSlice + d + 1];
            }
            *reinterpret_cast<uint32_t *>(dst + d) =
                has ? pack_bf16x2(fmaf(acc0, sc, p.pro_vadd), fmaf(acc1, sc, p.pro_vadd)) : 0u;
          }
          if (sl == 0 && p.lse) p.lse[(int64_t)h * p.total_q + t] = lse_v;
        }
      }
    }
  }
}

// Combine kernel: one warp per (row t, head h).
template <int D>
__global__ void __launch_bounds__(256) fa_combine_kernel(const float *__restrict__ o_part,
                                                         const float *__restrict__ lse_part, int num_splits,
                                                         int64_t n_rows, int hq, __nv_bfloat16 *__restrict__ out,
                                                         float *__restrict__ lse) {
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= n_rows * hq) return;
  const int64_t t = wid / hq;
  const int h = (int)(wid % hq);
  float M = -INFINITY;
  for (int s = lane; s < num_splits; s += 32) M = fmaxf(M, lse_part[((int64_t)s * hq + h) * n_rows + t]);
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  constexpr int kPer = D / 32;
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  float L = -INFINITY;
  if (M != -INFINITY) {
    float den = 0.f;
    for (int s = lane; s < num_splits; s += 32) den += __expf(lse_part[((int64_t)s * hq + h) * n_rows + t] - M);
#pragma unroll
    for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    L = M + __logf(den);
    for (int s = 0; s < num_splits; ++s) {
      const float ls = lse_part[((int64_t)s * hq + h) * n_rows + t];
      if (ls == -INFINITY) continue;
      const float w = __expf(ls - L);
      const float *src = o_part + (((int64_t)s * n_rows + t) * hq + h) * D + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; e += 2) {
        const float2 v = *reinterpret_cast<const float2 *>(src + e);
        acc[e] += w * v.x;
        acc[e + 1] += w * v.y;
      }
    }
  }
  __nv_bfloat16 *dst = out + (t * hq + h) * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; e += 2) *reinterpret_cast<uint32_t *>(dst + e) = pack_bf16x2(acc[e], acc[e + 1]);
  if (lse && lane == 0) lse[(int64_t)h * n_rows + t] = L;
}

}  // namespace fa
