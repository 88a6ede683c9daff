// fa_prefill3.cuh -- two-query-tile (ping-pong) tcgen05 FlashAttention forward
// with a chunked K ring: the kernel for Q/K head dim 192 (V/O 128) and for
// e4m3 K/V caches of every head dim.
//
// The schedule is the one of fa_prefill2.cuh: one CTA computes 256 query rows
// of one (sequence, head) as two 128-row tiles A and B, each owned by a softmax
// warpgroup, while the tensor core alternates between them:
//
//   MMA order:  QK_A(0) QK_B(0) | PV_A(0) QK_A(1) PV_B(0) QK_B(1) | PV_A(1) ...
//
// What changes is the staging of K.  With Dk = 192 the two Q tiles alone take
// 96 KB of shared memory, so K is kept as a ring of 16 KB chunks (one 64-column
// block of 128 keys each) rather than whole-tile stages: a chunk is refilled as
// soon as the last QK that reads it completes, and the QK of the next tile can
// start on its first chunk while the others still load.  V keeps whole-tile
// stages (the PV operand spans its 64-column blocks at a fixed stride).
//
// e4m3 caches (FlyDSL PR #1066: paged FP8 K/V with per-token scales) and int8
// caches (fkl_python PR #7: per-token int8 KV dequantisation) are staged by
// TMA as raw bytes and turned into f16 MMA operands in shared memory by six
// converter warps:
//   K' = RN_f16(dec(k) * k_scale),  V' = RN_f16(dec(v) * v_scale)
// (one rounding each, fp32 product).  Q is brought to f16 in place with a
// per-row power-of-two factor 2^e (exact for every bf16 value within 2^-28 of
// the row maximum; the factor 2^-e returns in the softmax scale), so both
// contractions run as kind::f16 with fp32 accumulation and P is packed as f16.
// Each converted 32-row slice is staged in the upper half of its own output
// region, so one warp converts it in place without waiting for other warps.
//
// TMEM (512 columns):  S_A [0,128)  S_B [128,256)  O_A [256,384)  O_B [384,512)
// with P_X (16-bit, the A operand of PV) written over the first 64 columns of S_X.
//
// Warps: 0-3 softmax A, 4-7 softmax B, 8 TMA producer, 9 TMEM allocation + MMA
// issue; e4m3: 10-15 converters (16 warps); bf16: 10-11 idle in the 12-warp
// variant (warpgroup 2 hands its registers to the softmax warpgroups).
//
// Q8 (e4m3 Q with e4m3 K/V, Dk 128 or 192, Dv 128; FlyDSL PR #1066
// description: OCP E4M3 Q/K/V with scalar descales): Q and K are the operands
// of a kind::f8f6f4 QK as stored -- TMA drops them 128-byte swizzled in
// chunks of 128 columns, no conversion -- so S' = sum_d q8 k8 and the score
// is S'_ij * k_scale_j (the per-tensor Q scale is part of softmax_scale).
// At Dk 192 a row spans two chunks; TMA fills columns 192..255 of the second
// with zeros and the QK skips them.  The producer lanes copy the 128 K
// scales of a tile with cp.async into a ring of their own (one slot per
// tile); the softmax multiplies each S column by its scale before the max.
// V is still converted to f16 and PV runs kind::f16 with P in f16.
#pragma once
#include "fa_prefill2.cuh"

namespace fa {

// PV8 (with Q8): P * V on the e4m3 bytes as well -- P in e4m3 in shared
// memory, V transposed by the converters into a K-major e4m3 operand,
// kind::f8f6f4 -- an opt-in precision mode (see the P8 notes in the kernel).
template <int DK, int DV, bool PAGED, bool FP8, int MOD, bool BIGREG, bool Q8 = false, bool PV8 = false>
struct Prefill3Cfg {
  // 16 KB chunks per K tile: 64 bf16/f16 columns, or (Q8) 128 e4m3 columns
  // (Dk 192: two chunks, the second half zero-filled by TMA)
  static constexpr int KC = Q8 ? (DK + 127) / 128 : DK / 64;
  static constexpr int VC = DV / 64;              // 64-column blocks per V tile
  static constexpr int kChunkBytes = kBlockN * 128;
  static constexpr int kQTileBytes = Q8 ? KC * kBlockM * 128 : kBlockM * DK * 2;
  static constexpr int kVBytes = VC * kChunkBytes;
  // Q8: a ring of NSS tiles' K scales (NSS >= NSV + 1: see the producer);
  // PV8 adds the V scales beside them and two e4m3 P tiles
  static constexpr int NSS = Q8 ? 4 : 1;
  static constexpr int kKsBytes = Q8 ? (PV8 ? 2 : 1) * NSS * kBlockN * 4 : 0;
  static constexpr int kPBytes = PV8 ? 2 * kBlockM * 128 : 0;
  static constexpr int kRing = 229376 - 2 * kQTileBytes - kPBytes;   // 224 KB minus the Q (and P) tiles
  static constexpr int NSV = (DV <= 64) ? 6 : 2;
  static constexpr int NCK_raw = (kRing - NSV * kVBytes - kKsBytes) / kChunkBytes;
  static constexpr int NCK = NCK_raw > 8 ? 8 : NCK_raw;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = 2 * kQTileBytes;
  static constexpr int kOffV = kOffK + NCK * kChunkBytes;
  static constexpr int kOffP = kOffV + NSV * kVBytes;
  static constexpr int kOffKs = kOffP + kPBytes;
  static constexpr int kOffBar = kOffKs + kKsBytes;
  // q_full, q_conv[2], kc_full/kc_empty/kc_stage[NCK], v_full/v_empty/v_stage[NSV],
  // s_full[2], p_full[2], o_done[2], Q8: ks_full[NSS]
  static constexpr int kNumBars = 3 + 3 * NCK + 3 * NSV + 6 + (Q8 ? NSS : 0);
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 64;
  // e4m3: 16 warps, always with the register split; bf16: BIGREG selects the
  // 12-warp split variant, otherwise 10 warps without setmaxnreg.
  static constexpr bool kSplitRegs = FP8 || BIGREG;
  static constexpr int kWarps = FP8 ? 16 : (BIGREG ? 12 : 10);
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kRegsSoftmax = FP8 ? 168 : 208;
  static constexpr int kRegsOther = FP8 ? 88 : 80;
  // Softmax over the whole S row at once (BIGREG, e4m3 with kOnePassFP8) or
  // in two 64-column halves.
  static constexpr bool kOnePassFP8 = false;
  static constexpr bool kOnePass = FP8 ? kOnePassFP8 : BIGREG;
  static constexpr int kPoolNeeded = 8 * 32 * kRegsSoftmax + (kWarps - 8) * 32 * kRegsOther;
  static constexpr int kConverters = 6;
  static constexpr int kKSlices = Q8 ? 0 : KC * 4;      // 32-row K slices to convert per tile
  static constexpr int kSlicesPerTile = kKSlices + VC * 4;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(DK % 64 == 0 && DV % 64 == 0 && DV <= 128, "head dims");
  static_assert(NCK >= KC, "the K ring holds at least one tile");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(!kSplitRegs || kPoolNeeded <= 65536, "register split exceeds the register file");
  static_assert(!Q8 || (FP8 && (DK == 128 || DK == 192) && DV == 128),
                "e4m3 Q runs with e4m3 K/V at Dk 128 or 192, Dv 128");
  static_assert(!Q8 || NSS >= NSV + 1, "K scales outlive their readers");
  static_assert(!PV8 || (Q8 && DV == 128), "e4m3 P * V: with e4m3 Q, Dv 128");
};

// tcgen05 MMA with A and B from shared memory, e4m3 x e4m3 -> fp32 (K = 32 per
// instruction); descriptor words as in mma_ss_w.
template <int ACC>
__device__ __forceinline__ void mma_ss_f8_w(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                            uint32_t b_hi, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "n"(ACC)
      : "memory");
}

// 4-byte global -> shared copy (cp.async); `bytes` 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}

// One arrival on `bar` once this thread's earlier cp.async copies have landed
// (counted in the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Packed fp32 products a *= b (one rounding each).
__device__ __forceinline__ void mul2(float &a0, float &a1, float b0, float b1) {
  asm("{\n\t.reg .b64 x, y, r;\n\t"
      "mov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
      "mul.f32x2 r, x, y;\n\tmov.b64 {%0, %1}, r;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

// f16 pair (packed) -> two fp32 values.
__device__ __forceinline__ void unpack_f16x2(uint32_t h, float &lo, float &hi) {
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h));
}

// Four floats -> four e4m3 bytes (a in the low byte), round to nearest,
// saturating at +-448; and back (exact).
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 l, h;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 l, %2, %1;\n\tcvt.rn.satfinite.e4m3x2.f32 h, %4, %3;\n\t"
      "mov.b32 %0, {l, h};\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}
__device__ __forceinline__ void unpack_e4m3x4(uint32_t w, float &a, float &b, float &c, float &d) {
  uint32_t lo, hi;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
  unpack_f16x2(lo, a, b);
  unpack_f16x2(hi, c, d);
}


// Two e4m3 bytes (low 16 bits of `two`) -> f16 pair, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t h;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "r"(two));
  return h;
}

// Four e4m3 bytes times an fp32 scale -> two f16 pairs (one rounding each).
__device__ __forceinline__ void e4m3x4_scaled_f16(uint32_t w, float s, uint32_t &o0, uint32_t &o1) {
  float a, b, c, d;
  unpack_f16x2(e4m3x2_to_f16x2(w & 0xFFFFu), a, b);
  unpack_f16x2(e4m3x2_to_f16x2(w >> 16), c, d);
  fma2(a, b, a, b, s, 0.f);   // packed fp32 products, rounded once
  fma2(c, d, c, d, s, 0.f);
  o0 = pack_f16x2(a, b);
  o1 = pack_f16x2(c, d);
}

// Four int8 bytes times an fp32 scale -> two f16 pairs.  Each byte becomes an
// exact fp32 through the float 2^23 + (x + 128) -- the byte, offset by 128,
// in the low mantissa bits -- minus 2^23 + 128; then one product and one
// rounding to f16.
__device__ __forceinline__ void i8x4_scaled_f16(uint32_t w, float s, uint32_t &o0, uint32_t &o1) {
  const uint32_t u = w ^ 0x80808080u;
  float a = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650));
  float b = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651));
  float c = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652));
  float d = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653));
  add2(a, b, -8388736.f, -8388736.f);
  add2(c, d, -8388736.f, -8388736.f);
  fma2(a, b, a, b, s, 0.f);
  fma2(c, d, c, d, s, 0.f);
  o0 = pack_f16x2(a, b);
  o1 = pack_f16x2(c, d);
}

// I8 (with FP8): the byte cache holds int8 values instead of e4m3.
// Q8 (with FP8, not I8): Q is e4m3 too and QK runs on the e4m3 bytes.
// V5 (with FP8 and PAGED, not Q8): the pages are in the vectorized 5-D
// layouts; kernels of their own, so that the token-major kernels carry none
// of the 5-D code.
template <int DK, int DV, bool PAGED, bool FP8, int MOD, bool BIGREG, bool I8, bool Q8 = false, bool V5 = false,
          bool PV8 = false>
__global__ void __launch_bounds__(Prefill3Cfg<DK, DV, PAGED, FP8, MOD, BIGREG, Q8, PV8>::kThreads, 1)
    fa_prefill3_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using Cfg = Prefill3Cfg<DK, DV, PAGED, FP8, MOD, BIGREG, Q8, PV8>;
  static_assert(!V5 || (FP8 && PAGED && !Q8), "5-D pages: paged byte caches with bf16 Q");
  // MOD: 0 plain scores, 1 ALiBi, 2 soft-cap; 3 and 4 are 1 and 2 with the
  // prologue's score terms (KT): a Q add's per-key term and, under the
  // soft-cap, the row term of a K add
  constexpr int MK = MOD >= 3 ? MOD - 2 : MOD;
  constexpr bool KT = MOD >= 3;
  static_assert(!(Q8 && I8), "int8 keys have no e4m3 QK");
  constexpr int KC = Cfg::KC, VC = Cfg::VC, NCK = Cfg::NCK, NSV = Cfg::NSV;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // 128-byte-swizzled operands need 1024-byte aligned chunks.
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) record_error(p.err, kErrBounds);
    return;
  }

  // ------------------------------------------------------------ work tile --
  PairInfo pi;
  int pt;
  if (!decode_block(p, (int)blockIdx.x, pi.b, pi.h, pt)) return;
  pi.hk = pi.h / p.group;
  {
    const int qa = __ldg(p.cu_q + pi.b), qb = __ldg(p.cu_q + pi.b + 1);
    const int ka = __ldg(p.cu_k + pi.b), kb = __ldg(p.cu_k + pi.b + 1);
    pi.sq = qb - qa;
    pi.sk = kb - ka;
    pi.q_row0 = qa + pt * 2 * kBlockM;
    pi.k_row0 = ka;
  }
  if (pt * 2 * kBlockM >= pi.sq) return;
  pi.kt_lo = 1 << 30;
  pi.kt_hi = 0;
#pragma unroll
  for (int X = 0; X < 2; ++X) {
    Half &hx = pi.x[X];
    hx.qt = pt * 2 + X;
    hx.q0 = hx.qt * kBlockM;
    hx.valid = hx.q0 < pi.sq;
    hx.klo = hx.khi = 0;
    if (!hx.valid) continue;
    const int last = min(hx.q0 + kBlockM, pi.sq) - 1;
    hx.ip_min = hx.q0 + pi.sk - pi.sq;
    hx.ip_max = last + pi.sk - pi.sq;
    int lo = 0, hi = pi.sk;
    if (p.causal) hi = min(hi, hx.ip_max + 1);
    if (p.window > 0) {
      lo = max(lo, hx.ip_min - p.window + 1);
      if (!p.causal) hi = min(hi, hx.ip_max + p.window);
    }
    if (hi > lo) {
      hx.klo = lo / kBlockN;
      hx.khi = (hi + kBlockN - 1) / kBlockN;
      pi.kt_lo = min(pi.kt_lo, hx.klo);
      pi.kt_hi = max(pi.kt_hi, hx.khi);
    }
  }
  if (pi.kt_hi == 0) pi.kt_lo = 0;
  int first_kt = pi.kt_lo;
  if (first_kt < pi.kt_hi && !half_active(p, pi, 0, first_kt) && !half_active(p, pi, 1, first_kt))
    first_kt = pair_next(p, pi, first_kt);
  int n_tiles = 0;
  for (int kt = first_kt; kt < pi.kt_hi; kt = pair_next(p, pi, kt)) ++n_tiles;

  if (n_tiles == 0) {
    for (int e = threadIdx.x; e < 2 * kBlockM; e += blockDim.x) {
      const int i = pt * 2 * kBlockM + e;
      if (i >= pi.sq) break;
      const int64_t t = (int64_t)pi.q_row0 + e;
      __nv_bfloat16 *o = p.out + t * p.out_stride_t + (int64_t)pi.h * p.out_stride_h;
      for (int d = 0; d < DV; d += 8) *reinterpret_cast<uint4 *>(o + d) = make_uint4(0, 0, 0, 0);
      if (p.lse) p.lse[(int64_t)pi.h * p.total_q + t] = -INFINITY;
    }
    return;
  }

  // ----------------------------------------------------------- shared mem --
  uint8_t *sQ = smem + Cfg::kOffQ;
  uint8_t *sK = smem + Cfg::kOffK;
  uint8_t *sV = smem + Cfg::kOffV;
  float *sKs = reinterpret_cast<float *>(smem + Cfg::kOffKs);   // Q8: [NSS][kBlockN]
  float *sVs = sKs + Cfg::NSS * kBlockN;                         // PV8: [NSS][kBlockN] V scales
  uint8_t *sP = smem + Cfg::kOffP;                               // PV8: [2][128 rows][128 keys] e4m3
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
  uint64_t *q_full = bars;
  uint64_t *q_conv = bars + 1;          // [2] Q tile in f16 (e4m3 caches)
  uint64_t *kc_full = bars + 3;         // [NCK] chunk holds its MMA operand
  uint64_t *kc_empty = kc_full + NCK;   // [NCK] last QK reading it completed
  uint64_t *kc_stage = kc_empty + NCK;  // [NCK] e4m3 bytes landed
  uint64_t *v_full = kc_stage + NCK;
  uint64_t *v_empty = v_full + NSV;
  uint64_t *v_stage = v_empty + NSV;
  uint64_t *s_full = v_stage + NSV;     // [2]
  uint64_t *p_full = s_full + 2;        // [2]
  uint64_t *o_done = p_full + 2;        // [2]
  uint64_t *ks_full = o_done + 2;       // Q8: [NSS] a tile's K scales landed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 8);

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    mbar_init(smem_u32(q_conv + 0), kBlockM);
    mbar_init(smem_u32(q_conv + 1), kBlockM);
    // barriers the producer fills: one arrival with the TMA bytes, or one per
    // producer lane for gathered rows (pages of < 16 keys, never with Q8)
    const uint32_t n_fill = (PAGED && !Q8 && p.gather) ? 32u : 1u;
    for (int s = 0; s < NCK; ++s) {
      // converted K: one arrive per slice; Q8: the TMA arrive
      mbar_init(smem_u32(kc_full + s), Q8 ? 1 : (FP8 ? 4 : n_fill));
      mbar_init(smem_u32(kc_empty + s), 1);
      mbar_init(smem_u32(kc_stage + s), n_fill);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(smem_u32(v_full + s), FP8 ? 4 * VC : n_fill);
      mbar_init(smem_u32(v_empty + s), 1);
      mbar_init(smem_u32(v_stage + s), n_fill);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(s_full + x), 1);
      mbar_init(smem_u32(p_full + x), kBlockM);
      mbar_init(smem_u32(o_done + x), 1);
    }
    if constexpr (Q8)
      for (int s = 0; s < Cfg::NSS; ++s) mbar_init(smem_u32(ks_full + s), 32);   // one per producer lane
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Register split: the softmax warpgroups take what the other warpgroups
  // release.  The host launches a split variant only when the kernel's launch
  // register count makes Cfg::kPoolNeeded fit the CTA's register pool.
  if (Cfg::kSplitRegs && warp >= 8) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::kRegsOther));

  const int32_t *bt = PAGED ? p.block_table + (int64_t)pi.b * p.bt_stride : nullptr;

  if (warp == 8) {
    // ------------------------------------------------ producer: Q, K, V --
    // Lane 0 waits for ring slots and arms the barriers; the boxes of a
    // 64-column block (one per `rows_per_box` keys) are issued by lanes
    // 0..n-1 in parallel, each with its own page id, looked up one tile ahead.
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_expect_tx(smem_u32(q_full), 2 * Cfg::kQTileBytes);
#pragma unroll
      for (int X = 0; X < 2; ++X)
#pragma unroll
        for (int cb = 0; cb < KC; ++cb)
          tma_load_3d(smem_u32(sQ + X * Cfg::kQTileBytes + cb * kBlockM * 128), &tm_q, smem_u32(q_full),
                      cb * (Q8 ? 128 : 64), pi.h, pi.q_row0 + X * kBlockM);
    }
    const int rb = p.rows_per_box;
    const int nbox = kBlockN / rb;                    // 1..8 boxes per 64-column block (pages >= 16 keys)
    const int r0 = lane * rb;                         // this lane's first key row in a tile
    const bool boxer = lane < nbox;
    auto page_at = [&](int kt) -> int {
      if constexpr (PAGED) {
        const int key0 = kt * kBlockN + r0;
        return (boxer && kt < pi.kt_hi && key0 < pi.sk) ? __ldg(bt + (key0 >> p.page_shift)) : -1;
      } else {
        return 0;
      }
    };
    // One 128-byte-row block of a K or V tile into a 16 KB chunk: bf16 rows
    // (64 columns) and Q8 key rows (128 e4m3 columns) land swizzled, the MMA
    // operand; staged byte rows (64 columns) land raw in the upper half of
    // their 32-row slice, for the converters.
    // Vectorized 5-D byte caches (V5): a box of a page piece lands as
    // [4 column groups][rows][16 bytes] for K and [rows / 16][64 dims][16
    // tokens] for V, in the same bytes the token-major box fills; the
    // converters read either form.  PV8: a V block's byte rows (64 columns)
    // land raw and contiguous ([128 keys][64 bytes]) in the upper half of the
    // V stage, and the converters transpose them into its lower half.
    auto load_block = [&](const CUtensorMap *tm, uint8_t *dst, uint64_t *bar, int x, int kt, int page, bool staged,
                          bool isv) {
      if (!boxer) return;
      const uint32_t at = (PV8 && isv) ? smem_u32(dst + r0 * 64)
                          : staged     ? smem_u32(dst + (r0 >> 5) * 4096 + 2048 + (r0 & 31) * 64)
                                       : smem_u32(dst + r0 * 128);
      if constexpr (PAGED) {
        const int slot = (kt * kBlockN + r0) & (p.page_size - 1);
        if constexpr (V5) {
          if (isv) tma_load_5d(at, tm, smem_u32(bar), 0, x, slot >> 4, pi.hk, page);
          else tma_load_5d(at, tm, smem_u32(bar), 0, slot, x >> 4, pi.hk, page);
        } else {
          tma_load_4d(at, tm, smem_u32(bar), x, pi.hk, slot, page);
        }
      } else {
        tma_load_3d(at, tm, smem_u32(bar), x, pi.hk, pi.k_row0 + kt * kBlockN + r0);
      }
    };
    constexpr bool kStageK = FP8 && !Q8;
    constexpr uint32_t kKBlockBytes = kStageK ? kBlockN * 64 : kBlockN * 128;
    constexpr uint32_t kVBlockBytes = FP8 ? kBlockN * 64 : kBlockN * 128;
    // Q8: lane l copies the scales of keys 4l .. 4l+3 of a tile (one page:
    // pages hold >= 16 keys), looked up one tile ahead like the box pages,
    // into slot j mod NSS of the scale ring.  The slot's previous tile,
    // j - NSS <= j - 1 - NSV, is done with it: before the loads of tile j the
    // producer waited for the release of V stage j - 1 - NSV, which follows
    // the PV of that tile, which follows its softmax's reads of the scales.
    auto ks_page_at = [&](int kt) -> int {
      if constexpr (Q8 && PAGED) {
        const int key0 = kt * kBlockN + 4 * lane;
        return (kt < pi.kt_hi && key0 < pi.sk) ? __ldg(bt + (key0 >> p.page_shift)) : 0;
      } else {
        return 0;
      }
    };
    auto load_scales = [&](int slot, int kt, int kpage) {
      const uint32_t dst = smem_u32(sKs + slot * kBlockN + 4 * lane);   // slot = tile j mod NSS
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int key = kt * kBlockN + 4 * lane + u;
        const bool live = key < pi.sk;
        int64_t tok;
        if constexpr (PAGED) tok = (int64_t)kpage * p.page_size + (key & (p.page_size - 1));
        else tok = (int64_t)pi.k_row0 + key;
        cp_async_4(dst + 4 * u, live ? p.k_scale + tok * p.hkv + pi.hk : p.k_scale, live ? 4u : 0u);
        if constexpr (PV8)
          cp_async_4(dst + 4 * u + Cfg::NSS * kBlockN * 4, live ? p.v_scale + tok * p.hkv + pi.hk : p.v_scale,
                     live ? 4u : 0u);
      }
      cp_async_arrive_noinc(smem_u32(ks_full + slot));
    };
    bool gathered = false;
    if constexpr (PAGED && !Q8) {
      if (p.gather) {
        // Pages of < 16 keys: every key row by its own page-table read and
        // 16-byte copies (fa_gather.cuh) into the layout a box would fill:
        // swizzled bf16 blocks, or staged byte rows for the converters.
        gathered = true;
        auto pages_of = [&](int kt, int (&pg)[4]) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int key = kt * kBlockN + lane + 32 * u;
            pg[u] = (kt < pi.kt_hi && key < pi.sk) ? __ldg(bt + (key >> p.page_shift)) : -1;
          }
        };
        // one slot in flight: with Dk 192 a tile has KC = 3 chunks in a
        // ring of NCK = 4, so the chunk slot the producer waits for frees
        // only after a QK that reads the chunk committed just before
        GatherPipe<1> gp;
        int pg[4], pgn[4];
        pages_of(first_kt, pg);
        int j = 0;
        bool ok = true;
        for (int kt = first_kt; ok && kt < pi.kt_hi; ++j) {
          const int kn = pair_next(p, pi, kt);
          pages_of(kn, pgn);
#pragma unroll 1
          for (int c = 0; c < KC; ++c) {
            const int n = j * KC + c, slot = n % NCK;
            if (lane == 0 && n >= NCK) ok = mbar_wait(smem_u32(kc_empty + slot), ((n / NCK) - 1) & 1, abort_flag, p.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            uint8_t *dst = sK + slot * Cfg::kChunkBytes;
            if constexpr (kStageK)
              gather_block<kBlockN, 64, kGatherStage>(dst, p.gk, pi.hk, kt * kBlockN, p.page_size - 1, c * 64, pg, lane);
            else
              gather_block<kBlockN, 128, kGatherSw128>(dst, p.gk, pi.hk, kt * kBlockN, p.page_size - 1, c * 128, pg,
                                                       lane);
            gp.commit(smem_u32(kStageK ? kc_stage + slot : kc_full + slot));
          }
          if (!ok) break;
          const int sv = j % NSV;
          if (lane == 0 && j >= NSV) ok = mbar_wait(smem_u32(v_empty + sv), ((j / NSV) - 1) & 1, abort_flag, p.err);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
#pragma unroll
          for (int c = 0; c < VC; ++c) {
            uint8_t *dst = sV + sv * Cfg::kVBytes + c * Cfg::kChunkBytes;
            if constexpr (FP8)
              gather_block<kBlockN, 64, kGatherStage>(dst, p.gv, pi.hk, kt * kBlockN, p.page_size - 1, c * 64, pg, lane);
            else
              gather_block<kBlockN, 128, kGatherSw128>(dst, p.gv, pi.hk, kt * kBlockN, p.page_size - 1, c * 128, pg,
                                                       lane);
          }
          gp.commit(smem_u32(FP8 ? v_stage + sv : v_full + sv));
          kt = kn;
#pragma unroll
          for (int u = 0; u < 4; ++u) pg[u] = pgn[u];
        }
        gp.drain();
      }
    }
    int j = 0;
    bool ok = !gathered;
    int page = gathered ? -1 : page_at(first_kt);
    int kpage = ks_page_at(first_kt);
    for (int kt = first_kt; ok && kt < pi.kt_hi; ++j) {
      const int kn = pair_next(p, pi, kt);
      const int page_next = page_at(kn);
      const int kpage_next = ks_page_at(kn);
#pragma unroll 1
      for (int c = 0; c < KC; ++c) {
        const int n = j * KC + c, slot = n % NCK;
        uint64_t *bar = kStageK ? kc_stage + slot : kc_full + slot;
        if (lane == 0) {
          if (n >= NCK) ok = mbar_wait(smem_u32(kc_empty + slot), ((n / NCK) - 1) & 1, abort_flag, p.err);
          if (ok) mbar_expect_tx(smem_u32(bar), kKBlockBytes);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        load_block(&tm_k, sK + slot * Cfg::kChunkBytes, bar, c * (Q8 ? 128 : 64), kt, page, kStageK, false);
        if constexpr (Q8) {
          if (c == 0) load_scales(j % Cfg::NSS, kt, kpage);
        }
      }
      if (!ok) break;
      const int sv = j % NSV;
      uint64_t *vbar = FP8 ? v_stage + sv : v_full + sv;
      if (lane == 0) {
        if (j >= NSV) ok = mbar_wait(smem_u32(v_empty + sv), ((j / NSV) - 1) & 1, abort_flag, p.err);
        if (ok) mbar_expect_tx(smem_u32(vbar), VC * kVBlockBytes);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
#pragma unroll
      for (int c = 0; c < VC; ++c)
        load_block(&tm_v, sV + sv * Cfg::kVBytes + (PV8 ? Cfg::kChunkBytes + c * kBlockN * 64 : c * Cfg::kChunkBytes),
                   vbar, c * 64, kt, page, FP8, true);
      kt = kn;
      page = page_next;
      kpage = kpage_next;
    }
    // Q8: no scale copy may still be in flight when the CTA ends (error exits).
    if constexpr (Q8) asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == 9) {
    // ------------------------------------------------------- MMA issuer --
    // Q8: kind::f8f6f4 with A = B = e4m3 (format code 0 in the A and B fields,
    // as f16 is for kind::f16) and an fp32 accumulator: the same word.
    constexpr uint32_t idesc_qk = FP8 ? idesc_f16_f32(kBlockM, kBlockN, 0, 0) : idesc_bf16_f32(kBlockM, kBlockN, 0, 0);
    constexpr uint32_t idesc_pv = FP8 ? idesc_f16_f32(kBlockM, DV, 0, 1) : idesc_bf16_f32(kBlockM, DV, 0, 1);
    const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
    int n_pv[2] = {0, 0};
    bool ok = mbar_wait(smem_u32(q_full), 0, abort_flag, p.err);
    bool q_ready[2] = {!FP8 || Q8, !FP8 || Q8};   // converted Q (e4m3 / int8 caches with bf16 Q)

    // Descriptor words, computed once.  K-major 128-byte-swizzled operands
    // step 32 bytes per K slice (16 two-byte or 32 one-byte columns) inside a
    // 128-byte block; a Q tile's blocks
    // are 16 KB apart and each K block sits in its own ring chunk.  V
    // (MN-major) has its two 64-column blocks 16 KB apart and steps 16 rows.
    const uint64_t dq0 = smem_desc_sw128(sQa, 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(sKa, 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(sVa, Cfg::kChunkBytes, 1024);
    const uint32_t q_lo = (uint32_t)dq0, k_lo = (uint32_t)dk0, qk_hi = (uint32_t)(dq0 >> 32);
    const uint32_t v_lo = (uint32_t)dv0, v_hi = (uint32_t)(dv0 >> 32);
    // QK_X of the j-th tile.  `first`: wait for each chunk to be filled;
    // `last`: release each chunk once this QK has read it.
    auto qk = [&](int X, int j, bool first, bool last) -> bool {
      if (!q_ready[X]) {
        if (!mbar_wait(smem_u32(q_conv + X), 0, abort_flag, p.err)) return false;
        q_ready[X] = true;
      }
      const uint32_t d = tmem + (X ? 128u : 0u);
      const uint32_t a0 = q_lo + (uint32_t)(X * (Cfg::kQTileBytes >> 4));
#pragma unroll
      for (int c = 0; c < KC; ++c) {
        const int n = j * KC + c, slot = n % NCK;
        if (first) {
          if (!mbar_wait(smem_u32(kc_full + slot), (n / NCK) & 1, abort_flag, p.err)) return false;
          tc_fence_after();
        }
        const uint32_t a = a0 + (uint32_t)(c * ((kBlockM * 128) >> 4));
        const uint32_t b = k_lo + (uint32_t)(slot * (Cfg::kChunkBytes >> 4));
        // Q8 at Dk 192: the second chunk's columns 192..255 are zeros
        const int n_ks = Q8 ? min(4, (DK - 128 * c) / 32) : 4;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          if (ks >= n_ks) break;
          if constexpr (Q8) {
            if (c == 0 && ks == 0) mma_ss_f8_w<0>(d, a, qk_hi, b, qk_hi, idesc_qk);
            else mma_ss_f8_w<1>(d, a + 2 * ks, qk_hi, b + 2 * ks, qk_hi, idesc_qk);
          } else {
            if (c == 0 && ks == 0) mma_ss_w<0>(d, a, qk_hi, b, qk_hi, idesc_qk);
            else mma_ss_w<1>(d, a + 2 * ks, qk_hi, b + 2 * ks, qk_hi, idesc_qk);
          }
        }
        if (last) tc_commit(smem_u32(kc_empty + slot));
      }
      tc_commit(smem_u32(s_full + X));
      return true;
    };
    // PV8: A = the e4m3 P tile X, B = the transposed e4m3 V tile, both
    // K-major and 128-byte swizzled like the Q8 QK's operands (the same
    // descriptor high word), kind::f8f6f4 with K = 32 keys per instruction.
    constexpr uint32_t idesc_pv8 = idesc_f16_f32(kBlockM, DV, 0, 0);
    const uint32_t p8_lo = (uint32_t)smem_desc_sw128(smem_u32(sP), 16, 1024);
    const uint32_t vt_lo = (uint32_t)smem_desc_sw128(sVa, 16, 1024);
    auto pv = [&](int X, int sv) {
      const uint32_t d = tmem + 256u + (X ? 128u : 0u);
      if constexpr (PV8) {
        const uint32_t a = p8_lo + (uint32_t)(X * ((kBlockM * 128) >> 4));
        const uint32_t b = vt_lo + (uint32_t)(sv * (Cfg::kVBytes >> 4));
#pragma unroll
        for (int ks = 0; ks < kBlockN / 32; ++ks) {
          if (ks == 0 && n_pv[X] == 0) mma_ss_f8_w<0>(d, a, qk_hi, b, qk_hi, idesc_pv8);
          else mma_ss_f8_w<1>(d, a + 2 * ks, qk_hi, b + 2 * ks, qk_hi, idesc_pv8);
        }
      } else {
        const uint32_t a = tmem + (X ? 128u : 0u);                 // P_X aliases S_X
        uint32_t b = v_lo + (uint32_t)(sv * (Cfg::kVBytes >> 4));
        const uint32_t acc0 = n_pv[X] > 0 ? 1u : 0u;
#pragma unroll
        for (int ks = 0; ks < kBlockN / 16; ++ks) {
          mma_ts_w(d, a + ks * 8, b, v_hi, idesc_pv, ks > 0 ? 1u : acc0);
          b += (16 * 128) >> 4;
        }
      }
      tc_commit(smem_u32(o_done + X));
    };

    if (lane == 0 && ok) {
      bool a0 = half_active(p, pi, 0, first_kt), a1 = half_active(p, pi, 1, first_kt);
      if (a0) ok = qk(0, 0, true, !a1);
      if (ok && a1) ok = qk(1, 0, !a0, true);
      int j = 0;
      for (int kt = first_kt; ok && kt < pi.kt_hi; ++j) {
        const int kn = pair_next(p, pi, kt);
        const bool more = kn < pi.kt_hi;
        const bool n0 = more && half_active(p, pi, 0, kn);
        const bool n1 = more && half_active(p, pi, 1, kn);
        const int sv = j % NSV;
        if (!(ok = mbar_wait(smem_u32(v_full + sv), (j / NSV) & 1, abort_flag, p.err))) break;
        if (a0) {
          if (!(ok = mbar_wait(smem_u32(p_full + 0), n_pv[0] & 1, abort_flag, p.err))) break;
          tc_fence_after();
          pv(0, sv);
          ++n_pv[0];
        }
        if (n0 && !(ok = qk(0, j + 1, true, !n1))) break;
        if (a1) {
          if (!(ok = mbar_wait(smem_u32(p_full + 1), n_pv[1] & 1, abort_flag, p.err))) break;
          tc_fence_after();
          pv(1, sv);
          ++n_pv[1];
        }
        tc_commit(smem_u32(v_empty + sv));
        if (n1 && !(ok = qk(1, j + 1, !n0, true))) break;
        a0 = n0;
        a1 = n1;
        kt = kn;
      }
    }
  } else if (warp >= 10) {
    if constexpr (FP8) {
      // ----------------------------------------- e4m3 -> f16 converters --
      // Slice g (32 rows of one 64-column block; K blocks of a tile first --
      // none with Q8 -- then V blocks; g counts slices over the pair's tile list) goes to warp
      // g mod 6.  Lane l handles the scale of row l; each step converts 8
      // rows, 16 dims per lane, into the swizzled layout.  Rows past the
      // sequence end are written as zeros.  The scale loads are software
      // pipelined: the page of a slice two ahead and the scale of the next
      // slice are in flight while the current slice is converted.
      constexpr int S = Cfg::kSlicesPerTile;
      static_assert(S >= Cfg::kConverters, "a warp's first slice lies in the first tile");
      const int cw = warp - 10;
      struct It { int g, j, kt; };
      auto adv = [&](It &it) {
        it.g += Cfg::kConverters;
        const int jn = it.g / S;
        while (it.j < jn && it.kt < pi.kt_hi) { it.kt = pair_next(p, pi, it.kt); ++it.j; }
      };
      auto key_of = [&](const It &it) { return it.kt * kBlockN + ((it.g % S) & 3) * 32 + lane; };
      auto page_of = [&](const It &it) -> int {
        if constexpr (PAGED && !PV8) {
          const int key = key_of(it);
          return (it.kt < pi.kt_hi && key < pi.sk) ? __ldg(bt + (key >> p.page_shift)) : 0;
        } else {
          return 0;
        }
      };
      auto scale_of = [&](const It &it, int page) -> float {
        if constexpr (PV8) return 0.f;   // the V scales go into P
        const int key = key_of(it);
        if (!(it.kt < pi.kt_hi && key < pi.sk)) return 0.f;
        int64_t tok;
        if constexpr (PAGED) tok = (int64_t)page * p.page_size + (key & (p.page_size - 1));
        else tok = (int64_t)pi.k_row0 + key;
        const bool isv = (it.g % S) >= Cfg::kKSlices;
        return __ldg((isv ? p.v_scale : p.k_scale) + tok * p.hkv + pi.hk);
      };
      It a{cw, 0, first_kt};
      It b = a;
      adv(b);
      It c = b;
      adv(c);
      float sa = scale_of(a, page_of(a));
      int pb = page_of(b);
      bool ok = true;
      while (ok && a.kt < pi.kt_hi) {
        const float sb = scale_of(b, pb);
        const int pc = page_of(c);
        const int s = a.g % S, j = a.j, kt = a.kt;
        const bool isv = s >= Cfg::kKSlices;
        const int cb = isv ? (s - Cfg::kKSlices) >> 2 : s >> 2, q = s & 3;
        uint8_t *base;
        uint64_t *stage_bar, *full_bar;
        uint32_t par;
        if (!isv) {
          const int n = j * KC + cb, slot = n % NCK;
          base = sK + slot * Cfg::kChunkBytes;
          stage_bar = kc_stage + slot;
          full_bar = kc_full + slot;
          par = (n / NCK) & 1;
        } else {
          const int sv = j % NSV;
          base = sV + sv * Cfg::kVBytes + cb * Cfg::kChunkBytes;
          stage_bar = v_stage + sv;
          full_bar = v_full + sv;
          par = (j / NSV) & 1;
        }
        ok = mbar_wait(smem_u32(stage_bar), par, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const uint8_t *stg = base + q * 4096 + 2048;
        // e4m3 or int8 bytes times the row's scale -> one 16-byte f16 chunk
        auto conv16 = [&](uint32_t w0, uint32_t w1, float s, uint32_t (&o)[4]) {
          if constexpr (I8) {
            i8x4_scaled_f16(w0, s, o[0], o[1]);
            i8x4_scaled_f16(w1, s, o[2], o[3]);
          } else {
            e4m3x4_scaled_f16(w0, s, o[0], o[1]);
            e4m3x4_scaled_f16(w1, s, o[2], o[3]);
          }
        };
        if constexpr (PV8) {
          // e4m3 P * V: V becomes the K-major operand V^T [128 dims][128 keys]
          // (128-byte swizzled, like a Q8 key tile) in the stage's lower half,
          // its bytes unscaled (the V scales go into P).  The slice -- keys
          // q*32 .. +31 of dims cb*64 .. +63, staged [key][64 bytes] in the
          // upper half -- is 4 x 8 blocks of 8 x 8 bytes: lane (key group kg,
          // dim group dg) transposes one and writes 8 dims' rows of 8 keys.
          // Keys past the sequence end become zeros (their bytes may be
          // anything, and 0 * NaN would be NaN).
          uint8_t *vt = sV + (j % NSV) * Cfg::kVBytes;
          const uint8_t *src = vt + Cfg::kChunkBytes + cb * (kBlockN * 64) + q * 32 * 64;
          const int kg = lane >> 3, dg = lane & 7;
          uint2 in[8], tr[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) in[k] = *reinterpret_cast<const uint2 *>(src + (kg * 8 + k) * 64 + dg * 8);
          transpose_8x8_bytes(in, tr);
          const int nlive = min(max(pi.sk - (kt * kBlockN + q * 32 + kg * 8), 0), 8);
          const uint32_t mlo = nlive >= 4 ? 0xFFFFFFFFu : (uint32_t)((1ull << (8 * nlive)) - 1);
          const uint32_t mhi = nlive >= 8 ? 0xFFFFFFFFu : (nlive <= 4 ? 0u : (uint32_t)((1ull << (8 * (nlive - 4))) - 1));
          const int kb = q * 32 + kg * 8;   // the 8 keys' first byte in a 128-byte row
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const int d = cb * 64 + dg * 8 + t;
            *reinterpret_cast<uint2 *>(vt + d * 128 + ((((kb >> 4) ^ (d & 7))) << 4) + (kb & 15)) =
                make_uint2(tr[t].x & mlo, tr[t].y & mhi);
          }
        } else {
        const int part = lane & 3;
        // one staged row piece (16 bytes, row rr of the slice) -> 16 f16
        // values of row q * 32 + rr, zeros past the sequence end
        auto put_row = [&](const uint4 raw, int rr) {
          const float s_row = __shfl_sync(0xffffffffu, sa, rr);
          const bool live = kt * kBlockN + q * 32 + rr < pi.sk;
          uint32_t o[8];
          conv16(raw.x, raw.y, s_row, *reinterpret_cast<uint32_t(*)[4]>(o));
          conv16(raw.z, raw.w, s_row, *reinterpret_cast<uint32_t(*)[4]>(o + 4));
          if (!live) {
#pragma unroll
            for (int k = 0; k < 8; ++k) o[k] = 0u;
          }
          const int r = q * 32 + rr;
          uint8_t *row = base + r * 128;
          *reinterpret_cast<uint4 *>(row + (((2 * part) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4 *>(row + (((2 * part + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
        };
        if constexpr (!V5) {
          // Token rows of 64 bytes, read and written step by step: the
          // staging rows a step overwrites were read in earlier steps.
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int rr = 8 * t + (lane >> 2);              // row within the slice
            put_row(*reinterpret_cast<const uint4 *>(stg + rr * 64 + part * 16), rr);
          }
        } else if (isv) {
          // 5-D V: the slice's staging is [2 groups of 16 tokens][64 dims]
          // [16 bytes].  Lane (g, octet oc, half th) takes tokens 16g + 8th
          // .. +7 of dims 8oc .. 8oc+7, transposes the 8 x 8 bytes and writes
          // 8 row chunks; every lane reads before any lane writes (the
          // staging lies in the upper half of the output).
          const int g = lane >> 4, oc = (lane >> 1) & 7, th = lane & 1;
          uint2 in[8], tr[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            in[k] = *reinterpret_cast<const uint2 *>(stg + g * 1024 + (8 * oc + k) * 16 + 8 * th);
          __syncwarp();
          transpose_8x8_bytes(in, tr);
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const int rr = 16 * g + 8 * th + t;            // row within the slice
            const float s_row = __shfl_sync(0xffffffffu, sa, rr);
            const bool live = kt * kBlockN + q * 32 + rr < pi.sk;
            uint32_t o[4];
            conv16(tr[t].x, tr[t].y, s_row, o);
            if (!live) o[0] = o[1] = o[2] = o[3] = 0u;
            const int r = q * 32 + rr;
            *reinterpret_cast<uint4 *>(base + r * 128 + ((oc ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        } else {
          // 5-D K: a box of R = rows_per_box rows (a power of two) lands as
          // [4 column groups][R rows][16 bytes], which spreads a row's bytes
          // over the whole staging half, so every lane reads its four pieces
          // before the warp writes any.
          const int R = p.rows_per_box, lg = __ffs(R) - 1;
          uint4 raw[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int rr = 8 * t + (lane >> 2);
            raw[t] = *reinterpret_cast<const uint4 *>(stg + ((rr >> lg) << (6 + lg)) + (part << (4 + lg)) +
                                                      ((rr & (R - 1)) << 4));
          }
          __syncwarp();
#pragma unroll
          for (int t = 0; t < 4; ++t) put_row(raw[t], 8 * t + (lane >> 2));
        }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(full_bar));
        a = b;
        sa = sb;
        b = c;
        pb = pc;
        adv(c);
      }
    }
  } else {
    // ---------------------------------------------------------- softmax --
    if constexpr (Cfg::kSplitRegs) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::kRegsSoftmax));
    const int X = warp >> 2;                  // 0: tile A, 1: tile B
    const int r = threadIdx.x & 127;          // row in the tile == TMEM lane
    const Half hx = X ? pi.x[1] : pi.x[0];
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t colS = X ? 128u : 0u, colO = 256u + (X ? 128u : 0u);
    const int i = hx.q0 + r;
    const int ip = i + pi.sk - pi.sq;
    // Prologue terms (see PrefillParams; kernels with KT only): the row term
    // enters the scores under the soft-cap; the per-key term of a Q add, when
    // present, is read per 32-key chunk (all lanes read the same addresses;
    // the address is formed from the parameter block there, so nothing stays
    // live).
    const float row_term =
        (KT && MK == 2 && i < pi.sq) ? softcap_row_term<DK>(p, (int64_t)pi.q_row0 + X * kBlockM + r, pi.h) : 0.f;
    float m_ref = -INFINITY, l = 0.f;
    int cnt = 0;
    bool ok = true;
    // Row factor of the f16 Q row (e4m3 caches): S carries 2^e, undone here.
    float rowf = 1.f;
    if constexpr (FP8 && !Q8) {
      ok = mbar_wait(smem_u32(q_full), 0, abort_flag, p.err);
      if (ok) {
        // Row r owns 128 bytes of each 64-column block; its 16-byte units are
        // visited from unit r mod 8 on, so a warp's accesses spread over all banks.
        uint8_t *qrow = sQ + X * Cfg::kQTileBytes + r * 128;
        float amax = 0.f;
#pragma unroll
        for (int cb = 0; cb < KC; ++cb)
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 w = *reinterpret_cast<const uint4 *>(qrow + cb * kBlockM * 128 + ((u + r) & 7) * 16);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
              amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(ww[k] << 16)), fabsf(__uint_as_float(ww[k] & 0xFFFF0000u))));
          }
        int sh = 0;
        if (amax > 0.f && amax <= 3.0e38f) {
          const int E = (int)((__float_as_uint(amax) >> 23) & 0xFF);
          sh = min(141 - E, 126);               // amax * 2^sh in [2^14, 2^15)
        }
        const float up = __uint_as_float((uint32_t)(sh + 127) << 23);
        rowf = __uint_as_float((uint32_t)(127 - sh) << 23);
#pragma unroll
        for (int cb = 0; cb < KC; ++cb)
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            uint4 *ptr = reinterpret_cast<uint4 *>(qrow + cb * kBlockM * 128 + ((u + r) & 7) * 16);
            const uint4 w = *ptr;
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
            uint32_t hh[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
              hh[k] = pack_f16x2(__uint_as_float(ww[k] << 16) * up, __uint_as_float(ww[k] & 0xFFFF0000u) * up);
            *ptr = make_uint4(hh[0], hh[1], hh[2], hh[3]);
          }
        fence_proxy_async_smem();
      }
      mbar_arrive(smem_u32(q_conv + X));
    }
    // PV8 (P8 below): the weights go to e4m3 as p * v_scale * 2^-pexp, with
    // 2^pexp above the largest V scale of the sequence (a pre-pass writes
    // that maximum), so that with the max taken first (p <= 2^8) every
    // weight stays below 2^8, inside the e4m3 range (448).  The factor is
    // folded into the exponent's reference (p' = 2^(x - m - pexp)): the row
    // sum then carries it too, O / l needs no correction, and the LSE adds
    // pexp back.
    int pexp = 0;
    if constexpr (PV8) {
      const float vmax = __ldg(p.pv_vmax + (int64_t)pi.b * p.hkv + pi.hk);
      if (vmax > 0.f && vmax <= 3.0e38f) pexp = (int)((__float_as_uint(vmax) >> 23) & 0xFF) - 126;
    }
    const float mshift = (float)pexp;
    // MOD 0 runs with a positive scale only (the host routes other scales to
    // the general path), so raw scores can be maxed before scaling.
    constexpr bool fast = (MK == 0);
    // Deferred-max guard on a tile's row sum: P must stay finite in its
    // packed type (f16 for e4m3 caches: below 65504; bf16: any fp32 value).
    constexpr float kGuard = FP8 ? 0x1p15f : kGuardSum;
    static_assert(!PV8 || !Cfg::kOnePass, "e4m3 P: the two-half softmax");
    const float sl2 = p.scale_log2 * rowf;
    const float c2u = 2.f * kLog2e * p.softcap_arg * rowf;   // soft-cap: raw score -> 2u log2(e)
    auto pack_p = [](float a, float b) -> uint32_t { return FP8 ? pack_f16x2(a, b) : pack_bf16x2(a, b); };
    auto unpack_p = [](uint32_t w, float &a, float &b) {
      if constexpr (FP8) {
        unpack_f16x2(w, a, b);
      } else {
        a = __uint_as_float(w << 16);
        b = __uint_as_float(w & 0xFFFF0000u);
      }
    };
    auto chunk_exp = [&](const float (&v)[32], float c, float m, uint32_t (&pk)[16], float (&acc)[4]) {
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float t0, t1;
        fma2(t0, t1, v[e], v[e + 1], c, -m);
        const float a0 = ex2(t0), a1 = ex2(t1);
        const int q = ((e >> 1) & 1) * 2;
        add2(acc[q], acc[q + 1], a0, a1);
        pk[e >> 1] = pack_p(a0, a1);
      }
    };
    const float cexp = fast ? sl2 : 1.f;
    constexpr bool kDeferredMax = (MK == 2) && !PV8;   // soft-cap only, as in fa_prefill2.cuh
    // PV8: row r of the e4m3 P tile, 128 keys in eight 16-byte chunks,
    // 128-byte swizzled (the K-major A operand of the e4m3 PV)
    uint8_t *prow = sP + X * (kBlockM * 128) + r * 128;
    // 32 weights of keys jc .. jc+31 (relative to the tile start: kr) times
    // their V scales, to e4m3, into P row r
    auto store_p8 = [&](const float (&w)[32], int kr, const float *vs) {
      uint32_t b[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 s4 = *reinterpret_cast<const float4 *>(vs + kr + 4 * k);
        b[k] = pack_e4m3x4(w[4 * k] * s4.x, w[4 * k + 1] * s4.y, w[4 * k + 2] * s4.z, w[4 * k + 3] * s4.w);
      }
      const int c0 = kr >> 4;
      *reinterpret_cast<uint4 *>(prow + (((c0) ^ (r & 7)) << 4)) = make_uint4(b[0], b[1], b[2], b[3]);
      *reinterpret_cast<uint4 *>(prow + (((c0 + 1) ^ (r & 7)) << 4)) = make_uint4(b[4], b[5], b[6], b[7]);
    };
    int j = -1;   // index of the tile in the pair's list (ring position)
    for (int kt = first_kt; ok && kt < pi.kt_hi; kt = pair_next(p, pi, kt)) {
      ++j;
      if (!half_active_h(p, pi, hx, kt)) continue;
      ok = mbar_wait(smem_u32(s_full + X), cnt & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sa = tmem + lane_base + colS;
      // Q8: the tile's K scales, slot j mod NSS of their ring.
      const float *ks_tile = sKs + (j % Cfg::NSS) * kBlockN;
      if constexpr (Q8) {
        ok = mbar_wait(smem_u32(ks_full + j % Cfg::NSS), (j / Cfg::NSS) & 1, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
      const int j0 = kt * kBlockN;
      bool need_mask = (j0 + kBlockN > pi.sk);
      if (p.causal && j0 + kBlockN - 1 > hx.ip_min) need_mask = true;
      if (p.window > 0) {
        if (j0 < hx.ip_max - p.window + 1) need_mask = true;
        if (!p.causal && j0 + kBlockN - 1 > hx.ip_min + p.window - 1) need_mask = true;
      }
      auto scores = [&](float (&v)[32], int jc) {
        if constexpr (Q8) {
          const float4 *kp = reinterpret_cast<const float4 *>(ks_tile + (jc - j0));
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 s4 = kp[e >> 2];
            mul2(v[e], v[e + 1], s4.x, s4.y);
            mul2(v[e + 2], v[e + 3], s4.z, s4.w);
          }
        }
        if (!fast) {
          const float dbase = (float)(ip - jc);   // ALiBi: |i' - j| = |dbase - e|, exact in fp32
          if constexpr (KT) {
            // scaled score (log2 units; soft-cap: its argument 2u log2(e))
            // plus the row term (soft-cap) and the key's term; no term is
            // read past cb_ld (the pre-pass flags such keys)
            const float lin = MK == 2 ? c2u : sl2;
            const bool in_ld = p.col_bias != nullptr && jc + 32 <= p.cb_ld;
            const float4 *c4 =
                reinterpret_cast<const float4 *>(p.col_bias + ((int64_t)pi.b * p.hkv + pi.hk) * p.cb_ld + jc);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 c = in_ld ? c4[e >> 2] : make_float4(0.f, 0.f, 0.f, 0.f);
              v[e] = fmaf(v[e], lin, c.x + row_term);
              v[e + 1] = fmaf(v[e + 1], lin, c.y + row_term);
              v[e + 2] = fmaf(v[e + 2], lin, c.z + row_term);
              v[e + 3] = fmaf(v[e + 3], lin, c.w + row_term);
            }
          }
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float x;
            if constexpr (KT) {
              x = v[e];
            } else if constexpr (MK == 2) {
              x = v[e] * c2u;
            } else {
              x = v[e] * sl2;
            }
            if constexpr (MK == 2) {
              float r;
              x = softcap_log2_score(ex2(x), p.softcap_log2, r);
            }
            if constexpr (MK == 1) x -= p.alibi_log2 * fabsf(dbase - (float)e);
            v[e] = x;
          }
        }
        if (need_mask) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int jj = jc + e;
            bool allowed = jj < pi.sk;
            if (p.causal) allowed = allowed && (jj <= ip);
            if (p.window > 0) allowed = allowed && (p.causal ? (ip - jj < p.window) : (abs(ip - jj) < p.window));
            v[e] = allowed ? v[e] : -INFINITY;
          }
        }
      };
      float alpha_tile = 1.f;
      bool warp_need = false;
      float sum[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (Cfg::kOnePass) {
        float sv[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(sa + c * 32, sv[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) scores(sv[c], j0 + c * 32);
        auto exp_store = [&](float m_use, float (&acc)[4]) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
            chunk_exp(sv[c], cexp, m_use, pk, acc);
            tmem_st16(sa + c * 16, pk);
          }
        };
        // Deferred max (as in fa_prefill2.cuh): exponentials against the
        // running reference unless the row has none yet or the tile's sum
        // exceeds kGuard, in which case the max is taken and P redone.
        bool slow = !kDeferredMax || __any_sync(0xffffffffu, m_ref == -INFINITY);
        if (!slow) {
          exp_store(m_ref, sum);
          const float ts = (sum[0] + sum[1]) + (sum[2] + sum[3]);
          slow = __any_sync(0xffffffffu, !(ts <= kGuard));
          if (slow) {
            tmem_wait_st();
            sum[0] = sum[1] = sum[2] = sum[3] = 0.f;
          }
        }
        if (slow) {
          float t1[43];
#pragma unroll
          for (int k = 0; k < 42; ++k) {
            const int e = 3 * k;
            t1[k] = max3(sv[e >> 5][e & 31], sv[(e + 1) >> 5][(e + 1) & 31], sv[(e + 2) >> 5][(e + 2) & 31]);
          }
          t1[42] = fmaxf(sv[3][30], sv[3][31]);
          float t2[15];
#pragma unroll
          for (int k = 0; k < 14; ++k) t2[k] = max3(t1[3 * k], t1[3 * k + 1], t1[3 * k + 2]);
          t2[14] = t1[42];
          float t3[5];
#pragma unroll
          for (int k = 0; k < 5; ++k) t3[k] = max3(t2[3 * k], t2[3 * k + 1], t2[3 * k + 2]);
          float tmax = fmaxf(max3(t3[0], t3[1], t3[2]), fmaxf(t3[3], t3[4]));
          if (fast && tmax != -INFINITY) tmax *= sl2;
          const float m_new = fmaxf(m_ref, tmax);
          const bool need = m_new > m_ref + kRescaleThreshold;
          warp_need = __any_sync(0xffffffffu, need);
          if (need) {
            alpha_tile = ex2(m_ref - m_new);
            l *= alpha_tile;
            m_ref = m_new;
          }
          exp_store((m_ref == -INFINITY) ? 0.f : m_ref, sum);
        }
      } else {
        // Two halves of 64 columns with the deferred max of the one-pass form;
        // when the second half moves the reference, the first half's P
        // (already in TMEM) is rescaled too.
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          float sv[2][32];
          tmem_ld32(sa + hf * 64, sv[0]);
          tmem_ld32(sa + hf * 64 + 32, sv[1]);
          tmem_wait_ld();
          scores(sv[0], j0 + hf * 64);
          scores(sv[1], j0 + hf * 64 + 32);
          float hsum[4] = {0.f, 0.f, 0.f, 0.f};
          auto exp_store = [&](float m_use) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              if constexpr (PV8) {
                float w[32];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                  float t0, t1;
                  fma2(t0, t1, sv[c][e], sv[c][e + 1], cexp, -(m_use + mshift));
                  w[e] = ex2(t0);
                  w[e + 1] = ex2(t1);
                  const int qq = ((e >> 1) & 1) * 2;
                  add2(hsum[qq], hsum[qq + 1], w[e], w[e + 1]);
                }
                store_p8(w, hf * 64 + c * 32, sVs + (j % Cfg::NSS) * kBlockN);
              } else {
                uint32_t pk[16];
                chunk_exp(sv[c], cexp, m_use, pk, hsum);
                tmem_st16(sa + hf * 32 + c * 16, pk);
              }
            }
          };
          bool slow = !kDeferredMax || __any_sync(0xffffffffu, m_ref == -INFINITY);
          if (!slow) {
            exp_store(m_ref);
            const float hs = (hsum[0] + hsum[1]) + (hsum[2] + hsum[3]);
            slow = __any_sync(0xffffffffu, !(hs <= kGuard));
            if (slow) {
              tmem_wait_st();
              hsum[0] = hsum[1] = hsum[2] = hsum[3] = 0.f;
            }
          }
          if (slow) {
            float t1[22];
#pragma unroll
            for (int k = 0; k < 21; ++k) {
              const int e = 3 * k;
              t1[k] = max3(sv[e >> 5][e & 31], sv[(e + 1) >> 5][(e + 1) & 31], sv[(e + 2) >> 5][(e + 2) & 31]);
            }
            t1[21] = sv[1][31];
            float t2[8];
#pragma unroll
            for (int k = 0; k < 7; ++k) t2[k] = max3(t1[3 * k], t1[3 * k + 1], t1[3 * k + 2]);
            t2[7] = t1[21];
            float hmax = fmaxf(max3(t2[0], t2[1], t2[2]), fmaxf(max3(t2[3], t2[4], t2[5]), fmaxf(t2[6], t2[7])));
            if (fast && hmax != -INFINITY) hmax *= sl2;
            const float m_new = fmaxf(m_ref, hmax);
            const bool need = m_new > m_ref + kRescaleThreshold;
            const bool wneed = __any_sync(0xffffffffu, need);
            if (wneed) {
              const float alpha = need ? ex2(m_ref - m_new) : 1.f;
              if (need) {
                m_ref = m_new;
                l *= alpha;
                sum[0] *= alpha;
                sum[1] *= alpha;
                sum[2] *= alpha;
                sum[3] *= alpha;
              }
              alpha_tile *= alpha;
              warp_need = true;
              if (hf == 1) {
                if constexpr (PV8) {
                  // the first half's e4m3 weights, rescaled in place (a
                  // second rounding, on a rare event that shrinks them by
                  // at least 2^-8)
#pragma unroll
                  for (int c = 0; c < 4; ++c) {
                    uint4 *ptr = reinterpret_cast<uint4 *>(prow + ((c ^ (r & 7)) << 4));
                    const uint4 u = *ptr;
                    const uint32_t uu[4] = {u.x, u.y, u.z, u.w};
                    uint32_t o[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                      float f0, f1, f2, f3;
                      unpack_e4m3x4(uu[k], f0, f1, f2, f3);
                      o[k] = pack_e4m3x4(f0 * alpha, f1 * alpha, f2 * alpha, f3 * alpha);
                    }
                    *ptr = make_uint4(o[0], o[1], o[2], o[3]);
                  }
                } else {
                tmem_wait_st();
                float pw[32];
                tmem_ld32(sa, pw);
                tmem_wait_ld();
                uint32_t w[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                  const uint32_t u = __float_as_uint(pw[e]);
                  float lo, hi;
                  unpack_p(u, lo, hi);
                  w[e] = pack_p(lo * alpha, hi * alpha);
                }
                tmem_st32(sa, w);
                }
              }
            }
            exp_store((m_ref == -INFINITY) ? 0.f : m_ref);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) sum[q] += hsum[q];
        }
      }
      const float alpha = alpha_tile;
      l += (sum[0] + sum[1]) + (sum[2] + sum[3]);
      if (warp_need && cnt > 0) {
        ok = mbar_wait(smem_u32(o_done + X), (cnt - 1) & 1, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const uint32_t oa = tmem + lane_base + colO;
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          float o[32];
          tmem_ld32(oa + c * 32, o);
          tmem_wait_ld();
          uint32_t w[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(o[e] * alpha);
          tmem_st32(oa + c * 32, w);
        }
      }
      if constexpr (!FP8) {
        // bf16 keys past the sequence end may hold anything (NaN-poisoned
        // page slots): their V rows are cleared before P is released, by
        // warpgroup A, or by B when A skips the tile.  (The e4m3 converters
        // write those rows as zeros.)
        const int valid = pi.sk - j0;
        if (valid < kBlockN && (X == 0 || !half_active(p, pi, 0, kt))) {
          const int sv = j % NSV;
          ok = mbar_wait(smem_u32(v_full + sv), (j / NSV) & 1, abort_flag, p.err);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          uint8_t *vt = sV + sv * Cfg::kVBytes;
          const int per_cb = (kBlockN - valid) * 8;
          for (int idx = r; idx < per_cb * VC; idx += kBlockM) {
            const int cb = idx / per_cb, rem = idx - cb * per_cb;
            *reinterpret_cast<uint4 *>(vt + cb * Cfg::kChunkBytes + valid * 128 + rem * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
      }
      if constexpr (PV8) fence_proxy_async_smem();   // P8 for the tensor core
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(p_full + X));
      ++cnt;
    }

    // -------------------------------------------------------- epilogue --
    if (hx.valid) {
      const bool row_ok = i < pi.sq;
      const int64_t t = (int64_t)pi.q_row0 + X * kBlockM + r;
      __nv_bfloat16 *orow = p.out + t * p.out_stride_t + (int64_t)pi.h * p.out_stride_h;
      if (cnt == 0) {
        if (row_ok && ok) {
          for (int d = 0; d < DV; d += 8) *reinterpret_cast<uint4 *>(orow + d) = make_uint4(0, 0, 0, 0);
          if (p.lse) p.lse[(int64_t)pi.h * p.total_q + t] = -INFINITY;
        }
      } else if (ok) {
        ok = mbar_wait(smem_u32(o_done + X), (cnt - 1) & 1, abort_flag, p.err);
        if (__all_sync(0xffffffffu, ok)) {
          tc_fence_after();
          const bool has = l > 0.f;
          const float inv_l = has ? 1.f / l : 0.f;
          const float sc = inv_l * p.pro_vmul;   // prologue's V map folded into the normalisation
          const uint32_t oa = tmem + lane_base + colO;
#pragma unroll
          for (int c = 0; c < DV / 32; ++c) {
            float o[32];
            tmem_ld32(oa + c * 32, o);
            tmem_wait_ld();
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[e] = has ? pack_bf16x2(fmaf(o[2 * e], sc, p.pro_vadd), fmaf(o[2 * e + 1], sc, p.pro_vadd)) : 0u;
            if (row_ok) {
              uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
            }
          }
          if (row_ok && p.lse) {
            float lv = has ? ((PV8 ? m_ref + mshift : m_ref) + __log2f(l)) * kLn2 : -INFINITY;
            // the prologue's row term: the softmax cancels it, the LSE carries it
            if (has) lv += p.pro_lse_c;
            if (has && p.pro_lse_k != 0.f)
              lv += p.pro_lse_k * q_row_sum<DK>(p.q + t * p.q_stride_t + (int64_t)pi.h * p.q_stride_h);
            p.lse[(int64_t)pi.h * p.total_q + t] = lv;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace fa
