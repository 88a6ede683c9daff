// fa_prefill2.cuh -- two-query-tile (ping-pong) tcgen05 FlashAttention forward.
//
// One CTA computes 256 query rows of one (sequence, head) as two 128-row
// tiles A and B, each owned by its own softmax warpgroup, against one stream
// of K/V tiles that both share.  While warpgroup A turns S_A into P_A, the
// tensor core works on B's contractions and vice versa, so the softmax
// latency of one tile hides behind the other tile's MMAs:
//
//   MMA order:  QK_A(0) QK_B(0) | PV_A(0) QK_A(1) PV_B(0) QK_B(1) | PV_A(1) ...
//
// This is the same method as fa_prefill.cuh (tiled QK^T, online softmax with
// lazy rescaling, PV, LSE; RL-Kernel PR #237 and FlyDSL PR #1066), scheduled
// for the tensor-memory accumulators of sm_103a.
//
// TMEM (512 columns):  S_A [0,128)  S_B [128,256)  O_A [256,384)  O_B [384,512)
// P_X (bf16, the A operand of PV) overwrites the first 64 columns of S_X once
// the softmax has read S_X; tcgen05.mma ops issued by one thread run in issue
// order, so QK_X(j+1) (which rewrites S_X) cannot overtake PV_X(j).
//
// Warps: 0-3 softmax A, 4-7 softmax B, 8 TMA producer (Q, K, V), 9 TMEM
// allocation + MMA issue; the 12-warp variant adds two idle warps so that
// warpgroup 2 can hand its registers to the softmax warpgroups (setmaxnreg).
//
// NT = 1: one query tile per CTA (warps 0-3 softmax, 4 producer, 5 MMA, and
// 6-7 idle: setmaxnreg is executed by whole warpgroups), 256 TMEM columns (S [0,128), O [128,256)) and about 96 KB of shared memory,
// so that two CTAs share an SM: the tensor core alternates between the two
// CTAs' tiles as it does between A and B, and one CTA's set-up, pipeline
// fill and epilogue run under the other's main loop.  For short or ragged
// sequences, where those fixed costs weigh most.
#pragma once
#include "fa_prefill.cuh"

namespace fa {

template <int DK, int DV, bool PAGED, int MOD, bool BIGREG, int NT = 2>
struct Prefill2Cfg {
  static_assert(NT == 2 || (NT == 1 && BIGREG), "one query tile per CTA: register-split variant only");
  static_assert(MOD != 5 || BIGREG, "ALiBi in the contraction: register-split variants only");
  // K/V ring depths; one tile per CTA keeps two CTAs' rings within an SM
  // (MOD 5 at Dk 128 with two tiles: one K stage fewer, for its 12 KB of
  // constant operands)
  static constexpr int NSK = NT == 2 ? ((DK <= 64) ? 4 : (MOD == 5 ? 2 : 3)) : ((DK <= 64) ? 3 : 1);
  static constexpr int NSV = NT == 2 ? ((DK <= 64) ? 4 : 2) : ((DK <= 64) ? 2 : 1);
  static constexpr int kQTileBytes = kBlockM * DK * 2;
  static constexpr int kKBytes = kBlockN * DK * 2;
  static constexpr int kVBytes = kBlockN * DV * 2;
  static constexpr int kOffQ = 0;
  // MOD 5 (ALiBi with the bias in the contraction, one tile per CTA): three
  // 4 KB operands of one K=16 step, 32-byte swizzled -- Q rows (+a_hi, +a_lo),
  // (-a_hi, -a_lo) and key rows (n, n) -- after the Q tile
  static constexpr int kAugBytes = MOD == 5 ? 3 * 4096 : 0;
  static constexpr int kOffAug = NT * kQTileBytes;
  static constexpr int kOffK = kOffAug + kAugBytes;
  static constexpr int kOffV = kOffK + NSK * kKBytes;
  static constexpr int kOffBar = kOffV + NSV * kVBytes;
  static constexpr int kNumBars = 1 + 2 * NSK + 2 * NSV + 6;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 64 + 1024;
  // BIGREG: 12 warps; the producer/MMA warpgroup gives registers to the two
  // softmax warpgroups (setmaxnreg), so a whole S row fits in registers.
  // setmaxnreg acts on whole warpgroups, so the register-split variants fill
  // the last warpgroup with idle warps
  static constexpr int kThreads = NT == 2 ? (BIGREG ? 12 : 10) * 32 : 8 * 32;
  static constexpr int kSoftmaxWarps = 4 * NT;
  static constexpr int kProducerWarp = 4 * NT, kMmaWarp = 4 * NT + 1;
  static constexpr int kCtasPerSm = NT == 2 ? 1 : 2;
  static constexpr int kRegsSoftmax = NT == 2 ? 208 : 200, kRegsOther = NT == 2 ? 80 : 56;
  // registers the split needs from the CTA's pool, and the launch registers
  // per thread that provide them
  static constexpr int kPoolNeeded = kSoftmaxWarps * 32 * kRegsSoftmax + (kThreads - kSoftmaxWarps * 32) * kRegsOther;
  static constexpr int kMinLaunchRegs = (kPoolNeeded + kThreads - 1) / kThreads;
  static constexpr uint32_t kTmemCols = NT == 2 ? 512 : 256;
  static_assert(DV <= 128, "O_A/O_B hold 128 columns each");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(NT == 2 || 2 * (kSmemBytes + 1024) <= 233472, "two CTAs per SM");
  static_assert(NT == 2 || kMinLaunchRegs * kThreads * 2 <= 65536, "two CTAs' register pools per SM");
  static_assert(kThreads % 128 == 0 || !BIGREG, "setmaxnreg needs whole warpgroups");
};

struct Half {
  int valid;          // tile has rows
  int q0;             // first sequence-local row
  int ip_min, ip_max; // bottom-right aligned positions of its first/last row
  int klo, khi;       // key-tile range [klo, khi)
  int qt;             // 128-row block index (block mask)
};

struct PairInfo {
  int b, h, hk;
  int sq, sk;
  int q_row0;       // global token of the pair's first row
  int k_row0;
  int kt_lo, kt_hi; // union key-tile range
  Half x[2];
};

__device__ __forceinline__ bool half_active_h(const PrefillParams &p, const PairInfo &pi, const Half &hx, int kt) {
  if (!hx.valid || kt < hx.klo || kt >= hx.khi) return false;
  if (p.block_mask == nullptr) return true;
  if (kt >= p.n_kblk || hx.qt >= p.n_qblk) return false;
  const int64_t idx = ((int64_t)(pi.b * p.hq + pi.h) * p.n_qblk + hx.qt) * p.n_kblk + kt;
  return p.block_mask[idx] != 0;
}

__device__ __forceinline__ bool half_active(const PrefillParams &p, const PairInfo &pi, int X, int kt) {
  return X ? half_active_h(p, pi, pi.x[1], kt) : half_active_h(p, pi, pi.x[0], kt);
}

// ALiBi with the bias in the contraction (MOD 5): which linear form the key
// tile starting at kt * 128 takes for every row of the query tile -- +1 when
// all its keys are at or left of every row's diagonal i' (or under a causal
// mask, which hides the others), -1 when all are right of it, 0 when it
// straddles (the softmax then takes |i' - j| per element).
__device__ __forceinline__ int alibi_side(const PrefillParams &p, const Half &hx, int kt) {
  const int j0 = kt * kBlockN;
  if (p.causal || j0 + kBlockN - 1 <= hx.ip_min) return 1;
  if (j0 > hx.ip_max) return -1;
  return 0;
}

// Shared-memory descriptor of a K-major operand with 32-byte rows (K = 16
// bf16), 32-byte swizzle (mode 6), 8-row groups 256 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw32(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)(16 >> 4) << 16;
  d |= (uint64_t)(256 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)6 << 61;
  return d;
}

__device__ __forceinline__ int pair_next(const PrefillParams &p, const PairInfo &pi, int kt) {
  ++kt;
  while (kt < pi.kt_hi && !half_active(p, pi, 0, kt) && !half_active(p, pi, 1, kt)) ++kt;
  return kt;
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

template <int DK, int DV, bool PAGED, int MOD, bool BIGREG, int NT = 2>
__global__ void __launch_bounds__(Prefill2Cfg<DK, DV, PAGED, MOD, BIGREG, NT>::kThreads,
                                  Prefill2Cfg<DK, DV, PAGED, MOD, BIGREG, NT>::kCtasPerSm)
    fa_prefill2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using Cfg = Prefill2Cfg<DK, DV, PAGED, MOD, BIGREG, NT>;
  constexpr int kProducerWarp = Cfg::kProducerWarp, kMmaWarp = Cfg::kMmaWarp;
  // MOD: 0 plain scores, 1 ALiBi, 2 soft-cap; 3 and 4 are 1 and 2 with the
  // prologue's score terms (KT): a Q add's per-key term and, under the
  // soft-cap, the row term of a K add
  // MOD 5: ALiBi whose linear part rides in the QK contraction (one extra
  // K=16 step against constant operands), so the softmax is the plain one
  // plus a per-tile row constant; see the notes at the MMA issuer
  constexpr bool AMMA = MOD == 5;
  constexpr int MK = AMMA ? 0 : (MOD >= 3 ? MOD - 2 : MOD);
  constexpr bool KT = MOD == 3 || MOD == 4;
  constexpr int NSK = Cfg::NSK, NSV = Cfg::NSV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

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
    pi.q_row0 = qa + pt * NT * kBlockM;
    pi.k_row0 = ka;
  }
  if (pt * NT * kBlockM >= pi.sq) return;
  pi.kt_lo = 1 << 30;
  pi.kt_hi = 0;
#pragma unroll
  for (int X = 0; X < 2; ++X) {
    Half &hx = pi.x[X];
    hx.qt = pt * NT + X;
    hx.q0 = hx.qt * kBlockM;
    hx.valid = X < NT && hx.q0 < pi.sq;
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
    for (int e = threadIdx.x; e < NT * kBlockM; e += blockDim.x) {
      const int i = pt * NT * kBlockM + e;
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
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1;
  uint64_t *k_empty = k_full + NSK;
  uint64_t *v_full = k_empty + NSK;
  uint64_t *v_empty = v_full + NSV;
  uint64_t *s_full = v_empty + NSV;   // [2]
  uint64_t *p_full = s_full + 2;      // [2]
  uint64_t *o_done = p_full + 2;      // [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 8);

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    // full barriers: one arrival with the TMA bytes, or one per producer lane
    // for gathered rows
    const uint32_t n_fill = (PAGED && p.gather) ? 32u : 1u;
    for (int s = 0; s < NSK; ++s) {
      mbar_init(smem_u32(k_full + s), n_fill);
      mbar_init(smem_u32(k_empty + s), 1);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(smem_u32(v_full + s), n_fill);
      mbar_init(smem_u32(v_empty + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(s_full + x), 1);
      mbar_init(smem_u32(p_full + x), kBlockM);
      mbar_init(smem_u32(o_done + x), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  if constexpr (AMMA) {
    // The slope in raw-score units, a = alibi_log2 / scale_log2 (scale > 0),
    // as a bf16 pair a_hi + a_lo (products with key offsets n <= 127, exact
    // in bf16, then carry a to about 2^-17).  32-byte swizzle: a row's
    // 16-byte chunk c sits at chunk c ^ ((row >> 2) & 1).
    const float a = p.alibi_log2 / p.scale_log2;
    const __nv_bfloat16 ah = __float2bfloat16_rn(a);
    const __nv_bfloat16 al = __float2bfloat16_rn(a - __bfloat162float(ah));
    const uint32_t qpos = pack_bf16x2(__bfloat162float(ah), __bfloat162float(al));
    const uint32_t qneg = pack_bf16x2(-__bfloat162float(ah), -__bfloat162float(al));
    uint8_t *aug = smem + Cfg::kOffAug;
    for (int row = threadIdx.x; row < 128; row += blockDim.x) {
      const uint32_t kn = pack_bf16x2((float)row, (float)row);
      const int sw = (row >> 2) & 1;
      const uint32_t vals[3] = {qpos, qneg, kn};
#pragma unroll
      for (int b = 0; b < 3; ++b) {
        uint8_t *base = aug + b * 4096 + row * 32;
        *reinterpret_cast<uint4 *>(base + (sw << 4)) = make_uint4(vals[b], 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(base + ((1 ^ sw) << 4)) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // BIGREG: the softmax warps take the registers the other warps release
  // (setmaxnreg at the head of each role's branch).  The host launches this
  // variant only when the kernel's launch register count makes the split
  // (Cfg::kPoolNeeded) fit the CTA's register pool.
  if (BIGREG && warp >= kProducerWarp) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::kRegsOther));

  if (warp == kProducerWarp) {
    // ------------------------------------------------ producer: Q, K, V --
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_expect_tx(smem_u32(q_full), NT * Cfg::kQTileBytes);
#pragma unroll
      for (int X = 0; X < NT; ++X)
#pragma unroll
        for (int cb = 0; cb < DK / 64; ++cb)
          tma_load_3d(smem_u32(sQ + X * Cfg::kQTileBytes + cb * kBlockM * 128), &tm_q, smem_u32(q_full), cb * 64,
                      pi.h, pi.q_row0 + X * kBlockM);
    }
    if constexpr (PAGED) {
      if (p.gather) {
        // Pages of < 16 keys: every key row by its own page-table read and
        // 16-byte copies (fa_gather.cuh), page ids read one tile ahead.
        const int32_t *bt = p.block_table + (int64_t)pi.b * p.bt_stride;
        auto pages_of = [&](int kt, int (&pg)[4]) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int key = kt * kBlockN + lane + 32 * u;
            pg[u] = (kt < pi.kt_hi && key < pi.sk) ? __ldg(bt + (key >> p.page_shift)) : -1;
          }
        };
        // one slot in flight: a K slot frees after QK_B(j-3), which needs
        // K(j-3) and V(j-4); a V slot after PV_B(j-2), issued after
        // QK_A(j-1), so it needs K(j-1) and V(j-2); the newest slot before
        // those waits is V(j-1) or K(j) (two in flight would also be safe,
        // but measured slower)
        GatherPipe<1> gp;
        int pg[4], pgn[4];
        pages_of(first_kt, pg);
        int j = 0;
        bool ok = true;
        for (int kt = first_kt; kt < pi.kt_hi; ++j) {
          const int kn = pair_next(p, pi, kt);
          pages_of(kn, pgn);
          const int st = j % NSK, sv = j % NSV;
          if (lane == 0 && j >= NSK) ok = mbar_wait(smem_u32(k_empty + st), ((j / NSK) - 1) & 1, abort_flag, p.err);
          if (!__shfl_sync(0xffffffffu, ok, 0)) break;
#pragma unroll
          for (int cb = 0; cb < DK / 64; ++cb)
            gather_block<kBlockN, 128, kGatherSw128>(sK + st * Cfg::kKBytes + cb * kBlockN * 128, p.gk, pi.hk,
                                                     kt * kBlockN, p.page_size - 1, cb * 128, pg, lane);
          gp.commit(smem_u32(k_full + st));
          if (lane == 0 && j >= NSV) ok = mbar_wait(smem_u32(v_empty + sv), ((j / NSV) - 1) & 1, abort_flag, p.err);
          if (!__shfl_sync(0xffffffffu, ok, 0)) break;
#pragma unroll
          for (int cb = 0; cb < DV / 64; ++cb)
            gather_block<kBlockN, 128, kGatherSw128>(sV + sv * Cfg::kVBytes + cb * kBlockN * 128, p.gv, pi.hk,
                                                     kt * kBlockN, p.page_size - 1, cb * 128, pg, lane);
          gp.commit(smem_u32(v_full + sv));
          kt = kn;
#pragma unroll
          for (int u = 0; u < 4; ++u) pg[u] = pgn[u];
        }
        gp.drain();
      } else {
      // Paged K/V with pages of >= 16 keys: one TMA box and one page-table
      // read per page piece.  Lane 0 waits for the ring slot and arms its
      // barrier; the boxes are then issued by all lanes in parallel.
      const int32_t *bt = p.block_table + (int64_t)pi.b * p.bt_stride;
      auto load_pages = [&](const CUtensorMap *tm, uint8_t *dst, uint64_t *bar, int ncb, int kt) {
        for (int pg = lane; pg < p.pages_per_tile; pg += 32) {
          const int key0 = kt * kBlockN + pg * p.rows_per_box;
          const int page = key0 < pi.sk ? __ldg(bt + (key0 >> p.page_shift)) : -1;
          const int slot = key0 & (p.page_size - 1);
          for (int cb = 0; cb < ncb; ++cb)
            tma_load_4d(smem_u32(dst + cb * kBlockN * 128 + pg * p.rows_per_box * 128), tm, smem_u32(bar), cb * 64,
                        pi.hk, slot, page);
        }
      };
      int j = 0;
      bool ok = true;
      for (int kt = first_kt; kt < pi.kt_hi; kt = pair_next(p, pi, kt), ++j) {
        const int st = j % NSK, sv = j % NSV;
        if (lane == 0) {
          if (j >= NSK) ok = mbar_wait(smem_u32(k_empty + st), ((j / NSK) - 1) & 1, abort_flag, p.err);
          if (ok) mbar_expect_tx(smem_u32(k_full + st), Cfg::kKBytes);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        load_pages(&tm_k, sK + st * Cfg::kKBytes, k_full + st, DK / 64, kt);
        if (lane == 0) {
          if (j >= NSV) ok = mbar_wait(smem_u32(v_empty + sv), ((j / NSV) - 1) & 1, abort_flag, p.err);
          if (ok) mbar_expect_tx(smem_u32(v_full + sv), Cfg::kVBytes);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        load_pages(&tm_v, sV + sv * Cfg::kVBytes, v_full + sv, DV / 64, kt);
      }
      }
    } else if (lane == 0) {
      int j = 0;
      for (int kt = first_kt; kt < pi.kt_hi; kt = pair_next(p, pi, kt), ++j) {
        {
          const int st = j % NSK;
          if (j >= NSK && !mbar_wait(smem_u32(k_empty + st), ((j / NSK) - 1) & 1, abort_flag, p.err)) break;
          mbar_expect_tx(smem_u32(k_full + st), Cfg::kKBytes);
          uint8_t *dst = sK + st * Cfg::kKBytes;
#pragma unroll
          for (int cb = 0; cb < DK / 64; ++cb)
            tma_load_3d(smem_u32(dst + cb * kBlockN * 128), &tm_k, smem_u32(k_full + st), cb * 64, pi.hk,
                        pi.k_row0 + kt * kBlockN);
        }
        {
          const int sv = j % NSV;
          if (j >= NSV && !mbar_wait(smem_u32(v_empty + sv), ((j / NSV) - 1) & 1, abort_flag, p.err)) break;
          mbar_expect_tx(smem_u32(v_full + sv), Cfg::kVBytes);
          uint8_t *dst = sV + sv * Cfg::kVBytes;
#pragma unroll
          for (int cb = 0; cb < DV / 64; ++cb)
            tma_load_3d(smem_u32(dst + cb * kBlockN * 128), &tm_v, smem_u32(v_full + sv), cb * 64, pi.hk,
                        pi.k_row0 + kt * kBlockN);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------- MMA issuer --
    constexpr uint32_t idesc_qk = idesc_bf16_f32(kBlockM, kBlockN, 0, 0);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kBlockM, DV, 0, 1);
    const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
    int n_pv[2] = {0, 0};
    bool ok = mbar_wait(smem_u32(q_full), 0, abort_flag, p.err);

    // Descriptor words, computed once: a K-major 128-byte-swizzled operand
    // steps 32 bytes per K=16 slice and jumps to the next 64-column block
    // (rows * 128 bytes) every fourth slice; V (MN-major) steps 16 rows.
    const uint64_t dq0 = smem_desc_sw128(sQa, 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(sKa, 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(sVa, kBlockN * 128, 1024);
    const uint32_t q_lo = (uint32_t)dq0, k_lo = (uint32_t)dk0, qk_hi = (uint32_t)(dq0 >> 32);
    const uint32_t v_lo = (uint32_t)dv0, v_hi = (uint32_t)(dv0 >> 32);
    // MOD 5: one more K=16 step adds a * (j - j0) (left of every row's
    // diagonal, or under a causal mask) or -a * (j - j0) (right of it) to
    // each score of the key tile starting at j0; tiles that straddle the
    // diagonal get no extra step (the softmax takes |i' - j| per element).
    const uint64_t aug_q0 = smem_desc_sw32(smem_u32(smem + Cfg::kOffAug));
    const uint32_t aug_lo = (uint32_t)aug_q0, aug_hi = (uint32_t)(aug_q0 >> 32);
    auto qk = [&](int X, int st, int kt) {
      const uint32_t d = tmem + (X ? 128u : 0u);
      uint32_t a = q_lo + (uint32_t)(X * (Cfg::kQTileBytes >> 4));
      uint32_t b = k_lo + (uint32_t)(st * (Cfg::kKBytes >> 4));
#pragma unroll
      for (int ks = 0; ks < DK / 16; ++ks) {
        if (ks == 0) mma_ss_w<0>(d, a, qk_hi, b, qk_hi, idesc_qk);
        else mma_ss_w<1>(d, a, qk_hi, b, qk_hi, idesc_qk);
        const uint32_t step = ((ks + 1) & 3) ? 2u : (uint32_t)((kBlockM * 128 - 96) >> 4);
        a += step;
        b += step;
      }
      if constexpr (AMMA) {
        const int side = alibi_side(p, X ? pi.x[1] : pi.x[0], kt);
        if (side != 0)
          mma_ss_w<1>(d, aug_lo + (side > 0 ? 0u : (4096u >> 4)), aug_hi, aug_lo + (2u * 4096u >> 4), aug_hi,
                      idesc_qk);
      }
      tc_commit(smem_u32(s_full + X));
    };
    auto pv = [&](int X, int sv) {
      const uint32_t a = tmem + (X ? 128u : 0u);                 // P_X aliases S_X
      const uint32_t d = tmem + NT * 128u + (X ? 128u : 0u);
      uint32_t b = v_lo + (uint32_t)(sv * (Cfg::kVBytes >> 4));
      const uint32_t acc0 = n_pv[X] > 0 ? 1u : 0u;
#pragma unroll
      for (int ks = 0; ks < kBlockN / 16; ++ks) {
        mma_ts_w(d, a + ks * 8, b, v_hi, idesc_pv, ks > 0 ? 1u : acc0);
        b += (16 * 128) >> 4;
      }
      tc_commit(smem_u32(o_done + X));
    };

    // One lane runs the whole issue loop (no warp-wide steps): the tensor
    // core is fed only while this thread is free, so the loop keeps its
    // bookkeeping small -- activity flags of the next tile are carried over.
    if (lane == 0 && ok) {
      bool a0 = half_active(p, pi, 0, first_kt), a1 = half_active(p, pi, 1, first_kt);
      ok = mbar_wait(smem_u32(k_full + 0), 0, abort_flag, p.err);
      if (ok) {
        tc_fence_after();
        if (a0) qk(0, 0, first_kt);
        if (a1) qk(1, 0, first_kt);
        tc_commit(smem_u32(k_empty + 0));
      }
      int j = 0;
      for (int kt = first_kt; ok && kt < pi.kt_hi; ++j) {
        const int kn = pair_next(p, pi, kt);
        const bool more = kn < pi.kt_hi;
        const bool n0 = more && half_active(p, pi, 0, kn);
        const bool n1 = more && half_active(p, pi, 1, kn);
        const int sv = j % NSV;
        const int st = (j + 1) % NSK;
        // V of this tile; rows past the sequence end were cleared by the
        // softmax warpgroup before it released P (see the softmax loop).
        if (!(ok = mbar_wait(smem_u32(v_full + sv), (j / NSV) & 1, abort_flag, p.err))) break;
        if (a0) {
          if (!(ok = mbar_wait(smem_u32(p_full + 0), n_pv[0] & 1, abort_flag, p.err))) break;
          tc_fence_after();
          pv(0, sv);
          ++n_pv[0];
        }
        if (more) {
          if (!(ok = mbar_wait(smem_u32(k_full + st), ((j + 1) / NSK) & 1, abort_flag, p.err))) break;
          tc_fence_after();
          if (n0) qk(0, st, kn);
        }
        if (a1) {
          if (!(ok = mbar_wait(smem_u32(p_full + 1), n_pv[1] & 1, abort_flag, p.err))) break;
          tc_fence_after();
          pv(1, sv);
          ++n_pv[1];
        }
        tc_commit(smem_u32(v_empty + sv));
        if (more) {
          if (n1) qk(1, st, kn);
          tc_commit(smem_u32(k_empty + st));
        }
        a0 = n0;
        a1 = n1;
        kt = kn;
      }
    }
  } else if (warp < Cfg::kSoftmaxWarps) {
    // ---------------------------------------------------------- softmax --
    if constexpr (BIGREG) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::kRegsSoftmax));
    const int X = warp >> 2;                  // 0: tile A, 1: tile B
    const int r = threadIdx.x & 127;          // row in the tile == TMEM lane
    const Half hx = X ? pi.x[1] : pi.x[0];
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t colS = X ? 128u : 0u, colO = NT * 128u + (X ? 128u : 0u);
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
    // MOD 0 runs with a positive scale only (the host routes other scales to
    // the general path), so raw scores can be maxed before scaling.
    constexpr bool fast = (MK == 0);
    // Exponentials 2^(c*v - m) of a 32-column chunk with packed fp32 math,
    // their row sums and the bf16 packing of P.
    auto chunk_exp = [&](const float (&v)[32], float c, float m, uint32_t (&pk)[16], float (&acc)[4]) {
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float t0, t1;
        fma2(t0, t1, v[e], v[e + 1], c, -m);
        const float a0 = ex2(t0), a1 = ex2(t1);
        const int q = ((e >> 1) & 1) * 2;
        add2(acc[q], acc[q + 1], a0, a1);
        pk[e >> 1] = pack_bf16x2(a0, a1);
      }
    };
    const float cexp = fast ? p.scale_log2 : 1.f;
    // The deferred max (below) shortens the softmax; it pays where the
    // softmax is the critical path, i.e. with a score mod.  Plain scores keep
    // the max-first order, and so does ALiBi, for accuracy: its bias puts a
    // row's mass on the nearest keys, and each tile toward them raises the
    // row max past the rescale threshold, so with the max taken first the
    // reference lands on the dominant key and its P is exactly 1.  Against a
    // deferred reference that P can be anything up to 2^64, and its bf16
    // rounding (up to 2^-9 relative, not mirrored in the fp32 row sum) moved
    // outputs of magnitude 2 by a whole bf16 step.  Soft-capped scores are
    // bounded, so no single key takes over a row and the deferred max stays.
    constexpr bool kDeferredMax = (MK == 2);
    int j = -1;   // index of the tile in the pair's list (K/V ring position)
    for (int kt = first_kt; kt < pi.kt_hi; kt = pair_next(p, pi, kt)) {
      ++j;
      if (!half_active_h(p, pi, hx, kt)) continue;
      ok = mbar_wait(smem_u32(s_full + X), cnt & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sa = tmem + lane_base + colS;
      const int j0 = kt * kBlockN;
      bool need_mask = (j0 + kBlockN > pi.sk);
      if (p.causal && j0 + kBlockN - 1 > hx.ip_min) need_mask = true;
      if (p.window > 0) {
        if (j0 < hx.ip_max - p.window + 1) need_mask = true;
        if (!p.causal && j0 + kBlockN - 1 > hx.ip_min + p.window - 1) need_mask = true;
      }
      // MOD 5: S already holds -+slope (j - j0) in raw units for a tile on
      // one side of the diagonal; the rest of the bias, -+slope (i' - j0),
      // is a row constant (ct, log2 units) that joins the max and the
      // exponent's reference.  A straddling tile (lin false) takes the
      // per-element form instead.
      bool lin = true;
      float ct = 0.f;
      if constexpr (AMMA) {
        const int side = alibi_side(p, hx, kt);
        lin = side != 0;
        ct = side > 0 ? p.alibi_log2 * (float)(j0 - ip) : p.alibi_log2 * (float)(ip - j0);
      }
      const float cexp_t = AMMA ? (lin ? p.scale_log2 : 1.f) : cexp;
      const float mshift_t = (AMMA && lin) ? ct : 0.f;
      // Scores of 32 keys starting at key jc, in scaled log2 units (the fast
      // path keeps raw scores and folds the scale into the exponent's FMA).
      auto scores = [&](float (&v)[32], int jc) {
        if constexpr (MK == 2) {
          // Soft-cap: each step runs over the whole chunk before the next,
          // with packed pairs, so that the 32 independent chains of its two
          // transcendental steps interleave.
          const float c2u = 2.f * kLog2e * p.softcap_arg;   // raw score -> 2u log2(e)
          if constexpr (KT) {
            // plus the row term and the key's term (in the same units); no
            // term is read past cb_ld (the pre-pass flags such keys)
            const bool in_ld = p.col_bias != nullptr && jc + 32 <= p.cb_ld;
            const float4 *c4 =
                reinterpret_cast<const float4 *>(p.col_bias + ((int64_t)pi.b * p.hkv + pi.hk) * p.cb_ld + jc);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 c = in_ld ? c4[e >> 2] : make_float4(0.f, 0.f, 0.f, 0.f);
              fma2v(v[e], v[e + 1], c2u, c.x + row_term, c.y + row_term);
              fma2v(v[e + 2], v[e + 3], c2u, c.z + row_term, c.w + row_term);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; e += 2) mul2(v[e], v[e + 1], c2u);
          }
          // cl tanh(u) = cl - 2 cl / (1 + e^{2u})  (see softcap_log2_score)
          const float cl = p.softcap_log2;
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = ex2(v[e]);
#pragma unroll
          for (int e = 0; e < 32; e += 2) add2(v[e], v[e + 1], 1.f, 1.f);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = rcp_approx(v[e]);
#pragma unroll
          for (int e = 0; e < 32; e += 2) fma2(v[e], v[e + 1], v[e], v[e + 1], -2.f * cl, cl);
        } else if constexpr (!fast) {
          const float dbase = (float)(ip - jc);   // ALiBi: |i' - j| = |dbase - e|, exact in fp32
          if constexpr (KT) {
            // scaled score (log2 units) plus the key's term; no term is read
            // past cb_ld (the pre-pass flags such keys)
            const bool in_ld = p.col_bias != nullptr && jc + 32 <= p.cb_ld;
            const float4 *c4 =
                reinterpret_cast<const float4 *>(p.col_bias + ((int64_t)pi.b * p.hkv + pi.hk) * p.cb_ld + jc);
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float4 c = in_ld ? c4[e >> 2] : make_float4(0.f, 0.f, 0.f, 0.f);
              v[e] = fmaf(v[e], p.scale_log2, c.x + row_term);
              v[e + 1] = fmaf(v[e + 1], p.scale_log2, c.y + row_term);
              v[e + 2] = fmaf(v[e + 2], p.scale_log2, c.z + row_term);
              v[e + 3] = fmaf(v[e + 3], p.scale_log2, c.w + row_term);
            }
          }
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float x;
            if constexpr (KT) {
              x = v[e];
            } else {
              x = v[e] * p.scale_log2;
            }
            x -= p.alibi_log2 * fabsf(dbase - (float)e);
            v[e] = x;
          }
        }
        if constexpr (AMMA) {
          if (!lin) {
            const float dbase = (float)(ip - jc);   // |i' - j| = |dbase - e|, exact in fp32
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = fmaf(-p.alibi_log2, fabsf(dbase - (float)e), v[e] * p.scale_log2);
          }
        }
        if (need_mask) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = jc + e;
            bool allowed = j < pi.sk;
            if (p.causal) allowed = allowed && (j <= ip);
            if (p.window > 0) allowed = allowed && (p.causal ? (ip - j < p.window) : (abs(ip - j) < p.window));
            v[e] = allowed ? v[e] : -INFINITY;
          }
        }
      };
      float alpha_tile = 1.f;
      bool warp_need = false;
      float sum[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (BIGREG) {
        // One pass: the whole S row comes out of TMEM with a single wait.
        float sv[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(sa + c * 32, sv[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) scores(sv[c], j0 + c * 32);
        // Exponentials against the running reference, stored as P; the row
        // sum of the tile comes back in `acc`.
        auto exp_store = [&](float m_use, float (&acc)[4]) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
            chunk_exp(sv[c], cexp_t, AMMA ? m_use - mshift_t : m_use, pk, acc);
            tmem_st16(sa + c * 16, pk);
          }
        };
        // Deferred max: once a row has a reference, the tile's exponentials
        // are taken against it directly.  Only if the tile's sum exceeds
        // 2^64 (a score more than ~57 log2 units above the reference) is its
        // max computed and P redone -- fp32 O and l stay far from overflow in
        // between, and bf16 P keeps its relative precision at any magnitude.
        // A row's first tile (no reference yet) takes the max first.
        bool slow = !kDeferredMax || __any_sync(0xffffffffu, m_ref == -INFINITY);
        if (!slow) {
          exp_store(m_ref, sum);
          const float ts = (sum[0] + sum[1]) + (sum[2] + sum[3]);
          slow = __any_sync(0xffffffffu, !(ts <= kGuardSum));
          if (slow) {
            tmem_wait_st();   // P is written again below
            sum[0] = sum[1] = sum[2] = sum[3] = 0.f;
          }
        }
        if (slow) {
          // Balanced tree of 3-input maxima over the 128 scores (depth 5).
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
          if constexpr (AMMA) {
            if (lin && tmax != -INFINITY) tmax = fmaf(tmax, p.scale_log2, ct);
          } else {
            if (fast && tmax != -INFINITY) tmax *= p.scale_log2;
          }
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
        // The S row is processed in two halves of 64 columns, each with the
        // deferred max of the one-pass form: exponentials against the
        // running reference unless the row has none yet or the half's sum
        // exceeds 2^64; then the half's max moves the reference (lazily, by
        // the rescale threshold) and, for the second half, the first half's
        // P (already in TMEM) is rescaled too.
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
              uint32_t pk[16];
              chunk_exp(sv[c], cexp, m_use, pk, hsum);
              tmem_st16(sa + hf * 32 + c * 16, pk);
            }
          };
          bool slow = !kDeferredMax || __any_sync(0xffffffffu, m_ref == -INFINITY);
          if (!slow) {
            exp_store(m_ref);
            const float hs = (hsum[0] + hsum[1]) + (hsum[2] + hsum[3]);
            slow = __any_sync(0xffffffffu, !(hs <= kGuardSum));
            if (slow) {
              tmem_wait_st();
              hsum[0] = hsum[1] = hsum[2] = hsum[3] = 0.f;
            }
          }
          if (slow) {
            // tree of 3-input maxima over the 64 scores of this half
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
            if (fast && hmax != -INFINITY) hmax *= p.scale_log2;
            const float m_new = fmaxf(m_ref, hmax);
            const bool need = m_new > m_ref + kRescaleThreshold;
            const bool wneed = __any_sync(0xffffffffu, need);
            if (wneed) {
              const float alpha = need ? ex2(m_ref - m_new) : 1.f;   // 0 when m_ref = -inf
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
                // P of the first half was computed against the old reference.
                tmem_wait_st();
                float pw[32];
                tmem_ld32(sa, pw);
                tmem_wait_ld();
                uint32_t w[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                  const uint32_t u = __float_as_uint(pw[e]);
                  const float lo = __uint_as_float(u << 16) * alpha, hi = __uint_as_float(u & 0xFFFF0000u) * alpha;
                  w[e] = pack_bf16x2(lo, hi);
                }
                tmem_st32(sa, w);
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
        // O_X must hold PV_X(cnt-1) before it is rescaled.
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
      // Keys past the sequence end may hold anything (NaN-poisoned page
      // slots): P is 0 there, but 0 * NaN is NaN, so those V rows are cleared
      // before P is released -- by warpgroup A, or by B when A skips the tile.
      const int valid = pi.sk - j0;
      if (valid < kBlockN && (X == 0 || !half_active(p, pi, 0, kt))) {
        const int sv = j % NSV;
        ok = mbar_wait(smem_u32(v_full + sv), (j / NSV) & 1, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        uint8_t *vt = sV + sv * Cfg::kVBytes;
        const int per_cb = (kBlockN - valid) * 8;            // 16-byte chunks per column block
        for (int idx = r; idx < per_cb * (DV / 64); idx += kBlockM) {
          const int cb = idx / per_cb, rem = idx - cb * per_cb;
          *reinterpret_cast<uint4 *>(vt + cb * kBlockN * 128 + valid * 128 + rem * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
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
        if (row_ok) {
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
            float lv = has ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
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
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace fa
