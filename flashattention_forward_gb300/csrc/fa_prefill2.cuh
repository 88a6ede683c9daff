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
// Warps (320 threads): 0-3 softmax A, 4-7 softmax B, 8 TMA producer (Q, K, V),
// 9 TMEM allocation + MMA issue.
#pragma once
#include "fa_prefill.cuh"

namespace fa {

template <int DK, int DV, bool PAGED, int MOD>
struct Prefill2Cfg {
  static constexpr int NSK = (DK <= 64) ? 4 : 3;
  static constexpr int NSV = (DK <= 64) ? 4 : 2;
  static constexpr int kQTileBytes = kBlockM * DK * 2;
  static constexpr int kKBytes = kBlockN * DK * 2;
  static constexpr int kVBytes = kBlockN * DV * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = 2 * kQTileBytes;
  static constexpr int kOffV = kOffK + NSK * kKBytes;
  static constexpr int kOffBar = kOffV + NSV * kVBytes;
  static constexpr int kNumBars = 1 + 2 * NSK + 2 * NSV + 6;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 64 + 1024;
  static constexpr int kThreads = 10 * 32;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(DV <= 128, "O_A/O_B hold 128 columns each");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
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

template <int DK, int DV, bool PAGED, int MOD>
__global__ void __launch_bounds__(Prefill2Cfg<DK, DV, PAGED, MOD>::kThreads, 1)
    fa_prefill2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using Cfg = Prefill2Cfg<DK, DV, PAGED, MOD>;
  constexpr int NSK = Cfg::NSK, NSV = Cfg::NSV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ------------------------------------------------------------ work tile --
  PairInfo pi;
  pi.h = blockIdx.x;
  pi.b = blockIdx.y;
  const int pt = p.n_qtiles - 1 - (int)blockIdx.z;   // longest (latest) pairs first
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
    for (int s = 0; s < NSK; ++s) {
      mbar_init(smem_u32(k_full + s), 1);
      mbar_init(smem_u32(k_empty + s), 1);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(smem_u32(v_full + s), 1);
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
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------ producer: Q, K, V --
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_expect_tx(smem_u32(q_full), 2 * Cfg::kQTileBytes);
#pragma unroll
      for (int X = 0; X < 2; ++X)
#pragma unroll
        for (int cb = 0; cb < DK / 64; ++cb)
          tma_load_3d(smem_u32(sQ + X * Cfg::kQTileBytes + cb * kBlockM * 128), &tm_q, smem_u32(q_full), cb * 64,
                      pi.h, pi.q_row0 + X * kBlockM);
      const int32_t *bt = PAGED ? p.block_table + (int64_t)pi.b * p.bt_stride : nullptr;
      int j = 0;
      for (int kt = first_kt; kt < pi.kt_hi; kt = pair_next(p, pi, kt), ++j) {
        {
          const int st = j % NSK;
          if (j >= NSK && !mbar_wait(smem_u32(k_empty + st), ((j / NSK) - 1) & 1, abort_flag, p.err)) break;
          mbar_expect_tx(smem_u32(k_full + st), Cfg::kKBytes);
          uint8_t *dst = sK + st * Cfg::kKBytes;
          if constexpr (PAGED) {
            for (int pg = 0; pg < p.pages_per_tile; ++pg) {
              const int key0 = kt * kBlockN + pg * p.rows_per_box;
              const int page = key0 < pi.sk ? __ldg(bt + (key0 >> p.page_shift)) : -1;
              const int slot = key0 & (p.page_size - 1);
#pragma unroll
              for (int cb = 0; cb < DK / 64; ++cb)
                tma_load_4d(smem_u32(dst + cb * kBlockN * 128 + pg * p.rows_per_box * 128), &tm_k,
                            smem_u32(k_full + st), cb * 64, pi.hk, slot, page);
            }
          } else {
#pragma unroll
            for (int cb = 0; cb < DK / 64; ++cb)
              tma_load_3d(smem_u32(dst + cb * kBlockN * 128), &tm_k, smem_u32(k_full + st), cb * 64, pi.hk,
                          pi.k_row0 + kt * kBlockN);
          }
        }
        {
          const int sv = j % NSV;
          if (j >= NSV && !mbar_wait(smem_u32(v_empty + sv), ((j / NSV) - 1) & 1, abort_flag, p.err)) break;
          mbar_expect_tx(smem_u32(v_full + sv), Cfg::kVBytes);
          uint8_t *dst = sV + sv * Cfg::kVBytes;
          if constexpr (PAGED) {
            for (int pg = 0; pg < p.pages_per_tile; ++pg) {
              const int key0 = kt * kBlockN + pg * p.rows_per_box;
              const int page = key0 < pi.sk ? __ldg(bt + (key0 >> p.page_shift)) : -1;
              const int slot = key0 & (p.page_size - 1);
#pragma unroll
              for (int cb = 0; cb < DV / 64; ++cb)
                tma_load_4d(smem_u32(dst + cb * kBlockN * 128 + pg * p.rows_per_box * 128), &tm_v,
                            smem_u32(v_full + sv), cb * 64, pi.hk, slot, page);
            }
          } else {
#pragma unroll
            for (int cb = 0; cb < DV / 64; ++cb)
              tma_load_3d(smem_u32(dst + cb * kBlockN * 128), &tm_v, smem_u32(v_full + sv), cb * 64, pi.hk,
                          pi.k_row0 + kt * kBlockN);
          }
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------- MMA issuer --
    constexpr uint32_t idesc_qk = idesc_bf16_f32(kBlockM, kBlockN, 0, 0);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kBlockM, DV, 0, 1);
    const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
    int n_pv[2] = {0, 0};
    bool ok = mbar_wait(smem_u32(q_full), 0, abort_flag, p.err);

    auto qk = [&](int X, int st) {
      const uint32_t d = tmem + (X ? 128u : 0u);
#pragma unroll
      for (int ks = 0; ks < DK / 16; ++ks) {
        const uint32_t off = (ks >> 2) * (kBlockM * 128) + (ks & 3) * 32;
        const uint64_t da = smem_desc_sw128(sQa + X * Cfg::kQTileBytes + off, 16, 1024);
        const uint64_t db = smem_desc_sw128(sKa + st * Cfg::kKBytes + off, 16, 1024);
        mma_ss(d, da, db, idesc_qk, ks > 0);
      }
      tc_commit(smem_u32(s_full + X));
    };
    auto pv = [&](int X, int sv) {
      const uint32_t a = tmem + (X ? 128u : 0u);                 // P_X aliases S_X
      const uint32_t d = tmem + 256u + (X ? 128u : 0u);
#pragma unroll
      for (int ks = 0; ks < kBlockN / 16; ++ks) {
        const uint64_t db = smem_desc_sw128(sVa + sv * Cfg::kVBytes + ks * 16 * 128, kBlockN * 128, 1024);
        mma_ts(d, a + ks * 8, db, idesc_pv, (n_pv[X] > 0 || ks > 0) ? 1u : 0u);
      }
      tc_commit(smem_u32(o_done + X));
    };

    // prologue: QK of the first tile for both halves
    if (ok) {
      ok = mbar_wait(smem_u32(k_full + 0), 0, abort_flag, p.err);
      if (ok) {
        tc_fence_after();
        if (lane == 0) {
          if (half_active(p, pi, 0, first_kt)) qk(0, 0);
          if (half_active(p, pi, 1, first_kt)) qk(1, 0);
          tc_commit(smem_u32(k_empty + 0));
        }
        __syncwarp();
      }
    }
    int j = 0;
    for (int kt = first_kt; ok && kt < pi.kt_hi; ++j) {
      const int kn = pair_next(p, pi, kt);
      const int sv = j % NSV;
      const bool a0 = half_active(p, pi, 0, kt), a1 = half_active(p, pi, 1, kt);
      const bool n0 = kn < pi.kt_hi && half_active(p, pi, 0, kn);
      const bool n1 = kn < pi.kt_hi && half_active(p, pi, 1, kn);
      ok = mbar_wait(smem_u32(v_full + sv), (j / NSV) & 1, abort_flag, p.err);
      if (!ok) break;
      // Keys past the sequence end may be NaN-poisoned; clear those V rows.
      const int valid = pi.sk - kt * kBlockN;
      if (valid < kBlockN) {
        uint8_t *vt = sV + sv * Cfg::kVBytes;
#pragma unroll
        for (int cb = 0; cb < DV / 64; ++cb) {
          uint4 *z = reinterpret_cast<uint4 *>(vt + cb * kBlockN * 128 + valid * 128);
          const int n16 = (kBlockN - valid) * 8;
          for (int i = lane; i < n16; i += 32) z[i] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (a0) {
        ok = mbar_wait(smem_u32(p_full + 0), n_pv[0] & 1, abort_flag, p.err);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) pv(0, sv);
        ++n_pv[0];
        __syncwarp();
      }
      if (kn < pi.kt_hi) {
        const int st = (j + 1) % NSK;
        ok = mbar_wait(smem_u32(k_full + st), ((j + 1) / NSK) & 1, abort_flag, p.err);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0 && n0) qk(0, st);
        __syncwarp();
      }
      if (a1) {
        ok = mbar_wait(smem_u32(p_full + 1), n_pv[1] & 1, abort_flag, p.err);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) pv(1, sv);
        ++n_pv[1];
        __syncwarp();
      }
      if (lane == 0) tc_commit(smem_u32(v_empty + sv));
      if (kn < pi.kt_hi) {
        const int st = (j + 1) % NSK;
        if (lane == 0) {
          if (n1) qk(1, st);
          tc_commit(smem_u32(k_empty + st));
        }
      }
      __syncwarp();
      kt = kn;
    }
  } else if (warp < 8) {
    // ---------------------------------------------------------- softmax --
    const int X = warp >> 2;                  // 0: tile A, 1: tile B
    const int r = threadIdx.x & 127;          // row in the tile == TMEM lane
    const Half hx = X ? pi.x[1] : pi.x[0];
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t colS = X ? 128u : 0u, colO = 256u + (X ? 128u : 0u);
    const int i = hx.q0 + r;
    const int ip = i + pi.sk - pi.sq;
    float m_ref = -INFINITY, l = 0.f;
    int cnt = 0;
    bool ok = true;
    const bool fast = (MOD == 0) && (p.scale_log2 > 0.f);
    for (int kt = first_kt; kt < pi.kt_hi; kt = pair_next(p, pi, kt)) {
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
      // Scores of 32 keys starting at key jc, in scaled log2 units (the fast
      // path keeps raw scores and folds the scale into the exponent's FMA).
      auto scores = [&](float (&v)[32], int jc) {
        if (!fast) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float x;
            if constexpr (MOD == 2) {
              const float t = v[e] * p.softcap_arg;
              const float em = ex2(-2.f * kLog2e * fabsf(t));
              x = copysignf(__fdividef(1.f - em, 1.f + em), t) * p.softcap_log2;
            } else {
              x = v[e] * p.scale_log2;
            }
            if constexpr (MOD == 1) x -= p.alibi_log2 * (float)abs(ip - (jc + e));
            v[e] = x;
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
      // Pass 1: tile max (chunks of 32 columns, 8 independent max chains).
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; c += 2) {
        float s0[32], s1[32];
        tmem_ld32(sa + c * 32, s0);
        tmem_ld32(sa + c * 32 + 32, s1);
        tmem_wait_ld();
        scores(s0, j0 + c * 32);
        scores(s1, j0 + c * 32 + 32);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          mx[e & 7] = fmaxf(mx[e & 7], s0[e]);
          mx[e & 7] = fmaxf(mx[e & 7], s1[e]);
        }
      }
      float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      if (fast && tmax != -INFINITY) tmax *= p.scale_log2;

      const float m_new = fmaxf(m_ref, tmax);
      const bool need = m_new > m_ref + kRescaleThreshold;
      const bool warp_need = __any_sync(0xffffffffu, need);
      float alpha = 1.f;
      if (need) {
        alpha = ex2(m_ref - m_new);
        l *= alpha;
        m_ref = m_new;
      }
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      // Pass 2: p = 2^(x - m), row sum, bf16 P written over the S columns
      // already read (P chunk c occupies columns [16c, 16c+16)).
      float sum[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) sum[k] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; c += 2) {
        float s0[32], s1[32];
        tmem_ld32(sa + c * 32, s0);
        tmem_ld32(sa + c * 32 + 32, s1);
        tmem_wait_ld();
        scores(s0, j0 + c * 32);
        scores(s1, j0 + c * 32 + 32);
        uint32_t pk0[16], pk1[16];
        if (fast) {
          const float c2 = p.scale_log2;
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float a0 = ex2(fmaf(s0[e], c2, -m_use)), a1 = ex2(fmaf(s0[e + 1], c2, -m_use));
            const float b0 = ex2(fmaf(s1[e], c2, -m_use)), b1 = ex2(fmaf(s1[e + 1], c2, -m_use));
            sum[(e >> 1) & 3] += a0 + a1;
            sum[4 + ((e >> 1) & 3)] += b0 + b1;
            pk0[e >> 1] = pack_bf16x2(a0, a1);
            pk1[e >> 1] = pack_bf16x2(b0, b1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float a0 = ex2(s0[e] - m_use), a1 = ex2(s0[e + 1] - m_use);
            const float b0 = ex2(s1[e] - m_use), b1 = ex2(s1[e + 1] - m_use);
            sum[(e >> 1) & 3] += a0 + a1;
            sum[4 + ((e >> 1) & 3)] += b0 + b1;
            pk0[e >> 1] = pack_bf16x2(a0, a1);
            pk1[e >> 1] = pack_bf16x2(b0, b1);
          }
        }
        tmem_st16(sa + c * 16, pk0);
        tmem_st16(sa + c * 16 + 16, pk1);
      }
      l += ((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7]));
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
          const uint32_t oa = tmem + lane_base + colO;
#pragma unroll
          for (int c = 0; c < DV / 32; ++c) {
            float o[32];
            tmem_ld32(oa + c * 32, o);
            tmem_wait_ld();
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = has ? pack_bf16x2(o[2 * e] * inv_l, o[2 * e + 1] * inv_l) : 0u;
            if (row_ok) {
              uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
            }
          }
          if (row_ok && p.lse)
            p.lse[(int64_t)pi.h * p.total_q + t] = has ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
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
