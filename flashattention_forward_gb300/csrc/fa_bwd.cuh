// fa_bwd.cuh -- FlashAttention backward on tcgen05: gradients of
// L = sum(dO * out) with respect to Q, K and V from the forward's saved
// per-row log-sum-exp (RL-Kernel PR #237, backward commit: a Delta
// preprocess, then dQ/dK/dV recomputed from the saved LSE).
//
//   Delta_i = sum_x dO_ix * O_ix                       (fa_bwd_delta_kernel)
//   P_ij    = exp(scale * <q_i, k_j> - LSE_i)          (allowed (i, j) only)
//   dP_ij   = <dO_i, v_j>,   dS_ij = P_ij * (dP_ij - Delta_i)
//   dV_j    = sum_i P_ij dO_i,   dK_j = scale * sum_i dS_ij q_i
//   dQ_i    = scale * sum_j dS_ij k_j
//
// Score mods (fkl_python PR #7, flex commit), as in the forward: ALiBi adds
// -slope*|i' - j| to the scaled score, which leaves dS as it is; the soft-cap
// s = cap*tanh(u/cap), u = scale*<q, k>, multiplies the gradient by
// ds/du = 1 - tanh^2(u/cap), which the kernels fold into P before forming dS.
//
// Two kernels share the arithmetic and split the outputs so that no output
// needs an atomic: fa_bwd_dq_kernel (one 128-row query tile per CTA, looping
// over key tiles) and fa_bwd_dkdv_kernel (one 128-key tile per CTA, looping
// over the q heads of its kv head's group and their query tiles).  Each
// recomputes S and dP; the results are deterministic.
//
// Operands are the 128-byte-swizzled 64-column TMA tiles of the forward
// kernels.  A [rows, D] tile serves as a K-major operand (for S = Q K^T and
// dP = dO V^T, contraction over D) and as an MN-major B operand (for
// dQ += dS K, dV += P^T dO and dK += dS^T Q, contraction over the rows).
// P, dS and their transposes go from registers to TMEM as bf16 and are the
// A operand of the accumulating MMAs (A from TMEM).
#pragma once
#include "fa_prefill.cuh"
#include "fa_bwd_params.h"

namespace fa {

// Delta_i = <dO_i, O_i> in fp32.  Eight lanes per (token, head) row, each
// with 16-byte loads of O and dO (D/64 of them), four rows per warp.
__global__ void __launch_bounds__(256) fa_bwd_delta_kernel(const BwdDeltaParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * 4 + (lane >> 3);
  const int sub = lane & 7;
  float acc = 0.f;
  const bool live = row < p.total_q * p.hq;
  if (live) {
    const int64_t t = row / p.hq;
    const int h = (int)(row - t * p.hq);
    const __nv_bfloat16 *o = p.out + t * p.o_stride_t + (int64_t)h * p.o_stride_h;
    const __nv_bfloat16 *g = p.dout + t * p.do_stride_t + (int64_t)h * p.do_stride_h;
    uint4 ov[2], gv[2];
#pragma unroll
    for (int c = 0; c < 2; ++c)
      if (c * 64 + sub * 8 < p.d) {
        ov[c] = *reinterpret_cast<const uint4 *>(o + c * 64 + sub * 8);
        gv[c] = *reinterpret_cast<const uint4 *>(g + c * 64 + sub * 8);
      }
#pragma unroll
    for (int c = 0; c < 2; ++c)
      if (c * 64 + sub * 8 < p.d) {
        const __nv_bfloat162 *o2 = reinterpret_cast<const __nv_bfloat162 *>(&ov[c]);
        const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&gv[c]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 a = __bfloat1622float2(o2[e]), b = __bfloat1622float2(g2[e]);
          acc = fmaf(a.x, b.x, acc);
          acc = fmaf(a.y, b.y, acc);
        }
      }
  }
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (live && sub == 0) {
    const int64_t t = row / p.hq;
    p.delta[(row - t * p.hq) * p.total_q + t] = acc;
  }
}

template <int D>
struct BwdCfg {
  static constexpr int kTile = 128;
  static constexpr int kTileBytes = kTile * D * 2;   // one [128, D] bf16 tile
  // Ring depths.  The operand of the MMA that is issued ahead (K for S in the
  // dQ kernel, Q for S^T in the dK/dV kernel) gets three stages, the other
  // (V, dO) two: a stage is refilled only once the step that frees it has
  // run its accumulating MMAs, and three stages keep that refill off the path
  // of the MMA issued ahead.  Two [128, D] tiles + 3 + 2 stages: 224 KB at D = 128.
  static constexpr int NS3 = 3, NS2 = 2;
  static constexpr int kThreads = 6 * 32;            // 4 softmax warps, producer, MMA
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kSmemBytes = (2 + NS3 + NS2) * kTileBytes + 1024 + 256 + 1024;
};

// The K-major descriptor walk of a [128, D] tile: 32 bytes per K=16 slice,
// then the next 64-column block every fourth slice.
__device__ __forceinline__ uint32_t kmajor_step(int ks) {
  return ((ks + 1) & 3) ? 2u : (uint32_t)((128 * 128 - 96) >> 4);
}

// D[tmem] (+)= A[smem, K-major 128 x D] * B[smem, K-major 128 x D]^T: an
// M = N = 128 product contracted over the D columns of both tiles.
template <int D>
__device__ __forceinline__ void mma_rows_rows(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                              uint32_t idesc) {
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    if (ks == 0) mma_ss_w<0>(d_tmem, a_lo, hi, b_lo, hi, idesc);
    else mma_ss_w<1>(d_tmem, a_lo, hi, b_lo, hi, idesc);
    const uint32_t st = kmajor_step(ks);
    a_lo += st;
    b_lo += st;
  }
}

// D[tmem] (+)= A[tmem, 128 x 128 bf16] * B[smem, MN-major 128 x D]: contracted
// over the 128 rows of the B tile.  acc0 = 0 overwrites D.
__device__ __forceinline__ void mma_tmem_rows(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                              uint32_t idesc, uint32_t acc0) {
#pragma unroll
  for (int ks = 0; ks < 128 / 16; ++ks) {
    mma_ts_w(d_tmem, a_tmem + ks * 8, b_lo, b_hi, idesc, ks > 0 ? 1u : acc0);
    b_lo += (16 * 128) >> 4;
  }
}


// exp(s - LSE) of one (query, key) pair from the raw product <q, k>, with the
// score mod MOD (0 none, 1 ALiBi at distance `dist` = |i' - j|, exact in fp32,
// 2 soft-cap); `dfac` returns ds/du (1 unless soft-capped).  lse2 = LSE * log2(e).
template <int MOD>
__device__ __forceinline__ float bwd_prob(const BwdParams &p, float sraw, float lse2, float dist, float &dfac) {
  if constexpr (MOD == 2) {
    // the soft-capped score as the forward forms it; ds/du = 4 r (1 - r)
    float r;
    const float s2 = softcap_log2_score(ex2(sraw * (2.f * kLog2e * p.softcap_arg)), p.softcap_log2, r);
    dfac = 4.f * r * (1.f - r);
    return ex2(s2 - lse2);
  } else if constexpr (MOD == 1) {
    dfac = 1.f;
    return ex2(fmaf(sraw, p.scale_log2, -fmaf(p.alibi_log2, dist, lse2)));
  } else {
    dfac = 1.f;
    return ex2(fmaf(sraw, p.scale_log2, -lse2));
  }
}

// Block sparsity (fkl_python PR #7, flex commit; the forward's 128 x 128
// block mask): whether block (query tile qb, key tile kb) of head h of
// sequence b is computed.  Blocks outside the mask's extent are not.
__device__ __forceinline__ bool bwd_block_live(const BwdParams &p, int b, int h, int qb, int kb) {
  if (p.block_mask == nullptr) return true;
  if (qb >= p.n_qblk || kb >= p.n_kblk) return false;
  return p.block_mask[((int64_t)(b * p.hq + h) * p.n_qblk + qb) * p.n_kblk + kb] != 0;
}

// The raw step after `raw` (of `n`) whose block is live; n if none.  Every
// role walks the same live steps with its own cursor, so they agree on the
// order without a shared list.  Without a block mask (kernel parameter BM
// false) every block is live and the cursor is raw + 1.
template <class Live>
__device__ __forceinline__ int bwd_next_live(int raw, int n, Live live) {
  ++raw;
  while (raw < n && !live(raw)) ++raw;
  return raw;
}

// Barrier among `count` threads (whole warps) of the CTA, id 1..15.
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ void bwd_tmem_st16(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Loads a [128, D] bf16 tile (rows row0.., head `head`) as D/64 boxes of 64
// columns, 128-byte swizzled, onto barrier `bar`.
template <int D>
__device__ __forceinline__ void bwd_load_tile(uint8_t *dst, const CUtensorMap *tm, uint64_t *bar, int head, int row0) {
#pragma unroll
  for (int cb = 0; cb < D / 64; ++cb)
    tma_load_3d(smem_u32(dst + cb * 128 * 128), tm, smem_u32(bar), cb * 64, head, row0);
}

// ------------------------------------------------------------------- dQ --
// CTA (query tile, q head, sequence).  TMEM: S [0,128), dP [128,256),
// dQ [256, 256+D), dS (bf16) in two 64-column buffers [384,448), [448,512).
// Warps 0-3 own the tile's rows (TMEM lanes), warp 4 loads, warp 5 issues:
//   S(0) dP(0) | S(t+1) once S(t) is read | dP(t+1) once dP(t) is read |
//   dQ += dS(t) K(t)
// so the next tile's contractions run while the rows form dS(t).
template <int D, int MOD, bool BM>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const BwdParams p) {
  using Cfg = BwdCfg<D>;
  constexpr int NSK = Cfg::NS3, NSV = Cfg::NS2, TB = Cfg::kTileBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int qs = __ldg(p.cu_q + b), sq = __ldg(p.cu_q + b + 1) - qs;
  const int ks = __ldg(p.cu_k + b), sk = __ldg(p.cu_k + b + 1) - ks;
  const int q0 = qt * 128;
  if (q0 >= sq) return;
  const int hk = h / p.group;
  // key tiles that rows q0.. of this tile may see
  const int last = min(q0 + 128, sq) - 1;
  const int ip_min = q0 + sk - sq, ip_max = last + sk - sq;
  int lo = 0, hi = sk;
  if (p.causal) hi = min(hi, ip_max + 1);
  if (p.window > 0) {
    lo = max(lo, ip_min - p.window + 1);
    if (!p.causal) hi = min(hi, ip_max + p.window);
  }
  const int klo = lo / 128;
  const int n_raw = hi > lo ? (hi + 127) / 128 - klo : 0;
  // key tiles klo + r, r in [0, n_raw), whose block is live
  auto blk_live = [&](int r) { return !BM || bwd_block_live(p, b, h, qt, klo + r); };
  int n_tiles = 0;
  for (int r = bwd_next_live(-1, n_raw, blk_live); r < n_raw; r = bwd_next_live(r, n_raw, blk_live)) ++n_tiles;
  if (n_tiles == 0) {   // no key visible: dQ = 0
    for (int idx = threadIdx.x; idx < (last - q0 + 1) * (D / 8); idx += blockDim.x) {
      const int r = idx / (D / 8), c = idx - r * (D / 8);
      __nv_bfloat16 *o = p.dq + (int64_t)(qs + q0 + r) * p.dq_stride_t + (int64_t)h * p.dq_stride_h;
      *reinterpret_cast<uint4 *>(o + c * 8) = make_uint4(0, 0, 0, 0);
    }
    return;
  }

  uint8_t *sQ = smem, *sDO = smem + TB, *sK = smem + 2 * TB, *sV = smem + (2 + NSK) * TB;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (2 + NSK + NSV) * TB);
  uint64_t *q_full = bars, *k_full = bars + 1, *k_empty = k_full + NSK, *v_full = k_empty + NSK,
           *v_empty = v_full + NSV, *s_full = v_empty + NSV, *dp_full = s_full + 1, *s_read = dp_full + 1,
           *ds_full = s_read + 1, *dq_done = ds_full + 1, *dp_read = dq_done + 1, *ds_free = dp_read + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ds_free + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);
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
    mbar_init(smem_u32(s_full), 1);
    mbar_init(smem_u32(dp_full), 1);
    mbar_init(smem_u32(s_read), 128);
    mbar_init(smem_u32(ds_full), 128);
    mbar_init(smem_u32(dq_done), 1);
    mbar_init(smem_u32(dp_read), 128);
    mbar_init(smem_u32(ds_free), 1);
    mbar_init(smem_u32(ds_free + 1), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------- producer --
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_do);
      mbar_expect_tx(smem_u32(q_full), 2 * TB);
      bwd_load_tile<D>(sQ, &tm_q, q_full, h, qs + q0);
      bwd_load_tile<D>(sDO, &tm_do, q_full, h, qs + q0);
      // K runs ahead of V (its ring is deeper); issue order K(t), V(t - 1);
      // rk, rv: raw key-tile indices of K(t) and V(t - 1)
      int rk = bwd_next_live(-1, n_raw, blk_live), rv = rk;
      for (int t = 0; t <= n_tiles; ++t) {
        if (t < n_tiles) {
          const int st = t % NSK, row = ks + (klo + rk) * 128;
          rk = bwd_next_live(rk, n_raw, blk_live);
          if (t >= NSK && !mbar_wait(smem_u32(k_empty + st), ((t / NSK) - 1) & 1, abort_flag, p.err)) break;
          mbar_expect_tx(smem_u32(k_full + st), TB);
          bwd_load_tile<D>(sK + st * TB, &tm_k, k_full + st, hk, row);
        }
        if (t >= 1) {
          const int u = t - 1, sv = u % NSV, row = ks + (klo + rv) * 128;
          rv = bwd_next_live(rv, n_raw, blk_live);
          if (u >= NSV && !mbar_wait(smem_u32(v_empty + sv), ((u / NSV) - 1) & 1, abort_flag, p.err)) break;
          mbar_expect_tx(smem_u32(v_full + sv), TB);
          bwd_load_tile<D>(sV + sv * TB, &tm_v, v_full + sv, hk, row);
        }
      }
    }
  } else if (warp == 5) {
    // ----------------------------------------------------------- MMAs --
    if (lane == 0) {
      constexpr uint32_t id_ss = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t id_dq = idesc_bf16_f32(128, D, 0, 1);
      const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint32_t hi_k = (uint32_t)(dq0 >> 32);
      const uint32_t lo_q = (uint32_t)dq0, lo_do = (uint32_t)smem_desc_sw128(smem_u32(sDO), 16, 1024);
      const uint32_t lo_k = (uint32_t)smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint32_t lo_v = (uint32_t)smem_desc_sw128(smem_u32(sV), 16, 1024);
      const uint64_t dkmn = smem_desc_sw128(smem_u32(sK), 128 * 128, 1024);
      const uint32_t lo_kmn = (uint32_t)dkmn, hi_kmn = (uint32_t)(dkmn >> 32);
      const uint32_t tS = tmem, tP = tmem + 128, tQ = tmem + 256, tD = tmem + 384;
      bool ok = mbar_wait(smem_u32(q_full), 0, abort_flag, p.err);
      if (ok) ok = mbar_wait(smem_u32(k_full), 0, abort_flag, p.err);
      if (ok) {
        tc_fence_after();
        mma_rows_rows<D>(tS, lo_q, lo_k, hi_k, id_ss);
        tc_commit(smem_u32(s_full));
        ok = mbar_wait(smem_u32(v_full), 0, abort_flag, p.err);
      }
      if (ok) {
        tc_fence_after();
        mma_rows_rows<D>(tP, lo_do, lo_v, hi_k, id_ss);
        tc_commit(smem_u32(dp_full));
        tc_commit(smem_u32(v_empty));
      }
      for (int t = 0; ok && t < n_tiles; ++t) {
        const int st = t % NSK, nk = (t + 1) % NSK, nv = (t + 1) % NSV;
        const bool more = t + 1 < n_tiles;
        if (more) {
          if (!(ok = mbar_wait(smem_u32(s_read), t & 1, abort_flag, p.err))) break;
          if (!(ok = mbar_wait(smem_u32(k_full + nk), ((t + 1) / NSK) & 1, abort_flag, p.err))) break;
          tc_fence_after();
          mma_rows_rows<D>(tS, lo_q, lo_k + (uint32_t)(nk * (TB >> 4)), hi_k, id_ss);
          tc_commit(smem_u32(s_full));
        }
        if (more) {
          if (!(ok = mbar_wait(smem_u32(dp_read), t & 1, abort_flag, p.err))) break;
          if (!(ok = mbar_wait(smem_u32(v_full + nv), ((t + 1) / NSV) & 1, abort_flag, p.err))) break;
          tc_fence_after();
          mma_rows_rows<D>(tP, lo_do, lo_v + (uint32_t)(nv * (TB >> 4)), hi_k, id_ss);
          tc_commit(smem_u32(dp_full));
          tc_commit(smem_u32(v_empty + nv));
        }
        if (!(ok = mbar_wait(smem_u32(ds_full), t & 1, abort_flag, p.err))) break;
        tc_fence_after();
        mma_tmem_rows(tQ, tD + (uint32_t)((t & 1) * 64), lo_kmn + (uint32_t)(st * (TB >> 4)), hi_kmn, id_dq,
                      t > 0 ? 1u : 0u);
        tc_commit(smem_u32(k_empty + st));
        tc_commit(smem_u32(ds_free + (t & 1)));
      }
      tc_commit(smem_u32(dq_done));
    }
  } else {
    // ------------------------------------------------ rows: P, dS, dQ --
    const int r = threadIdx.x;               // row of the tile == TMEM lane
    const int i = q0 + r;
    const bool row_ok = i < sq;
    const int64_t t_glob = (int64_t)qs + i;
    const float lse = row_ok ? __ldg(p.lse + (int64_t)h * p.total_q + t_glob) : 0.f;
    const float delta = row_ok ? __ldg(p.delta + (int64_t)h * p.total_q + t_glob) : 0.f;
    const bool live = row_ok && lse != -INFINITY;
    const float lse2 = lse * kLog2e;
    const int ip = i + sk - sq;
    // keys [row_jlo, row_jhi) of the sequence that row i sees (empty if none)
    int row_jlo = 0, row_jhi = sk;
    if (p.causal) row_jhi = min(row_jhi, ip + 1);
    if (p.window > 0) {
      row_jlo = max(row_jlo, ip - p.window + 1);
      if (!p.causal) row_jhi = min(row_jhi, ip + p.window);
    }
    if (!live) row_jhi = row_jlo;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t rS = tmem + lane_base, rP = tmem + lane_base + 128, rQ = tmem + lane_base + 256;
    bool ok = true;
    int rt = bwd_next_live(-1, n_raw, blk_live);
    for (int t = 0; t < n_tiles; ++t) {
      const int j0 = (klo + rt) * 128;
      rt = bwd_next_live(rt, n_raw, blk_live);
      ok = mbar_wait(smem_u32(s_full), t & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      float pr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(rS + c * 32, *reinterpret_cast<float(*)[32]>(pr + c * 32));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(smem_u32(s_read));
      // the row's allowed keys are one interval; as tile columns: [elo, ehi)
      const int elo = row_jlo - j0, ehi = row_jhi - j0;
      // P times ds/du (only dS is formed from it here); ALiBi distance
      // |i' - j0 - e| from one integer conversion per tile
      const float dbase = (float)(ip - j0);
#pragma unroll
      for (int e = 0; e < 128; ++e) {
        float df;
        const float x = bwd_prob<MOD>(p, pr[e], lse2, fabsf(dbase - (float)e), df);
        pr[e] = (e >= elo && e < ehi) ? x * df : 0.f;
      }
      ok = mbar_wait(smem_u32(dp_full), t & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      // dS in two halves of 64 columns; once the second half of dP is in
      // registers the MMA warp may overwrite dP with the next tile's
      uint32_t ds[64];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float dp[64];
        tmem_ld32(rP + hf * 64, *reinterpret_cast<float(*)[32]>(dp));
        tmem_ld32(rP + hf * 64 + 32, *reinterpret_cast<float(*)[32]>(dp + 32));
        tmem_wait_ld();
        if (hf == 1) {
          tc_fence_before();
          mbar_arrive(smem_u32(dp_read));
        }
#pragma unroll
        for (int e = 0; e < 32; ++e)
          ds[hf * 32 + e] = pack_bf16x2(pr[hf * 64 + 2 * e] * (dp[2 * e] - delta),
                                        pr[hf * 64 + 2 * e + 1] * (dp[2 * e + 1] - delta));
      }
      // dS buffer t % 2 was last read by dQ(t - 2)
      if (t >= 2) {
        ok = mbar_wait(smem_u32(ds_free + (t & 1)), ((t >> 1) - 1) & 1, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      const uint32_t rD = tmem + lane_base + 384 + (uint32_t)((t & 1) * 64);
#pragma unroll
      for (int c = 0; c < 4; ++c) bwd_tmem_st16(rD + c * 16, ds + c * 16);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(ds_full));
    }
    if (ok) {
      ok = mbar_wait(smem_u32(dq_done), 0, abort_flag, p.err);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        __nv_bfloat16 *orow = p.dq + t_glob * p.dq_stride_t + (int64_t)h * p.dq_stride_h;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(rQ + c * 32, o);
          tmem_wait_ld();
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(o[2 * e] * p.scale, o[2 * e + 1] * p.scale);
          if (row_ok) {
            uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

// ----------------------------------------------------------------- dK, dV --
// CTA (key tile, kv head, sequence); it loops over the q heads of the kv
// head's group and, for each, over the query tiles that may see its keys.
// TMEM: S^T [0,128) with P^T (bf16) written over its last 64 columns once S^T
// is in registers, dP^T [128,256) with dS^T (bf16) over its first 64, dV
// [256, 256+D), dK [384, 384+D).  Warps 0-3 own the tile's keys (TMEM lanes)
// and stage each step's LSE and Delta in shared memory; warp 4 loads K and V
// once and then Q (three stages) and dO (two stages) per step; warp 5 issues:
//   S^T(0) dP^T(0) | dV += P^T(s) dO(s) once P^T is stored, S^T(s+1) |
//   dK += dS^T(s) Q(s) once dS^T is stored, dP^T(s+1)
// so dV and the next S^T run while the keys' warps form dS^T(s).
template <int D, int MOD, bool BM>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdParams p) {
  using Cfg = BwdCfg<D>;
  constexpr int NSQ = Cfg::NS3, NSO = Cfg::NS2, TB = Cfg::kTileBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kt = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int qs = __ldg(p.cu_q + b), sq = __ldg(p.cu_q + b + 1) - qs;
  const int ks = __ldg(p.cu_k + b), sk = __ldg(p.cu_k + b + 1) - ks;
  const int kj0 = kt * 128;
  if (kj0 >= sk) return;
  const int kl = min(kj0 + 128, sk) - 1;
  // query rows that may see keys kj0..kl: i' = i + sk - sq
  const int off = sk - sq;
  int qlo = 0, qhi = sq;
  if (p.causal) qlo = max(qlo, kj0 - off);
  if (p.window > 0) {
    qhi = min(qhi, kl + p.window - off);
    if (!p.causal) qlo = max(qlo, kj0 - p.window + 1 - off);
  }
  const int tlo = qlo / 128;
  const int nqt = qhi > qlo ? (qhi + 127) / 128 - tlo : 0;
  // raw step r: q head hk * group + r / nqt, query tile tlo + r % nqt; the
  // steps taken are the raw steps whose block is live
  const int n_raw = nqt * p.group;
  auto blk_live = [&](int r) { return !BM || bwd_block_live(p, b, hk * p.group + r / nqt, tlo + r % nqt, kt); };
  int steps = 0;
  for (int r = bwd_next_live(-1, n_raw, blk_live); r < n_raw; r = bwd_next_live(r, n_raw, blk_live)) ++steps;
  if (steps == 0) {   // no query sees these keys: dK = dV = 0
    for (int idx = threadIdx.x; idx < (kl - kj0 + 1) * (D / 8); idx += blockDim.x) {
      const int r = idx / (D / 8), c = idx - r * (D / 8);
      const int64_t tok = (int64_t)ks + kj0 + r;
      __nv_bfloat16 *a = p.dk + tok * p.dk_stride_t + (int64_t)hk * p.dk_stride_h;
      __nv_bfloat16 *v = p.dv + tok * p.dv_stride_t + (int64_t)hk * p.dv_stride_h;
      *reinterpret_cast<uint4 *>(a + c * 8) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4 *>(v + c * 8) = make_uint4(0, 0, 0, 0);
    }
    return;
  }

  uint8_t *sK = smem, *sV = smem + TB, *sQ = smem + 2 * TB, *sDO = smem + (2 + NSQ) * TB;
  float *sStat = reinterpret_cast<float *>(smem + (2 + NSQ + NSO) * TB);   // [2][128]: LSE*log2e, Delta
  uint64_t *bars = reinterpret_cast<uint64_t *>(sStat + 256);
  uint64_t *kv_full = bars, *q_full = bars + 1, *q_empty = q_full + NSQ, *o_full = q_empty + NSQ,
           *o_empty = o_full + NSO, *st_full = o_empty + NSO, *dpt_full = st_full + 1, *st_read = dpt_full + 1,
           *pds_full = st_read + 1, *done = pds_full + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(kv_full), 1);
    for (int s = 0; s < NSQ; ++s) {
      mbar_init(smem_u32(q_full + s), 1);
      mbar_init(smem_u32(q_empty + s), 1);
    }
    for (int s = 0; s < NSO; ++s) {
      mbar_init(smem_u32(o_full + s), 1);
      mbar_init(smem_u32(o_empty + s), 1);
    }
    mbar_init(smem_u32(st_full), 1);
    mbar_init(smem_u32(dpt_full), 1);
    mbar_init(smem_u32(st_read), 128);
    mbar_init(smem_u32(pds_full), 128);
    mbar_init(smem_u32(done), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------- producer --
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_do);
      mbar_expect_tx(smem_u32(kv_full), 2 * TB);
      bwd_load_tile<D>(sK, &tm_k, kv_full, hk, ks + kj0);
      bwd_load_tile<D>(sV, &tm_v, kv_full, hk, ks + kj0);
    }
    // Q runs ahead of dO (its ring is deeper): issue order Q(s), dO(s - 1)
    if (lane == 0) {
      int rq = bwd_next_live(-1, n_raw, blk_live), ro = rq;   // raw steps of Q(s) and dO(s - 1)
      for (int s = 0; s <= steps; ++s) {
        if (s < steps) {
          const int st = s % NSQ, h = hk * p.group + rq / nqt, q0 = (tlo + rq % nqt) * 128;
          rq = bwd_next_live(rq, n_raw, blk_live);
          if (s >= NSQ && !mbar_wait(smem_u32(q_empty + st), ((s / NSQ) - 1) & 1, abort_flag, p.err)) break;
          mbar_expect_tx(smem_u32(q_full + st), TB);
          bwd_load_tile<D>(sQ + st * TB, &tm_q, q_full + st, h, qs + q0);
        }
        if (s >= 1) {
          const int u = s - 1, so = u % NSO, h = hk * p.group + ro / nqt, q0 = (tlo + ro % nqt) * 128;
          ro = bwd_next_live(ro, n_raw, blk_live);
          if (u >= NSO && !mbar_wait(smem_u32(o_empty + so), ((u / NSO) - 1) & 1, abort_flag, p.err)) break;
          mbar_expect_tx(smem_u32(o_full + so), TB);
          bwd_load_tile<D>(sDO + so * TB, &tm_do, o_full + so, h, qs + q0);
        }
      }
    }
  } else if (warp == 5) {
    // ----------------------------------------------------------- MMAs --
    if (lane == 0) {
      constexpr uint32_t id_ss = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t id_acc = idesc_bf16_f32(128, D, 0, 1);
      const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint32_t hi = (uint32_t)(dk0 >> 32), lo_k = (uint32_t)dk0;
      const uint32_t lo_v = (uint32_t)smem_desc_sw128(smem_u32(sV), 16, 1024);
      const uint32_t lo_q = (uint32_t)smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint32_t lo_do = (uint32_t)smem_desc_sw128(smem_u32(sDO), 16, 1024);
      const uint64_t dqmn = smem_desc_sw128(smem_u32(sQ), 128 * 128, 1024);
      const uint32_t lo_qmn = (uint32_t)dqmn, hi_mn = (uint32_t)(dqmn >> 32);
      const uint32_t lo_domn = (uint32_t)smem_desc_sw128(smem_u32(sDO), 128 * 128, 1024);
      const uint32_t tS = tmem, tP = tmem + 128, tV = tmem + 256, tK = tmem + 384;
      bool ok = mbar_wait(smem_u32(kv_full), 0, abort_flag, p.err);
      if (ok) ok = mbar_wait(smem_u32(q_full), 0, abort_flag, p.err);
      if (ok) {
        tc_fence_after();
        mma_rows_rows<D>(tS, lo_k, lo_q, hi, id_ss);
        tc_commit(smem_u32(st_full));
        ok = mbar_wait(smem_u32(o_full), 0, abort_flag, p.err);
      }
      if (ok) {
        tc_fence_after();
        mma_rows_rows<D>(tP, lo_v, lo_do, hi, id_ss);
        tc_commit(smem_u32(dpt_full));
      }
      for (int s = 0; ok && s < steps; ++s) {
        const int sq_ = s % NSQ, so_ = s % NSO, nq = (s + 1) % NSQ, no = (s + 1) % NSO;
        const bool more = s + 1 < steps;
        // P^T(s) is in S^T's last 64 columns (S^T(s) itself already read)
        if (!(ok = mbar_wait(smem_u32(st_read), s & 1, abort_flag, p.err))) break;
        tc_fence_after();
        mma_tmem_rows(tV, tS + 64, lo_domn + (uint32_t)(so_ * (TB >> 4)), hi_mn, id_acc, s > 0 ? 1u : 0u);
        tc_commit(smem_u32(o_empty + so_));
        if (more) {
          if (!(ok = mbar_wait(smem_u32(q_full + nq), ((s + 1) / NSQ) & 1, abort_flag, p.err))) break;
          tc_fence_after();
          mma_rows_rows<D>(tS, lo_k, lo_q + (uint32_t)(nq * (TB >> 4)), hi, id_ss);
          tc_commit(smem_u32(st_full));
        }
        if (!(ok = mbar_wait(smem_u32(pds_full), s & 1, abort_flag, p.err))) break;
        tc_fence_after();
        mma_tmem_rows(tK, tP, lo_qmn + (uint32_t)(sq_ * (TB >> 4)), hi_mn, id_acc, s > 0 ? 1u : 0u);
        tc_commit(smem_u32(q_empty + sq_));
        if (more) {
          if (!(ok = mbar_wait(smem_u32(o_full + no), ((s + 1) / NSO) & 1, abort_flag, p.err))) break;
          tc_fence_after();
          mma_rows_rows<D>(tP, lo_v, lo_do + (uint32_t)(no * (TB >> 4)), hi, id_ss);
          tc_commit(smem_u32(dpt_full));
        }
      }
      tc_commit(smem_u32(done));
    }
  } else {
    // ------------------------------------------ keys: P^T, dS^T, dK, dV --
    const int r = threadIdx.x;               // key of the tile == TMEM lane
    const int j = kj0 + r;
    const bool key_ok = j < sk;
    // queries [key_qlo, key_qhi) of the sequence that see key j: i' = i + off
    int key_qlo = 0, key_qhi = sq;
    if (p.causal) key_qlo = max(key_qlo, j - off);
    if (p.window > 0) {
      key_qhi = min(key_qhi, j + p.window - off);
      if (!p.causal) key_qlo = max(key_qlo, j - p.window + 1 - off);
    }
    if (!key_ok) key_qhi = key_qlo;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t rS = tmem + lane_base, rP = tmem + lane_base + 128;
    bool ok = true;
    const float *stat = sStat;
    // Per-query LSE (log2 units) and Delta of a step, one query per thread;
    // queries past the sequence get LSE = +inf, so that their P is 0.  Loaded
    // a step ahead so that the global-load latency stays off the step.
    auto load_stat = [&](int rs, float &lv, float &dv) {   // rs: raw step
      const int h = hk * p.group + rs / nqt, i = (tlo + rs % nqt) * 128 + r;
      const int64_t at = (int64_t)h * p.total_q + qs + i;
      lv = i < sq ? __ldg(p.lse + at) * kLog2e : INFINITY;
      dv = i < sq ? __ldg(p.delta + at) : 0.f;
    };
    float lv_next, dv_next;
    int rs = bwd_next_live(-1, n_raw, blk_live);   // raw step of step s
    load_stat(rs, lv_next, dv_next);
    for (int s = 0; s < steps; ++s) {
      const int q0 = (tlo + rs % nqt) * 128;
      rs = bwd_next_live(rs, n_raw, blk_live);
      {
        const float lv = lv_next, dv = dv_next;
        if (s + 1 < steps) load_stat(rs, lv_next, dv_next);
        named_bar_sync(1, 128);   // the previous step's reads are done
        sStat[r] = lv;
        sStat[128 + r] = dv;
        named_bar_sync(1, 128);
      }
      // after a failed wait the loop still runs every step's two barriers
      // (no warp may leave while the others wait there), skipping the work
      if (!ok) continue;
      ok = mbar_wait(smem_u32(st_full), s & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; continue; }
      tc_fence_after();
      float pr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(rS + c * 32, *reinterpret_cast<float(*)[32]>(pr + c * 32));
      tmem_wait_ld();
      // the key's allowed queries are one interval; as tile columns: [elo, ehi)
      // (queries past the sequence already have P = 0 through LSE = +inf)
      const int elo = key_qlo - q0, ehi = key_qhi - q0;
      // P^T rounded to bf16 at once (the operand of dV += P^T dO; dS^T is
      // formed from the same rounded values), which halves its registers
      // soft-cap: dS^T is formed from P times ds/du, kept apart in ptk
      uint32_t ppk[64];
      uint32_t ptk[MOD == 2 ? 64 : 1];
      const float dbase = (float)(q0 + off - j);   // ALiBi: |i' - j| = |dbase + e|
#pragma unroll
      for (int e = 0; e < 128; e += 2) {
        float d0, d1;
        const float x0 = bwd_prob<MOD>(p, pr[e], stat[e], fabsf(dbase + (float)e), d0);
        const float x1 = bwd_prob<MOD>(p, pr[e + 1], stat[e + 1], fabsf(dbase + (float)(e + 1)), d1);
        const bool a0 = e >= elo && e < ehi, a1 = e + 1 >= elo && e + 1 < ehi;
        ppk[e >> 1] = pack_bf16x2(a0 ? x0 : 0.f, a1 ? x1 : 0.f);
        if constexpr (MOD == 2) ptk[e >> 1] = pack_bf16x2(a0 ? x0 * d0 : 0.f, a1 ? x1 * d1 : 0.f);
      }
      // P^T over S^T's last 64 columns: dV(s) may start
#pragma unroll
      for (int c = 0; c < 4; ++c) bwd_tmem_st16(rS + 64 + c * 16, ppk + c * 16);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(st_read));
      ok = mbar_wait(smem_u32(dpt_full), s & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; continue; }
      tc_fence_after();
      // dS^T in two halves of 64 columns, each read with one wait; half hf
      // writes dS^T columns [32 hf, 32 hf + 32), all read already
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float dp[64];
        tmem_ld32(rP + hf * 64, *reinterpret_cast<float(*)[32]>(dp));
        tmem_ld32(rP + hf * 64 + 32, *reinterpret_cast<float(*)[32]>(dp + 32));
        tmem_wait_ld();
        uint32_t w[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int q = hf * 64 + 2 * e;
          uint32_t u;
          if constexpr (MOD == 2) u = ptk[q >> 1];
          else u = ppk[q >> 1];
          const float p0 = __uint_as_float(u << 16), p1 = __uint_as_float(u & 0xFFFF0000u);
          w[e] = pack_bf16x2(p0 * (dp[2 * e] - stat[128 + q]), p1 * (dp[2 * e + 1] - stat[128 + q + 1]));
        }
        bwd_tmem_st16(rP + hf * 32, w);
        bwd_tmem_st16(rP + hf * 32 + 16, w + 16);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(pds_full));
    }
    if (ok) {
      ok = mbar_wait(smem_u32(done), 0, abort_flag, p.err);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        const int64_t tok = (int64_t)ks + j;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          const uint32_t src = tmem + lane_base + (which ? 384u : 256u);
          const float f = which ? p.scale : 1.f;
          __nv_bfloat16 *orow = which ? p.dk + tok * p.dk_stride_t + (int64_t)hk * p.dk_stride_h
                                      : p.dv + tok * p.dv_stride_t + (int64_t)hk * p.dv_stride_h;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(src + c * 32, o);
            tmem_wait_ld();
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(o[2 * e] * f, o[2 * e + 1] * f);
            if (key_ok) {
              uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
              for (int v = 0; v < 4; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace fa
