// fa_prefill.cuh -- tcgen05/TMEM/TMA FlashAttention forward kernel for sm_103a.
//
// One CTA computes one (sequence b, query head h, 128-row query tile).  It
// walks the key tiles of 128 keys that the masks leave, and for each:
//   S = Q K^T            tcgen05.mma, bf16 operands from shared memory, fp32 in TMEM
//   online softmax       one thread per query row: running max m, running sum l
//   O += P V             tcgen05.mma, P (bf16) from TMEM, V from shared memory
// and finally writes O / l as bf16 and LSE = (m + log2 l) * ln 2.
//
// The method is the tiled online-softmax forward of RL-Kernel PR #237 ("SM90
// TMA + mma.sync FlashAttention": TMA loads, QK^T, softmax, PV, LSE export) and
// FlyDSL PR #1066 (paged KV via block_table, lazy O rescaling with a threshold
// of 8 in scaled log2 units, logit scale folded into the max subtraction).
// Here the contractions run on the fifth-generation tensor cores with the
// accumulators in tensor memory instead of registers.
//
// Warp roles (224 threads):
//   warps 0-3  softmax: thread r owns TMEM lane r = query row r of S and O.
//   warp 4     producer: Q tile and K tiles by TMA (page gather when paged).
//   warp 5     producer: V tiles by TMA; e4m3 staging when the cache is fp8.
//   warp 6     allocates TMEM and issues every tcgen05.mma (one lane).
// With an e4m3 cache, warps 7-10 convert staged e4m3 tiles to bf16 operands.
//
// Pipelines (all mbarriers; each wait is bounded, see mbar_wait):
//   K/V shared-memory rings of NS stages (full: TMA -> MMA, empty: MMA -> TMA)
//   S double buffer in TMEM  (s_full: MMA -> softmax, s_free: softmax -> MMA)
//   P double buffer in TMEM  (p_full: softmax -> MMA, p_empty: MMA -> softmax)
// MMA issue order: QK_0, QK_1, PV_0, QK_2, PV_1, ... so that the tensor core
// computes S_{j+1} while the softmax warps work on S_j.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kBlockM = 128;   // query rows per tile (MMA M)
constexpr int kBlockN = 128;   // keys per tile (MMA N of QK^T, K of PV)
constexpr float kRescaleThreshold = 8.0f;   // lazy O rescale, scaled log2 units

struct PrefillParams {
  const int32_t *cu_q;
  const int32_t *cu_k;
  const int32_t *block_table;   // [B, bt_stride] or null
  int64_t bt_stride;
  const float *k_scale;         // per token and kv head (e4m3 only)
  const float *v_scale;
  __nv_bfloat16 *out;
  int64_t out_stride_t, out_stride_h;   // elements
  float *lse;                   // [Hq, T_q] or null
  int64_t total_q;
  const uint8_t *block_mask;    // [B*Hq, n_qblk, n_kblk] or null
  int32_t n_qblk, n_kblk;
  int32_t num_seqs, hq, hkv, group;
  int32_t page_size, page_shift, pages_per_tile, rows_per_box;
  int32_t n_qtiles;
  int32_t causal, window;
  float scale_log2;     // softmax_scale * log2(e)
  float softcap_arg;    // softmax_scale / cap
  float softcap_log2;   // cap * log2(e)
  float alibi_log2;     // slope * log2(e)
  int *err;             // device error word
  int32_t head_group;   // heads interleaved per group in the block order
  int32_t n_hgroups;    // ceil(hq / head_group)
};

// Block order: for each sequence, for each group of `head_group` heads, query
// tiles from the latest (longest under a causal mask) to the first, the heads
// of the group interleaved.  Concurrent CTAs then share the K/V of a few
// heads through L2, and long tiles start first.  Returns false for padding.
__device__ __forceinline__ bool decode_block(const PrefillParams &p, int &b, int &h, int &qt) {
  unsigned L = blockIdx.x;
  const int g_in = (int)(L % (unsigned)p.head_group);
  L /= (unsigned)p.head_group;
  const int pr = (int)(L % (unsigned)p.n_qtiles);
  L /= (unsigned)p.n_qtiles;
  const int hg = (int)(L % (unsigned)p.n_hgroups);
  b = (int)(L / (unsigned)p.n_hgroups);
  h = hg * p.head_group + g_in;
  qt = p.n_qtiles - 1 - pr;
  return h < p.hq;
}

template <int DK, int DV, bool PAGED, bool FP8, int MOD>
struct PrefillCfg {
  static constexpr int NS = (DK <= 64) ? 4 : 2;                 // K/V ring stages
  static constexpr int kQBytes = kBlockM * DK * 2;
  static constexpr int kKBytes = kBlockN * DK * 2;               // bf16 operand tile
  static constexpr int kVBytes = kBlockN * DV * 2;
  static constexpr int kK8Bytes = FP8 ? kBlockN * DK : 0;        // e4m3 staging tile
  static constexpr int kV8Bytes = FP8 ? kBlockN * DV : 0;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + NS * kKBytes;
  static constexpr int kOffK8 = kOffV + NS * kVBytes;
  static constexpr int kOffV8 = kOffK8 + NS * kK8Bytes;
  static constexpr int kOffKs = kOffV8 + NS * kV8Bytes;          // k scales [NS][128]
  static constexpr int kOffVs = kOffKs + (FP8 ? NS * kBlockN * 4 : 0);
  static constexpr int kOffBar = kOffVs + (FP8 ? NS * kBlockN * 4 : 0);
  static constexpr int kNumBars = 1 + 4 * NS + 8 + (FP8 ? 4 * NS : 0);
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 64 + 1024;        // + alignment slack
  static constexpr int kSoftmaxWarps = 4;
  static constexpr int kConvWarps = FP8 ? 4 : 0;
  static constexpr int kThreads = (7 + kConvWarps) * 32;
  // TMEM columns
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP0 = 384, kColP1 = 448;
  static_assert(DV <= 128, "O occupies 128 TMEM columns at most");
  static_assert(DK % 64 == 0 && DV % 64 == 0, "head dims are multiples of 64");
};

// Per-CTA work description shared by all roles.
struct TileInfo {
  int b, h, hk, qt;
  int q0;           // first query row (sequence-local)
  int sq, sk;       // lengths
  int q_row0;       // global token index of row q0
  int k_row0;       // global row of key 0 (packed layout)
  int kt_lo, kt_hi; // key tile range [kt_lo, kt_hi)
  int ip_min, ip_max;
};

template <typename Cfg>
__device__ __forceinline__ bool tile_active(const PrefillParams &p, const TileInfo &ti, int kt) {
  if (p.block_mask == nullptr) return true;
  if (kt >= p.n_kblk || ti.qt >= p.n_qblk) return false;
  int64_t idx = ((int64_t)(ti.b * p.hq + ti.h) * p.n_qblk + ti.qt) * p.n_kblk + kt;
  return p.block_mask[idx] != 0;
}

template <typename Cfg>
__device__ __forceinline__ int next_tile(const PrefillParams &p, const TileInfo &ti, int kt) {
  ++kt;
  while (kt < ti.kt_hi && !tile_active<Cfg>(p, ti, kt)) ++kt;
  return kt;
}

template <int DK, int DV, bool PAGED, bool FP8, int MOD>
__global__ void __launch_bounds__(PrefillCfg<DK, DV, PAGED, FP8, MOD>::kThreads, 1)
    fa_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using Cfg = PrefillCfg<DK, DV, PAGED, FP8, MOD>;
  constexpr int NS = Cfg::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ------------------------------------------------------------ work tile --
  TileInfo ti;
  if (!decode_block(p, ti.b, ti.h, ti.qt)) return;
  ti.hk = ti.h / p.group;
  {
    const int qa = __ldg(p.cu_q + ti.b), qb = __ldg(p.cu_q + ti.b + 1);
    const int ka = __ldg(p.cu_k + ti.b), kb = __ldg(p.cu_k + ti.b + 1);
    ti.sq = qb - qa;
    ti.sk = kb - ka;
    ti.q_row0 = qa + ti.qt * kBlockM;
    ti.k_row0 = ka;
  }
  ti.q0 = ti.qt * kBlockM;
  if (ti.q0 >= ti.sq) return;   // no rows in this tile
  {
    const int last = min(ti.q0 + kBlockM, ti.sq) - 1;
    ti.ip_min = ti.q0 + ti.sk - ti.sq;
    ti.ip_max = last + ti.sk - ti.sq;
    int lo = 0, hi = ti.sk;
    if (p.causal) hi = min(hi, ti.ip_max + 1);
    if (p.window > 0) {
      lo = max(lo, ti.ip_min - p.window + 1);
      if (!p.causal) hi = min(hi, ti.ip_max + p.window);
    }
    if (hi <= lo) {
      ti.kt_lo = 0;
      ti.kt_hi = 0;
    } else {
      ti.kt_lo = lo / kBlockN;
      ti.kt_hi = (hi + kBlockN - 1) / kBlockN;
    }
  }
  int first_kt = ti.kt_lo;
  if (first_kt < ti.kt_hi && !tile_active<Cfg>(p, ti, first_kt)) first_kt = next_tile<Cfg>(p, ti, first_kt);
  int n_tiles = 0;
  for (int kt = first_kt; kt < ti.kt_hi; kt = next_tile<Cfg>(p, ti, kt)) ++n_tiles;

  if (n_tiles == 0) {
    // Every row of this tile has an empty key set: out = 0, LSE = -inf.
    for (int r = threadIdx.x; r < kBlockM; r += blockDim.x) {
      if (ti.q0 + r >= ti.sq) break;
      const int64_t t = (int64_t)ti.q_row0 + r;
      __nv_bfloat16 *o = p.out + t * p.out_stride_t + (int64_t)ti.h * p.out_stride_h;
      for (int d = 0; d < DV; d += 8) *reinterpret_cast<uint4 *>(o + d) = make_uint4(0, 0, 0, 0);
      if (p.lse) p.lse[(int64_t)ti.h * p.total_q + t] = -INFINITY;
    }
    return;
  }

  // ----------------------------------------------------------- shared mem --
  uint8_t *sQ = smem + Cfg::kOffQ;
  uint8_t *sK = smem + Cfg::kOffK;
  uint8_t *sV = smem + Cfg::kOffV;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
  uint64_t *q_full = bars + 0;
  uint64_t *k_full = bars + 1;
  uint64_t *k_empty = k_full + NS;
  uint64_t *v_full = k_empty + NS;
  uint64_t *v_empty = v_full + NS;
  uint64_t *s_full = v_empty + NS;   // [2]
  uint64_t *s_free = s_full + 2;     // [2]
  uint64_t *p_full = s_free + 2;     // [2]
  uint64_t *p_empty = p_full + 2;    // [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 8);

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(k_full + s), 1);
      mbar_init(smem_u32(k_empty + s), 1);
      mbar_init(smem_u32(v_full + s), 1);
      mbar_init(smem_u32(v_empty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(s_full + s), 1);
      mbar_init(smem_u32(s_free + s), kBlockM);
      mbar_init(smem_u32(p_full + s), kBlockM);
      mbar_init(smem_u32(p_empty + s), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 6) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------ producer: Q and K --
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      mbar_expect_tx(smem_u32(q_full), Cfg::kQBytes);
#pragma unroll
      for (int cb = 0; cb < DK / 64; ++cb)
        tma_load_3d(smem_u32(sQ + cb * kBlockM * 128), &tm_q, smem_u32(q_full), cb * 64, ti.h, ti.q_row0);
      int it = 0;
      for (int kt = first_kt; kt < ti.kt_hi; kt = next_tile<Cfg>(p, ti, kt), ++it) {
        const int st = it % NS;
        const uint32_t ph = (it / NS) & 1;
        if (it >= NS && !mbar_wait(smem_u32(k_empty + st), ph ^ 1, abort_flag, p.err)) break;
        mbar_expect_tx(smem_u32(k_full + st), Cfg::kKBytes);
        uint8_t *dst = sK + st * Cfg::kKBytes;
        if constexpr (PAGED) {
          const int32_t *bt = p.block_table + (int64_t)ti.b * p.bt_stride;
          for (int pg = 0; pg < p.pages_per_tile; ++pg) {
            const int key0 = kt * kBlockN + pg * p.rows_per_box;
            const int page = key0 < ti.sk ? __ldg(bt + (key0 >> p.page_shift)) : -1;
            const int slot = key0 & (p.page_size - 1);
#pragma unroll
            for (int cb = 0; cb < DK / 64; ++cb)
              tma_load_4d(smem_u32(dst + cb * kBlockN * 128 + pg * p.rows_per_box * 128), &tm_k,
                          smem_u32(k_full + st), cb * 64, ti.hk, slot, page);
          }
        } else {
#pragma unroll
          for (int cb = 0; cb < DK / 64; ++cb)
            tma_load_3d(smem_u32(dst + cb * kBlockN * 128), &tm_k, smem_u32(k_full + st), cb * 64, ti.hk,
                        ti.k_row0 + kt * kBlockN);
        }
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------- producer: V --
    if (lane == 0) {
      prefetch_tmap(&tm_v);
      int it = 0;
      for (int kt = first_kt; kt < ti.kt_hi; kt = next_tile<Cfg>(p, ti, kt), ++it) {
        const int st = it % NS;
        const uint32_t ph = (it / NS) & 1;
        if (it >= NS && !mbar_wait(smem_u32(v_empty + st), ph ^ 1, abort_flag, p.err)) break;
        mbar_expect_tx(smem_u32(v_full + st), Cfg::kVBytes);
        uint8_t *dst = sV + st * Cfg::kVBytes;
        if constexpr (PAGED) {
          const int32_t *bt = p.block_table + (int64_t)ti.b * p.bt_stride;
          for (int pg = 0; pg < p.pages_per_tile; ++pg) {
            const int key0 = kt * kBlockN + pg * p.rows_per_box;
            const int page = key0 < ti.sk ? __ldg(bt + (key0 >> p.page_shift)) : -1;
            const int slot = key0 & (p.page_size - 1);
#pragma unroll
            for (int cb = 0; cb < DV / 64; ++cb)
              tma_load_4d(smem_u32(dst + cb * kBlockN * 128 + pg * p.rows_per_box * 128), &tm_v,
                          smem_u32(v_full + st), cb * 64, ti.hk, slot, page);
          }
        } else {
#pragma unroll
          for (int cb = 0; cb < DV / 64; ++cb)
            tma_load_3d(smem_u32(dst + cb * kBlockN * 128), &tm_v, smem_u32(v_full + st), cb * 64, ti.hk,
                        ti.k_row0 + kt * kBlockN);
        }
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------------- MMA issuer --
    constexpr uint32_t idesc_qk = idesc_bf16_f32(kBlockM, kBlockN, 0, 0);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kBlockM, DV, 0, 1);
    const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
    bool ok = mbar_wait(smem_u32(q_full), 0, abort_flag, p.err);

    auto issue_qk = [&](int it) -> bool {
      const int st = it % NS, sb = it & 1;
      if (!mbar_wait(smem_u32(k_full + st), (it / NS) & 1, abort_flag, p.err)) return false;
      if (it >= 2 && !mbar_wait(smem_u32(s_free + sb), ((it - 2) >> 1) & 1, abort_flag, p.err)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t d = tmem + (sb ? Cfg::kColS1 : Cfg::kColS0);
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks) {
          const uint32_t off = (ks >> 2) * (kBlockM * 128) + (ks & 3) * 32;
          const uint64_t da = smem_desc_sw128(sQa + off, 16, 1024);
          const uint64_t db = smem_desc_sw128(sKa + st * Cfg::kKBytes + off, 16, 1024);
          mma_ss(d, da, db, idesc_qk, ks > 0);
        }
        tc_commit(smem_u32(s_full + sb));
        tc_commit(smem_u32(k_empty + st));
      }
      __syncwarp();
      return true;
    };
    auto issue_pv = [&](int it, int kt) -> bool {
      const int st = it % NS, pb = it & 1;
      if (!mbar_wait(smem_u32(v_full + st), (it / NS) & 1, abort_flag, p.err)) return false;
      // Keys past the sequence end may hold anything (NaN-poisoned page
      // slots); P is 0 there, but 0 * NaN is NaN, so clear those V rows.
      const int valid = ti.sk - kt * kBlockN;
      if (valid < kBlockN) {
        uint8_t *vt = sV + st * Cfg::kVBytes;
#pragma unroll
        for (int cb = 0; cb < DV / 64; ++cb) {
          uint4 *z = reinterpret_cast<uint4 *>(vt + cb * kBlockN * 128 + valid * 128);
          const int n16 = (kBlockN - valid) * 8;
          for (int i = lane; i < n16; i += 32) z[i] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (!mbar_wait(smem_u32(p_full + pb), (it >> 1) & 1, abort_flag, p.err)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t a = tmem + (pb ? Cfg::kColP1 : Cfg::kColP0);
#pragma unroll
        for (int ks = 0; ks < kBlockN / 16; ++ks) {
          const uint64_t db = smem_desc_sw128(sVa + st * Cfg::kVBytes + ks * 16 * 128, kBlockN * 128, 1024);
          mma_ts(tmem + Cfg::kColO, a + ks * 8, db, idesc_pv, (it > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(p_empty + pb));
        tc_commit(smem_u32(v_empty + st));
      }
      __syncwarp();
      return true;
    };

    if (ok) ok = issue_qk(0);
    int it = 0;
    for (int kt = first_kt; ok && kt < ti.kt_hi; ++it) {
      const int kn = next_tile<Cfg>(p, ti, kt);
      if (it + 1 < n_tiles) ok = issue_qk(it + 1);
      if (ok) ok = issue_pv(it, kt);
      kt = kn;
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------- softmax --
    const int r = threadIdx.x;               // row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int i = ti.q0 + r;                 // sequence-local query row
    const int ip = i + ti.sk - ti.sq;        // bottom-right aligned position
    float m_ref = -INFINITY;                 // reference max (scaled log2 units)
    float l = 0.f;
    int it = 0;
    bool ok = true;
    for (int kt = first_kt; kt < ti.kt_hi; kt = next_tile<Cfg>(p, ti, kt), ++it) {
      const int sb = it & 1;
      ok = mbar_wait(smem_u32(s_full + sb), (it >> 1) & 1, abort_flag, p.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      float s[4][32];
      const uint32_t sa = tmem + lane_base + (sb ? Cfg::kColS1 : Cfg::kColS0);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(sa + c * 32, s[c]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(smem_u32(s_free + sb));

      // Scores in scaled log2 units, with score mods and masks.
      const int j0 = kt * kBlockN;
      bool need_mask = (j0 + kBlockN > ti.sk);
      if (p.causal && j0 + kBlockN - 1 > ti.ip_min) need_mask = true;
      if (p.window > 0) {
        if (j0 < ti.ip_max - p.window + 1) need_mask = true;
        if (!p.causal && j0 + kBlockN - 1 > ti.ip_min + p.window - 1) need_mask = true;
      }
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int j = j0 + c * 32 + e;
          float x;
          if constexpr (MOD == 2) {
            // soft-cap on the scaled score: cap * tanh(scale * qk / cap)
            const float t = s[c][e] * p.softcap_arg;
            const float at = fabsf(t);
            const float em = ex2(-2.f * kLog2e * at);           // exp(-2|t|)
            const float th = __fdividef(1.f - em, 1.f + em);
            x = copysignf(th, t) * p.softcap_log2;
          } else {
            x = s[c][e] * p.scale_log2;
          }
          if constexpr (MOD == 1) x -= p.alibi_log2 * (float)abs(ip - j);
          if (need_mask) {
            bool allowed = j < ti.sk;
            if (p.causal) allowed = allowed && (j <= ip);
            if (p.window > 0) allowed = allowed && (p.causal ? (ip - j < p.window) : (abs(ip - j) < p.window));
            x = allowed ? x : -INFINITY;
          }
          s[c][e] = x;
          tmax = fmaxf(tmax, x);
        }
      }
      // Lazy rescaling: keep the reference max unless the tile max exceeds it
      // by more than the threshold (p <= 2^8 otherwise).  The decision is made
      // per row; TMEM traffic is warp-wide, so a warp rescales when any of its
      // rows must (alpha = 1 for the others).
      const float m_new = fmaxf(m_ref, tmax);
      const bool need = m_new > m_ref + kRescaleThreshold;
      const bool warp_need = __any_sync(0xffffffffu, need);
      float alpha = 1.f;
      if (need) {
        alpha = ex2(m_ref - m_new);   // 0 when m_ref = -inf (O row is still 0)
        l *= alpha;
        m_ref = m_new;
      }
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      uint32_t pk[2][32];
      float lsum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = ex2(s[c][e] - m_use);
          const float p1 = ex2(s[c][e + 1] - m_use);
          lsum += p0 + p1;
          pk[c >> 1][(c & 1) * 16 + (e >> 1)] = pack_bf16x2(p0, p1);
        }
      }
      l += lsum;
      if (warp_need && it > 0) {
        // O must hold PV_{it-1} before it is rescaled; PV_it waits for p_full.
        const int pb1 = (it - 1) & 1;
        ok = mbar_wait(smem_u32(p_empty + pb1), ((it - 1) >> 1) & 1, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const uint32_t oa = tmem + lane_base + Cfg::kColO;
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
        tmem_wait_st();
      }
      const int pb = it & 1;
      if (it >= 2) {
        ok = mbar_wait(smem_u32(p_empty + pb), ((it - 2) >> 1) & 1, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
      tc_fence_after();
      const uint32_t pa = tmem + lane_base + (pb ? Cfg::kColP1 : Cfg::kColP0);
      tmem_st32(pa, pk[0]);
      tmem_st32(pa + 32, pk[1]);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(p_full + pb));
    }

    // -------------------------------------------------------- epilogue --
    if (ok) {
      const int last = n_tiles - 1;
      ok = mbar_wait(smem_u32(p_empty + (last & 1)), (last >> 1) & 1, abort_flag, p.err);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const bool row_ok = i < ti.sq;
      const int64_t t = (int64_t)ti.q_row0 + r;
      __nv_bfloat16 *orow = p.out + t * p.out_stride_t + (int64_t)ti.h * p.out_stride_h;
      const bool has = l > 0.f;
      const float inv_l = has ? 1.f / l : 0.f;
      const uint32_t oa = tmem + lane_base + Cfg::kColO;
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        float o[32];
        tmem_ld32(oa + c * 32, o);   // warp-wide: every lane takes part
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
      if (row_ok && p.lse) p.lse[(int64_t)ti.h * p.total_q + t] = has ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 6) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace fa
