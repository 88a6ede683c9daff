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
  int32_t n_items;      // work items (persistent kernels stride over them)
};

// Block order: for each sequence, for each group of `head_group` heads, query
// tiles from the latest (longest under a causal mask) to the first, the heads
// of the group interleaved.  Concurrent CTAs then share the K/V of a few
// heads through L2, and long tiles start first.  Returns false for padding.
__device__ __forceinline__ bool decode_block(const PrefillParams &p, int item, int &b, int &h, int &qt) {
  unsigned L = (unsigned)item;
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

// e4m3 -> bf16 for two values (exact: every e4m3 value is a normal f16 or
// zero, and every such f16 is a bf16).  The f16 pair is rebiased field-wise:
// bf16 = sign | ((f16 & 0x7fff) >> 3) + (112 << 7) for non-zero magnitudes.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
  uint32_t h;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h) : "r"(two));
  const uint32_t sign = h & 0x80008000u;
  uint32_t mag = ((h & 0x7FFF7FFFu) >> 3) & 0x0FFF0FFFu;
  mag += 0x38003800u & __vcmpne2(mag, 0u);
  return sign | mag;
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

template <int DK, int DV, bool PAGED, bool FP8, int MOD>
struct PrefillCfg {
  static constexpr int NS = (DK <= 64) ? 4 : 2;                 // K/V ring stages
  static constexpr int kQBytes = kBlockM * DK * 2;
  static constexpr int kKBytes = kBlockN * DK * 2;               // bf16 operand tile
  static constexpr int kVBytes = kBlockN * DV * 2;
  // e4m3 tiles are staged (unswizzled, row-major) in the upper half of the
  // bf16 operand buffer they are converted into.
  static constexpr int kK8Off = kKBytes / 2, kV8Off = kVBytes / 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + NS * kKBytes;
  static constexpr int kOffSc = kOffV + NS * kVBytes;            // softmax scales [2][2][128]
  static constexpr int kOffBar = kOffSc + (FP8 ? 2 * 2 * kBlockN * 4 : 0);
  static constexpr int kNumBars = 1 + 4 * NS + 8 + (FP8 ? 2 * NS : 0);
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 64 + 1024;        // + alignment slack
  // Warp roles.  bf16: softmax 0-3, K 4, V 5, MMA 6.  e4m3: softmax 0-3,
  // converters 4-7, K 8, V 9, MMA 10, one idle warp (12 warps = 3 warpgroups
  // so that setmaxnreg can move registers to the softmax warpgroup).
  static constexpr int kWarpK = FP8 ? 8 : 4, kWarpV = FP8 ? 9 : 5, kWarpMMA = FP8 ? 10 : 6;
  static constexpr int kThreads = (FP8 ? 12 : 7) * 32;
  static constexpr int kRegsSoftmax = 232, kRegsProd = 56;       // e4m3 variant only
  static constexpr int kPoolNeeded = 128 * kRegsSoftmax + 128 * 168 + 128 * kRegsProd;
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
  if (!decode_block(p, (int)blockIdx.x, ti.b, ti.h, ti.qt)) return;
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
  uint64_t *k8_full = p_empty + 2;   // [NS] e4m3 staging landed (FP8 only)
  uint64_t *v8_full = k8_full + NS;
  float *sc = reinterpret_cast<float *>(smem + Cfg::kOffSc);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Cfg::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Cfg::kOffMisc + 8);

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    for (int s = 0; s < NS; ++s) {
      // bf16: filled by TMA (one arrive + bytes); e4m3: by the 128 converter threads
      mbar_init(smem_u32(k_full + s), FP8 ? 128 : 1);
      mbar_init(smem_u32(k_empty + s), 1);
      mbar_init(smem_u32(v_full + s), FP8 ? 128 : 1);
      mbar_init(smem_u32(v_empty + s), 1);
      if (FP8) {
        mbar_init(smem_u32(k8_full + s), 1);
        mbar_init(smem_u32(v8_full + s), 1);
      }
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
  if (warp == Cfg::kWarpMMA) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // e4m3 variant: the host launches it only when the launch register count
  // makes kPoolNeeded fit the CTA's pool (see the launcher).
  if (FP8 && warp >= 8) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::kRegsProd));

  if (warp == Cfg::kWarpK) {
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
        if constexpr (FP8) {
          // e4m3 rows (DK bytes each) into the upper half of the operand buffer
          uint64_t *bar = k8_full + st;
          mbar_expect_tx(smem_u32(bar), kBlockN * DK);
          uint8_t *dst = sK + st * Cfg::kKBytes + Cfg::kK8Off;
          if constexpr (PAGED) {
            const int32_t *bt = p.block_table + (int64_t)ti.b * p.bt_stride;
            for (int pg = 0; pg < p.pages_per_tile; ++pg) {
              const int key0 = kt * kBlockN + pg * p.rows_per_box;
              const int page = key0 < ti.sk ? __ldg(bt + (key0 >> p.page_shift)) : -1;
              tma_load_4d(smem_u32(dst + pg * p.rows_per_box * DK), &tm_k, smem_u32(bar), 0, ti.hk,
                          key0 & (p.page_size - 1), page);
            }
          } else {
            tma_load_3d(smem_u32(dst), &tm_k, smem_u32(bar), 0, ti.hk, ti.k_row0 + kt * kBlockN);
          }
          continue;
        }
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
  } else if (warp == Cfg::kWarpV) {
    // ---------------------------------------------------- producer: V --
    if (lane == 0) {
      prefetch_tmap(&tm_v);
      int it = 0;
      for (int kt = first_kt; kt < ti.kt_hi; kt = next_tile<Cfg>(p, ti, kt), ++it) {
        const int st = it % NS;
        const uint32_t ph = (it / NS) & 1;
        if (it >= NS && !mbar_wait(smem_u32(v_empty + st), ph ^ 1, abort_flag, p.err)) break;
        if constexpr (FP8) {
          uint64_t *bar = v8_full + st;
          mbar_expect_tx(smem_u32(bar), kBlockN * DV);
          uint8_t *dst = sV + st * Cfg::kVBytes + Cfg::kV8Off;
          if constexpr (PAGED) {
            const int32_t *bt = p.block_table + (int64_t)ti.b * p.bt_stride;
            for (int pg = 0; pg < p.pages_per_tile; ++pg) {
              const int key0 = kt * kBlockN + pg * p.rows_per_box;
              const int page = key0 < ti.sk ? __ldg(bt + (key0 >> p.page_shift)) : -1;
              tma_load_4d(smem_u32(dst + pg * p.rows_per_box * DV), &tm_v, smem_u32(bar), 0, ti.hk,
                          key0 & (p.page_size - 1), page);
            }
          } else {
            tma_load_3d(smem_u32(dst), &tm_v, smem_u32(bar), 0, ti.hk, ti.k_row0 + kt * kBlockN);
          }
          continue;
        }
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
  } else if (FP8 && warp >= 4 && warp < 8) {
    // --------------------------------------------- e4m3 -> bf16 converters --
    // Each tile: read the staged e4m3 rows into registers (all 128 threads),
    // sync, then write exact bf16 into the 128-byte-swizzled operand layout
    // that the MMA reads (the staging area is overwritten, hence the sync).
    const int c = threadIdx.x - 128;
    int it = 0;
    bool ok = true;
    for (int kt = first_kt; ok && kt < ti.kt_hi; kt = next_tile<Cfg>(p, ti, kt), ++it) {
      const int st = it % NS;
      const uint32_t ph = (it / NS) & 1;
#pragma unroll
      for (int opnd = 0; opnd < 2; ++opnd) {
        const int D = opnd == 0 ? DK : DV;
        constexpr int kMaxChunks = (DK > DV ? DK : DV) / 16;     // 16-byte e4m3 chunks per thread
        uint8_t *buf = opnd == 0 ? sK + st * Cfg::kKBytes : sV + st * Cfg::kVBytes;
        const uint8_t *stage = buf + (opnd == 0 ? Cfg::kK8Off : Cfg::kV8Off);
        ok = mbar_wait(smem_u32((opnd == 0 ? k8_full : v8_full) + st), ph, abort_flag, p.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const int per_row = D / 16;
        // V rows are scaled here, in fp32, before their single rounding: the
        // V operand is f16 RNE(e4m3(v) * v_scale).  (K keeps e4m3(k) exactly
        // as bf16; k_scale multiplies S in fp32 in the softmax.)
        float vsr[kMaxChunks];
        if (opnd == 1) {
          const int32_t *bt = PAGED ? p.block_table + (int64_t)ti.b * p.bt_stride : nullptr;
#pragma unroll
          for (int q = 0; q < kMaxChunks; ++q) {
            vsr[q] = 0.f;
            if (q < per_row) {
              const int key = kt * kBlockN + (c + 128 * q) / per_row;
              if (key < ti.sk) {
                int64_t tok;
                if constexpr (PAGED) {
                  const int page = __ldg(bt + (key >> p.page_shift));
                  tok = (int64_t)page * p.page_size + (key & (p.page_size - 1));
                } else {
                  tok = (int64_t)ti.k_row0 + key;
                }
                vsr[q] = __ldg(p.v_scale + tok * p.hkv + ti.hk);
              }
            }
          }
        }
        uint4 raw[kMaxChunks];
#pragma unroll
        for (int q = 0; q < kMaxChunks; ++q)
          if (q < per_row) raw[q] = *reinterpret_cast<const uint4 *>(stage + (size_t)(c + 128 * q) * 16);
        named_bar_sync(2, 128);
#pragma unroll
        for (int q = 0; q < kMaxChunks; ++q) {
          if (q >= per_row) break;
          const int idx = c + 128 * q;
          const int row = idx / per_row, ch = idx - row * per_row;   // 16 dims starting at 16*ch
          const uint32_t w[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
          uint32_t o[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            o[2 * k] = e4m3x2_to_bf16x2(w[k] & 0xFFFFu);
            o[2 * k + 1] = e4m3x2_to_bf16x2(w[k] >> 16);
          }
          if (opnd == 1) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              o[k] = pack_f16x2(__uint_as_float(o[k] << 16) * vsr[q], __uint_as_float(o[k] & 0xFFFF0000u) * vsr[q]);
          }
          const int d0 = ch * 16, cb = d0 >> 6, c8 = (d0 & 63) >> 3;
          uint8_t *blk = buf + cb * kBlockN * 128 + row * 128;
          *reinterpret_cast<uint4 *>(blk + (((c8) ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4 *>(blk + (((c8 + 1) ^ (row & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_u32((opnd == 0 ? k_full : v_full) + st));
        named_bar_sync(2, 128);   // staging of the next operand may reuse registers only
      }
    }
  } else if (warp == Cfg::kWarpMMA) {
    // ------------------------------------------------------- MMA issuer --
    constexpr uint32_t idesc_qk = idesc_bf16_f32(kBlockM, kBlockN, 0, 0);
    // e4m3 K/V: PV runs on f16 operands (P and the scaled V), whose 11-bit
    // mantissas keep the two extra roundings of that path well below bf16's.
    constexpr uint32_t idesc_pv = FP8 ? idesc_f16_f32(kBlockM, DV, 0, 1) : idesc_bf16_f32(kBlockM, DV, 0, 1);
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
    if constexpr (FP8) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::kRegsSoftmax));
    const int r = threadIdx.x;               // row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int i = ti.q0 + r;                 // sequence-local query row
    const int ip = i + ti.sk - ti.sq;        // bottom-right aligned position
    float m_ref = -INFINITY;                 // reference max (scaled log2 units)
    float l = 0.f;
    int it = 0;
    bool ok = true;
    const int32_t *btab = PAGED ? p.block_table + (int64_t)ti.b * p.bt_stride : nullptr;
    for (int kt = first_kt; kt < ti.kt_hi; kt = next_tile<Cfg>(p, ti, kt), ++it) {
      const int sb = it & 1;
      float *ksc = sc + (it & 1) * 2 * kBlockN;   // k scales of this tile's keys
      if constexpr (FP8) {
        // Per-token k scales of the tile's 128 keys: thread r fetches key j0 + r
        // (0 past the sequence end), shared through a softmax-only barrier.
        const int key = kt * kBlockN + r;
        float ks = 0.f;
        if (key < ti.sk) {
          int64_t tok;
          if constexpr (PAGED) {
            const int page = __ldg(btab + (key >> p.page_shift));
            tok = (int64_t)page * p.page_size + (key & (p.page_size - 1));
          } else {
            tok = (int64_t)ti.k_row0 + key;
          }
          ks = __ldg(p.k_scale + tok * p.hkv + ti.hk);
        }
        ksc[r] = ks;
        named_bar_sync(1, kBlockM);
      }
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
      if constexpr (FP8) {
        // S_ij = <q_i, e4m3(k_j)> * k_scale_j  (scale folded after the MMA)
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 k4 = *reinterpret_cast<const float4 *>(ksc + c * 32 + e);
            s[c][e] *= k4.x;
            s[c][e + 1] *= k4.y;
            s[c][e + 2] *= k4.z;
            s[c][e + 3] *= k4.w;
          }
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
          pk[c >> 1][(c & 1) * 16 + (e >> 1)] = FP8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
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
  if (warp == Cfg::kWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace fa
