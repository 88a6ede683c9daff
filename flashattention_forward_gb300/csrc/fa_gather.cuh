// fa_gather.cuh -- K/V rows of a paged cache gathered with 16-byte cp.async
// copies, for pages that hold fewer than 16 keys.
//
// The paged kernels normally land a K or V tile with one TMA box per page
// piece.  A box of a 128-byte-swizzled block must start on a 1024-byte swizzle
// atom, i.e. cover 8 rows of 128 bytes, and the byte staging boxes 16 rows of
// 64 bytes, so pages of 1, 2, 4 (and, for bytes, 8) keys cannot be boxed.
// Pages of one key are the lookup-bound case of the paged layout (FlyDSL
// PR #1066, the page-size note: page 1 against page 16); there every key row is
// fetched by its own page-table read and row copy, which is what this does:
// one warp, one or four lanes per key row, 16 bytes per copy, written
// straight into the layout the consumers read (the swizzle is applied by
// address, as TMA would).
//
// Completion: the copies of one ring slot form one cp.async group.  After the
// next slot's group is committed, each lane waits for all but that newest
// group, makes the bytes it copied visible to the tensor-core (async) proxy
// and arrives on the older slot's full barrier, so a gathered slot's full
// barrier counts 32 arrivals where the TMA path's counts one (with the
// bytes).  Only the newest slot is ever held back, and no consumer needs the
// newest slot to free an older one, so the producer's waits for free slots
// always end.
#pragma once
#include <cstdint>

#include "sm103_ptx.cuh"

namespace fa {

// Byte geometry of one K or V cache [N_pg, P_s, Hkv, D] for the row gather.
struct KvGather {
  const uint8_t *base;
  int64_t page_stride;   // bytes between pages
  int64_t slot_stride;   // bytes between the keys of a page
  int64_t head_stride;   // bytes between kv heads
};

// 16-byte global -> shared copy through L1 (a lane copies the chunks of one
// row in turn, so the row's line is fetched once); `bytes` 0 writes zeros and
// reads nothing.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}

// Shared-memory layouts a gathered block is written in.
enum GatherLayout : int {
  kGatherSw128 = 0,   // 128-byte rows, 16-byte chunk c of row r at r*128 + ((c ^ (r & 7)) * 16)
  kGatherPlain = 1,   // rows of ROW_BYTES bytes, back to back
  kGatherStage = 2,   // 64-byte rows in the upper half of 32-row, 4 KB slices
};

// Warp-collective: copy ROWS key rows x ROW_BYTES bytes, starting at byte
// `col0` of each key's row, of kv head `hk` into `dst`.  Key row r is the
// sequence key key0 + r; lane r & 31 holds its page id in pg[r >> 5] (-1 for
// a key past the sequence: the row is zero-filled, so that P = 0 never meets
// a stale non-finite value in the PV product).
//
// LPR lanes copy one row together.  LPR = 1: each lane copies whole rows
// (one address per row, no shuffles), for producers that run on few
// registers and read mostly from L2 (prefill).  LPR = 4: four lanes share a
// row, so a warp-wide copy touches 8 rows instead of 32 (fewer L1
// wavefronts), at one shuffle and one address per row and lane; measured
// 1.8x faster for the page-1 decode, which streams from HBM, and slower for
// the prefill kernels.
template <int ROWS, int ROW_BYTES, int LAYOUT, int LPR = 1>
__device__ __forceinline__ void gather_block(uint8_t *dst, const KvGather &g, int hk, int key0, int page_mask,
                                             int col0, const int (&pg)[ROWS / 32], int lane) {
  static_assert(ROW_BYTES == 64 || ROW_BYTES == 128, "rows of 4 or 8 chunks");
  static_assert(LAYOUT != kGatherSw128 || ROW_BYTES == 128, "swizzled rows are 128 bytes");
  static_assert(LAYOUT != kGatherStage || ROW_BYTES == 64, "staged rows are 64 bytes");
  static_assert(LPR == 1 || LPR == 4, "one or four lanes per row");
  constexpr int CH = ROW_BYTES / 16;   // chunks per row
  constexpr int CPL = CH / LPR;        // chunks per lane
  constexpr int RPI = 32 / LPR;        // rows per warp-wide copy
  const int sub = lane % LPR, rs = lane / LPR;
  const uint32_t dbase = smem_u32(dst);
  const uint8_t *head = g.base + (int64_t)hk * g.head_stride + col0 + sub * CPL * 16;
#pragma unroll
  for (int u = 0; u < ROWS / 32; ++u) {
    const int pgu = pg[u];
#pragma unroll
    for (int i = 0; i < 32 / RPI; ++i) {
      const int r32 = i * RPI + rs;   // row within the 32: the lane that holds its page id
      const int r = 32 * u + r32;
      const int page = LPR == 1 ? pgu : __shfl_sync(0xffffffffu, pgu, r32);
      const bool live = page >= 0;
      const uint8_t *src = live ? head + (int64_t)page * g.page_stride + (int64_t)((key0 + r) & page_mask) * g.slot_stride
                                : g.base;
      uint32_t row;
      if constexpr (LAYOUT == kGatherSw128) row = dbase + r * 128;
      else if constexpr (LAYOUT == kGatherPlain) row = dbase + r * ROW_BYTES;
      else row = dbase + (r >> 5) * 4096 + 2048 + (r & 31) * 64;
#pragma unroll
      for (int cc = 0; cc < CPL; ++cc) {
        const int c = sub * CPL + cc;
        const uint32_t at = LAYOUT == kGatherSw128 ? row + ((c ^ (r & 7)) << 4) : row + c * 16;
        cp_async_16(at, live ? src + cc * 16 : src, live ? 16u : 0u);
      }
    }
  }
}

// Completion of gathered ring slots (see the file comment).  One per warp.
// DEFER (1 or 2): how many of the newest committed slots may still be in
// flight when the warp goes on to wait for a free slot.  A kernel may defer
// k slots only if none of its consumers needs any of its k newest slots to
// free the slot the producer waits for next; each kernel states its bound.
template <int DEFER>
struct GatherPipe {
  static_assert(DEFER == 1 || DEFER == 2, "one or two slots in flight");
  uint32_t older = 0, newer = 0;   // full barriers of committed, not yet arrived slots (0: none)

  __device__ __forceinline__ void commit(uint32_t bar) {
    asm volatile("cp.async.commit_group;" ::: "memory");
    if constexpr (DEFER == 1) {
      if (newer) {
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        fence_proxy_async_smem();
        mbar_arrive(newer);
      }
    } else {
      if (older) {
        asm volatile("cp.async.wait_group 2;" ::: "memory");
        fence_proxy_async_smem();
        mbar_arrive(older);
      }
      older = newer;
    }
    newer = bar;
  }
  // All copies landed and every slot arrived; also run on error exits, so
  // that no copy is in flight when the CTA ends.
  __device__ __forceinline__ void drain() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    fence_proxy_async_smem();
    if (older) mbar_arrive(older);
    if (newer) mbar_arrive(newer);
    older = newer = 0;
  }
};

}  // namespace fa
