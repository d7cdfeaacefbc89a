// disco_bwd_tc.cu -- the transpose DISCO contraction on the tensor cores (bf16).
//
// DISCO Kernel Development Guide (torch-harmonics), §Architecture snapshot
// (the backward kernel: the transpose of the sparse contraction, from
// X-shaped gradients back to the input grid) and §Backward
// direction (gather direction, each input pixel accumulates from its
// neighbourhood, no atomics; every output element has exactly one owner).
//
// Polyphase form: with input column j = s q + p and offset delta = s e + p,
//
//   gx[bc, hi, s q + p] = sum_{ho} sum_k sum_e psi_k^{(ho,hi)}(s e + p) G[bc, k, ho, q - e].
//
// A tile owns 128 channels, a group of 8 input rows hi0 .. hi0+7 (they share
// most of their output-row neighbourhood, so each G row is loaded once for
// all eight) and 2 blocks of TQ = 32/s decimated positions (2 x 32 input
// columns).  For one output row ho of the group (window half-width MW) and one
// k, block b of the tile is the MMA
//
//   D_b[bc, (r, t, p)] += sum_i G[bc, k, ho, qb + b TQ - MW + i] * T[(r, t, p), i],
//   T[(r, t, p), i] = psi_k^{(ho, hi0 + r)}(s (t - i + MW) + p),
//
// M = 128 channels, N = 8 rows x 32 columns = 256, K = the window, 16 columns
// per step.  T does not depend on the block, so one T serves both blocks: the
// second block reads the G window TQ columns (kStep1 = TQ / 16 steps) further
// on, i.e. window step w meets T step w in block 0 and T step w - kStep1 in
// block 1.  The T values come from the psi tables by input-row group
// (disco_psi.gtab), laid out so that a 64-column chunk of T is one contiguous
// block per (ho, k, chunk): every builder thread reads 8 consecutive values
// with no bounds logic.
//
// One item per 64-column G box of the window: item c of (ho, k) holds box c
// (window steps 4c .. 4c+3) and T chunk c (T steps 4c .. 4c+3, for block 0
// and for block 1's steps from 4c on); block 1's first kStep1 steps are T
// chunk c - 1's last ones, read from the previous item's stage.  So each G
// box is loaded once per tile, output row and k (pairing both blocks with one
// window chunk instead would need the next box as well, and load most boxes
// of a long window twice), and a T chunk is released after the next item's
// MMAs.
//
// Operands are K-major in the 128-byte swizzled layout: the G window arrives
// by TMA in boxes of 64 columns x 128 channels; T is written in the same
// layout by the builder warps.  A window chunk that crosses the longitude
// seam arrives, for G in the API layout, as two boxes, the chunk's columns
// before the seam in one and those after it in the other, each zero
// elsewhere (columns outside the tensor read as zeros), and its MMAs run on
// both: two 128-row boxes instead of eight 8-column ones, since there a box
// costs by its rows (each in another channel's pages), not its bytes.  For G
// in rows of channels, where rows are cheap, it arrives as 8 wrapped 8-column
// boxes in the unswizzled layout, read with that layout's descriptor.
//
// Only the input rows of the group with support at the entry's output row
// take part: the MMAs have N = 32 x those rows and the builders build only
// their T rows; TMEM starts each tile at zero (the epilogue clears it after
// reading it out), so every MMA accumulates.
//
// Persistent kernel: one CTA per SM; tiles come from the launch's scheduler
// counter (disco_sched.cuh), in an order that puts the long polar row groups
// first and keeps the groups that share G rows close; the pipeline runs
// across tile boundaries.  Rings of G boxes (6 in the API layout, 4 over rows
// of channels), T chunks (3, 4) and 4 psi blocks; roles:
//   warp 0      tiles: the tile index and the group's entry list (bulk copy)
//               into one of two info slots; per item the psi block of its
//               chunk (bulk copy), up to 4 items ahead of the builders;
//   warp 1      MMA issuer (one thread; descriptors precomputed per stage);
//   warps 2, 3, 4, 6, 7, 12  build T into the item's stage;
//   warps 8-11  epilogue: tcgen05.ld, bf16, TMA stores (warp w reads TMEM
//               lanes 32 (w % 4) ..), then zeros back into TMEM;
//   warps 5, 13 G producers: boxes n % 2 == 0, 1, n counting the boxes (the
//               boxes of G in rows of channels, rows W_out apart, go faster
//               the more threads issue them).
// Warps w and w + 4 share one of the SM's four schedulers: the single-thread
// MMA issuer and G producers (w % 4 == 1) share theirs with no builder warp.
// Barriers complete with one arrival per warp (or one commit), not per thread.
// All mbarrier waits are bounded (time-out -> status flag, abort).

#include <cudaTypedefs.h>

#include "disco_bounds.cuh"
#include "disco_internal.cuh"
#include "disco_sched.cuh"
#include "disco_umma.cuh"

namespace disco {

__device__ int g_btc_status = 0;
__device__ unsigned long long g_btc_sched[kSchedSlots];

namespace {

constexpr int kGProducers = 2;              // warps 5, 13: the G boxes of items i % 2 == 0, 1
constexpr int kThreads = 384 + 32 * kGProducers;
constexpr int kBuilderThreads = 192;        // warps 2, 3, 4, 6, 7, 12
constexpr int kEpiThreads = 128;            // warps 8-11
constexpr int kN = 256;                     // MMA N = 8 rows x 32 columns
constexpr int kNT = 2;                      // column blocks per tile
constexpr int kTabSlots = 4;                // psi blocks fetched ahead of the builders
constexpr int kMaxEnt = 128;                // entries (output rows) of one group
constexpr uint32_t kBoxBytes = 128 * 128;   // 128 channels x 64 columns bf16
constexpr uint32_t kNarrowBytes = 128 * 16; // 128 channels x 8 columns
constexpr uint32_t kTBytes = kN * 128;      // T chunk: 256 rows x 64 columns
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr int kStatusBtcTimeout = 8;

__device__ __forceinline__ void btc_flag(int bit) { atomicOr(&g_btc_status, bit); }

__device__ __forceinline__ int wrapc(int c, int W) {
  int r = c % W;
  return r < 0 ? r + W : r;
}

__device__ __forceinline__ bool all_named(bool pred, int id, int n) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

struct BtcArgs {
  __nv_bfloat16* gx;  // [BC][Hin][Win]
  const int32_t* grp_ptr;
  const disco_grp_ent* grp;
  const uint16_t* gtab;
  int BC, Hin, Win, Hout, Wout, K;
  int ntx, nty, ntz;  // tiles along columns, channel blocks, row groups
  long long ngrp_ent, ngtab;  // entries and table elements of psi (extent checks of the bounds-checked build)
  unsigned long long launch_id;  // selects the scheduler slot
  int f16;                       // G, gx and the tables are fp16 (else bf16)
};

template <int S>
struct BGeom {
  static constexpr int TQ = grp_tq(S);
  static constexpr int CW = grp_cw(S);
  static constexpr int kStep1 = TQ / 16;  // K steps between the two blocks' windows (1 or 2)
  static constexpr uint32_t kTabBytes = (uint32_t)grp_block(S) * 2;  // the psi block of one chunk
};

template <int S, bool kTwoBox>
struct BCfg : BGeom<S> {
  using BGeom<S>::kTabBytes;
  // Ring depths (as much as shared memory holds).  T chunks: built ahead of
  // the MMAs and kept for the next item.  G boxes: in flight from L2 or
  // waiting for their MMAs; a seam item takes two with kTwoBox.  Over rows of
  // channels 4 T chunks ran faster than 3; in the API layout 3 + 6 and 4 + 4
  // ran alike.
  static constexpr int kTStages = kTwoBox ? 3 : 4;
  static constexpr int kGStages = kTwoBox ? 6 : 4;
  // a G producer waits on the G stage of its own earlier box: every G stage
  // must stay with one producer, or it would wait on a phase of another's box
  static_assert(kGStages % kGProducers == 0, "a G stage stays with one G producer");
  // layout: T stages | G stages | psi slots | entry lists | gx pieces | barriers
  static constexpr uint32_t kGOff = kTStages * kTBytes;
  static constexpr uint32_t kTabOff = kGOff + kGStages * kBoxBytes;
  static constexpr uint32_t kInfoOff = kTabOff + kTabSlots * kTabBytes;
  static constexpr uint32_t kInfoBytes = 2 * kMaxEnt * sizeof(disco_grp_ent);
  static constexpr uint32_t kOutOff = kInfoOff + kInfoBytes;
  static constexpr uint32_t kOutBytes = 128 * 32 * 2;  // one gx piece: 128 channels x 32 columns
  static constexpr uint32_t kBarOff = kOutOff + 2 * kOutBytes;
  static constexpr size_t kSmem = (size_t)kBarOff + 512 + 1024;  // + barriers, + alignment slack
  static_assert(kGOff % 1024 == 0 && kTabBytes % 16 == 0 && kInfoOff % 16 == 0 && kOutOff % 128 == 0,
                "alignment of the swizzled tiles and copy targets");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

// the z-th row group in processing order: poles first, then inwards, so the
// tiles in flight cover two bands of adjacent groups (which share G rows)
__device__ __forceinline__ int row_group(int z, int nz) { return (z & 1) ? nz - 1 - (z >> 1) : (z >> 1); }

template <int S>
__device__ __forceinline__ void tile_coords(const BtcArgs& a, int tile, int* qb, int* bc0, int* zg) {
  const int x = tile % a.ntx;
  const int rest = tile / a.ntx;
  const int z = rest % a.ntz;
  const int y = rest / a.ntz;
  *qb = x * (kNT * BGeom<S>::TQ);
  *bc0 = y * 128;
  *zg = row_group(z, a.ntz);
}

// Items of one entry (output row) and k: one per 64-column G box of the
// window.  Block 0 reads window steps 0 .. KB-1 and block 1 steps kStep1 ..
// KB-1+kStep1, so the window spans KB + kStep1 steps of 16 columns.
template <int S>
__device__ __forceinline__ int entry_items(const disco_grp_ent& en) {
  return ((int)en.KB + BGeom<S>::kStep1 + 3) / 4;
}

// kTwoBox: a window chunk across the longitude seam arrives as two zero-padded
// 64-column boxes and its MMAs run on both (G in the API layout, where a box
// costs by its 128 rows, each in another channel's pages); otherwise as 8
// wrapped 8-column boxes in the unswizzled layout (G in rows of channels,
// where rows are cheap and the MMAs are not doubled).
template <int S, bool kTwoBox>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap gwide, const __grid_constant__ CUtensorMap gnarrow,
                  const __grid_constant__ CUtensorMap gxmap, const BtcArgs a) {
  using Cfg = BCfg<S, kTwoBox>;
  constexpr int TQ = Cfg::TQ, CW = Cfg::CW;
  constexpr int kTStages = Cfg::kTStages, kGStages = Cfg::kGStages;
  constexpr int kStep1 = Cfg::kStep1;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled operand tiles
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  disco_grp_ent* infos = reinterpret_cast<disco_grp_ent*>(smem + Cfg::kInfoOff);
  uint8_t* outbuf = smem + Cfg::kOutOff;  // [2] gx pieces for TMA stores
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);
  uint64_t* fullA = bars;                      // [kGStages] G box landed
  uint64_t* emptyA = fullA + kGStages;         // [kGStages] MMAs that read it done (commit)
  uint64_t* fullB = emptyA + kGStages;         // [kTStages] T built (one arrival per builder warp)
  uint64_t* emptyT = fullB + kTStages;         // [kTStages] MMAs that read it done (commit)
  uint64_t* fullTab = emptyT + kTStages;       // [kTabSlots] psi block landed
  uint64_t* emptyTab = fullTab + kTabSlots;    // [kTabSlots] builders done reading (one arrival per warp)
  uint64_t* info_full = emptyTab + kTabSlots;  // [2] entry list landed
  uint64_t* info_empty = info_full + 2;        // [2] entry list released by all readers
  uint64_t* acc_full = info_full + 4;          // all MMAs of a tile done (commit)
  uint64_t* tmem_empty = info_full + 5;        // epilogue read TMEM out (one arrival per warp)
  uint64_t* drain = info_full + 6;             // MMAs in flight done, after a failure (commit)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(info_full + 7);
  int32_t* info_cnt = reinterpret_cast<int32_t*>(info_full + 8);  // [2]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(info_full + 9);
  volatile int* tile_id = reinterpret_cast<volatile int*>(info_full + 10);  // [2], -1 = no more tiles

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = a.ntx * a.nty * a.ntz;

  if (tid == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(&fullA[s], 1);
      mbar_init(&emptyA[s], 1);
    }
    for (int s = 0; s < kTStages; ++s) {
      mbar_init(&fullB[s], kBuilderThreads / 32);
      mbar_init(&emptyT[s], 1);
    }
    for (int s = 0; s < kTabSlots; ++s) {
      mbar_init(&fullTab[s], 1);
      mbar_init(&emptyTab[s], kBuilderThreads / 32);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&info_full[b], 1);
      mbar_init(&info_empty[b], kGProducers + 1 + (kBuilderThreads + kEpiThreads) / 32);
    }
    mbar_init(acc_full, 1);
    mbar_init(tmem_empty, kEpiThreads / 32);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    // ------------------------------------ tiles, entry lists, psi blocks --
    if (lane == 0) {
      int i = 0, tl = 0, done = 0;  // done: one past the last item whose psi block was issued
      bool ok = true;
      unsigned long long* slot = sched_join(g_btc_sched, a.launch_id, kWaitLimit);
      if (!slot) btc_flag(kStatusBtcTimeout);  // this CTA takes no tile
      for (; ok; ++tl) {
        const int b = tl & 1;
        if ((tl >= 2 && !mbar_wait(&info_empty[b], ((tl >> 1) - 1) & 1, kWaitLimit)) || *abort_flag) {
          ok = false;
          break;
        }
        const int tile = slot ? sched_next(slot) : ntiles;
        if (tile >= ntiles) {  // tell the other roles to stop
          tile_id[b] = -1;
          info_cnt[b] = 0;
          mbar_arrive(&info_full[b]);
          break;
        }
        tile_id[b] = tile;
        int qb, bc0, zg;
        tile_coords<S>(a, tile, &qb, &bc0, &zg);
        const int e0 = a.grp_ptr[zg];
        int ne = min(a.grp_ptr[zg + 1] - e0, kMaxEnt);
        if (!DISCO_IN_BOUNDS(zg >= 0 && zg < a.ntz && e0 >= 0 && ne >= 0 && e0 + (long long)ne <= a.ngrp_ent))
          ne = 0;
        info_cnt[b] = ne;
        disco_grp_ent* info = infos + b * kMaxEnt;
        if (ne > 0) {
          mbar_expect_tx(&info_full[b], ne * (uint32_t)sizeof(disco_grp_ent));
          bulk_copy(info, a.grp + e0, ne * (uint32_t)sizeof(disco_grp_ent), &info_full[b]);
          if (!mbar_wait(&info_full[b], (tl >> 1) & 1, kWaitLimit)) {
            ok = false;
            break;
          }
        } else {
          mbar_arrive(&info_full[b]);
        }
        // item (ho, k, c): the psi block of chunk c into psi slot i % kTabSlots
        for (int j = 0; j < ne && ok; ++j) {
          const disco_grp_ent en = info[j];
          const int nit = entry_items<S>(en);
          for (int k = 0; k < a.K && ok; ++k)
            for (int c = 0; c < nit && ok; ++c, ++i) {
              const int t = i % kTabSlots;
              if ((i >= kTabSlots && !mbar_wait(&emptyTab[t], ((i / kTabSlots) - 1) & 1, kWaitLimit)) ||
                  *abort_flag) {
                ok = false;
                break;
              }
              if (c < en.nch) {
                mbar_expect_tx(&fullTab[t], Cfg::kTabBytes);
                const long long toff = (long long)en.off + (long long)(k * en.nch + c) * grp_block(S);
                if (DISCO_IN_BOUNDS(k >= 0 && k < a.K && c >= 0 && toff >= 0 && toff + grp_block(S) <= a.ngtab))
                  bulk_copy(smem + Cfg::kTabOff + t * Cfg::kTabBytes, a.gtab + toff, Cfg::kTabBytes, &fullTab[t]);
                else
                  mbar_complete_tx(&fullTab[t], Cfg::kTabBytes);
              } else {
                mbar_arrive(&fullTab[t]);  // the item past the last chunk builds no T
              }
              done = i + 1;
            }
        }
      }
      if (!ok) {
        btc_flag(kStatusBtcTimeout);
        *abort_flag = 1;
        // let the copies in flight land before the CTA exits
        for (int li = done - 1; li >= 0 && li >= done - kTabSlots; --li)
          mbar_wait(&fullTab[li % kTabSlots], (li / kTabSlots) & 1, kWaitLimit);
      }
      if (slot) sched_leave(slot);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      // Descriptors of the first T chunk and G box (128-byte swizzled).  Stage
      // x and K step q add x * (stage bytes) / 16 and 2 q (32 bytes a step) to
      // the start-address field.
      const uint32_t sb = smem_u32(smem);
      const uint64_t dT0 = smem_desc_sw128(sb), dG0 = smem_desc_sw128(sb + Cfg::kGOff);
      // (8 wrapped 8-column boxes: unswizzled, K step q 4 KB further on)
      const uint64_t dN0 = smem_desc(sb + Cfg::kGOff, kNarrowBytes, 128);
      constexpr uint64_t kTStep = kTBytes >> 4, kGStep = kBoxBytes >> 4;
      int i = 0, nb = 0, tl = 0;  // items and G boxes so far
      bool ok = true;
      for (; ok; ++tl) {
        const int b = tl & 1;
        if (!mbar_wait(&info_full[b], (tl >> 1) & 1, kWaitLimit) || *abort_flag) {
          ok = false;
          break;
        }
        const int tile = tile_id[b];
        if (tile < 0) break;
        if (!mbar_wait(tmem_empty, tl & 1, kWaitLimit) || *abort_flag) {  // TMEM read out and zeroed
          ok = false;
          break;
        }
        tc_fence_after();
        int qb, bc0, zg;
        tile_coords<S>(a, tile, &qb, &bc0, &zg);
        // block 1 of the last column tile can lie past the ring (W_in / 32 odd):
        // its MMAs are skipped (the epilogue stores no such piece)
        const bool blk1 = S * (qb + TQ) < a.Win;
        const int ne = info_cnt[b];
        const disco_grp_ent* info = infos + b * kMaxEnt;
        for (int j = 0; j < ne && ok; ++j) {
          const int KB = info[j].KB, nit = entry_items<S>(info[j]);
          const int w0 = wrapc(qb - info[j].MW, a.Wout);  // ring column of box 0
          // only the rows r0 .. r1 of the group have support at this output
          // row: MMAs of N = 32 (r1 - r0 + 1) on T rows and TMEM columns from 32 r0
          const int r0 = info[j].r0, nr = info[j].r1 - r0 + 1;
          const uint32_t ide = idesc_16_f32(128, 32 * nr, a.f16 != 0);
          const uint32_t d0 = tmem + 32 * r0, d1 = tmem + kN + 32 * r0;
          const uint64_t toff = 256u * r0;  // 4 KB of T rows per input row
          for (int k = 0; k < a.K && ok; ++k) {
            int wc = w0;
            for (int c = 0; c < nit; ++c, ++i) {
              // a window chunk across the longitude seam: two boxes, each with
              // the other's columns zero, and the MMAs run on both (kTwoBox),
              // or one unswizzled tile of 8 wrapped boxes
              const bool cross = wc + 64 > a.Wout, seam = kTwoBox && cross;
              const int g0 = nb % kGStages, g1 = (nb + 1) % kGStages, x = i % kTStages;
              if (!mbar_wait(&fullA[g0], (nb / kGStages) & 1, kWaitLimit) ||
                  (seam && !mbar_wait(&fullA[g1], ((nb + 1) / kGStages) & 1, kWaitLimit)) ||
                  !mbar_wait(&fullB[x], (i / kTStages) & 1, kWaitLimit) || *abort_flag) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t dT = dT0 + x * kTStep + toff;
              // T chunk c - 1 (item i - 1, read when c >= 1): its last kStep1 steps
              const uint64_t dTp = dT0 + ((i + kTStages - 1) % kTStages) * kTStep + toff;
              const uint64_t dA0 = (!kTwoBox && cross ? dN0 : dG0) + g0 * kGStep, dA1 = dG0 + g1 * kGStep;
              const uint32_t dAq = !kTwoBox && cross ? 256u : 2u;
              // Box step q holds window step 4 c + q.  T step t = 4 c + m meets
              // it in block 0 at box step m and in block 1 at box step
              // m + kStep1 (T step t is this chunk's step m, or for m < 0 chunk
              // c - 1's step 4 + m).  Issued by T step, the MMAs alternate
              // between the two accumulators: MMAs into one accumulator back to
              // back run at well under half the rate.  A seam item's second box
              // in a second pass, in the same order (skipping the K steps that
              // lie wholly in a box's zero columns made the pass slower).
              for (int pass = 0; pass < (seam ? 2 : 1); ++pass) {
                const uint64_t dA = pass ? dA1 : dA0;
                const uint32_t dq = pass ? 2u : dAq;
#pragma unroll
                for (int m = -kStep1; m < 4; ++m) {
                  const int t = 4 * c + m;
                  if (t < 0 || t >= KB) continue;
                  const uint64_t bd = m >= 0 ? dT + 2 * m : dTp + 2 * (4 + m);
                  if (m >= 0) umma_bf16(d0, dA + m * dq, bd, ide, 1u);
                  if (m + kStep1 < 4 && blk1) umma_bf16(d1, dA + (m + kStep1) * dq, bd, ide, 1u);
                }
              }
              // item i's G boxes, and item i - 1's T chunk (whose last steps
              // item i read), are free once these MMAs complete
              umma_commit(&emptyA[g0]);
              if (seam) umma_commit(&emptyA[g1]);
              if (i >= 1) umma_commit(&emptyT[(i + kTStages - 1) % kTStages]);
              nb += seam ? 2 : 1;
              wc = wc + 64 >= a.Wout ? wc + 64 - a.Wout : wc + 64;
            }
          }
        }
        if (!ok) break;
        mbar_arrive(&info_empty[b]);
        // a tile without entries leaves the accumulators unwritten: the epilogue stores zeros
        umma_commit(acc_full);
      }
      if (!ok) {
        btc_flag(kStatusBtcTimeout);
        *abort_flag = 1;
        // let the MMAs in flight finish before TMEM is freed
        umma_commit(drain);
        mbar_wait(drain, 0, kWaitLimit);
      }
    }
  } else if ((warp != 5 && warp < 8) || warp == 12) {
    // -------------------------------- T builders (warps 2, 3, 4, 6, 7, 12) --
    const int btid = 32 * (warp == 12 ? 5 : warp < 5 ? warp - 2 : warp - 3) + lane;
    int i = 0, tl = 0;
    bool ok = true;
    for (; ok; ++tl) {
      const int b = tl & 1;
      {
        const bool mine = mbar_wait(&info_full[b], (tl >> 1) & 1, kWaitLimit) && !*abort_flag;
        ok = all_named(mine, 1, kBuilderThreads);
        if (!ok) break;
      }
      if (tile_id[b] < 0) break;  // same value for all builder threads
      const int ne = info_cnt[b];
      const disco_grp_ent* info = infos + b * kMaxEnt;
      for (int j = 0; j < ne && ok; ++j) {
        const int KB = info[j].KB, nch = info[j].nch, nit = entry_items<S>(info[j]);
        const int r0 = info[j].r0, nr = info[j].r1 - r0 + 1;  // the rows the MMAs read
        for (int k = 0; k < a.K && ok; ++k)
          for (int c = 0; c < nit; ++c, ++i) {
            const int t = i % kTabSlots, x = i % kTStages;
            // the item's psi block has landed and the MMAs that read the T
            // stage's previous chunk are done
            const bool mine = mbar_wait(&fullTab[t], (i / kTabSlots) & 1, kWaitLimit) &&
                              (i < kTStages || mbar_wait(&emptyT[x], ((i / kTStages) - 1) & 1, kWaitLimit)) &&
                              !*abort_flag;
            ok = all_named(mine, 1, kBuilderThreads);
            if (!ok) break;
            uint8_t* T = smem + x * kTBytes;
            const uint16_t* tab = reinterpret_cast<const uint16_t*>(smem + Cfg::kTabOff + t * Cfg::kTabBytes);
            // 16-byte chunks per T row (none for the item past the last chunk)
            const int nq = c < nch ? 2 * min(4, KB - 4 * c) : 0;
            // T[(r, t, p), 8 q8 + e] = tab[r][p][8 q8 + TQ - 1 - t + e]: the rows
            // t = 8 g + j (j = 0..7) of one (r, p, q8) read the same 16 table
            // values from the aligned index 8 q8 + TQ - 8 - 8 g on, shifted by
            // 7 - j.  One unit (r, p, g, q8) loads them with two 16-byte loads
            // and writes the 8 rows' chunks q8; q8 varies fastest across lanes
            // (conflict-free loads, and stores that cover all banks).  Only the
            // rows r0 .. r1 are built: the MMAs read no others
            constexpr int kG = TQ / 8;  // row groups of 8 t per (r, p)
            for (int u = btid; u < nr * S * kG * nq; u += kBuilderThreads) {
              const int q8 = u % nq, rest = u / nq;
              const int g = rest % kG, rp = rest / kG + r0 * S;  // rp = r S + p
              const int r = rp / S, p = rp - r * S;
              const uint4* src = reinterpret_cast<const uint4*>(tab + rp * CW + 8 * (q8 + kG - 1 - g));
              const uint4 lo = src[0], hi = src[1];
              const uint32_t v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int m = 7 - j;  // first of the row's 8 values among the 16 loaded
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  w[e] = (m & 1) ? __funnelshift_r(v[m / 2 + e], v[m / 2 + e + 1], 16) : v[m / 2 + e];
                const int n = r * 32 + (8 * g + j) * S + p;
                *reinterpret_cast<uint4*>(T + n * 128 + ((q8 ^ (n & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
            // every thread's T writes are visible to the tensor cores, then one
            // arrival per warp (192 arrivals on one barrier would serialise)
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(&fullB[x]);
              mbar_arrive(&emptyTab[t]);
            }
          }
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&info_empty[b]);
    }
    if (!ok) {
      btc_flag(kStatusBtcTimeout);
      *abort_flag = 1;
    }
  } else if (warp == 5 || warp == 13) {
    // ------------------------------ G producers (warps 5, 13): boxes n % 2 --
    // One 64-column box per item (with kTwoBox two where the window chunk
    // crosses the longitude seam: the box at the chunk's ring column, whose
    // columns past the seam are outside the tensor and arrive as zeros, and
    // the box one ring earlier, whose columns before the seam arrive as
    // zeros) into G stage n % kGStages, n counting boxes, as soon as the MMAs
    // that read the stage's previous box are done.
    const int who = warp == 5 ? 0 : 1;
    if (lane == 0) {
      int i = 0, nb = 0, done = 0;  // done: one past the last box this thread issued
      bool ok = true;
      for (int tl = 0; ok; ++tl) {
        const int b = tl & 1;
        if (!mbar_wait(&info_full[b], (tl >> 1) & 1, kWaitLimit) || *abort_flag) {
          ok = false;
          break;
        }
        const int tile = tile_id[b];
        if (tile < 0) break;
        int qb, bc0, zg;
        tile_coords<S>(a, tile, &qb, &bc0, &zg);
        const int ne = info_cnt[b];
        const disco_grp_ent* info = infos + b * kMaxEnt;
        for (int j = 0; j < ne && ok; ++j) {
          const disco_grp_ent en = info[j];
          const int nit = entry_items<S>(en);
          const int w0 = wrapc(qb - en.MW, a.Wout);
          [[maybe_unused]] const bool rows_ok =
              DISCO_IN_BOUNDS(en.ho >= 0 && en.ho < a.Hout && bc0 >= 0 && bc0 < a.BC);
          for (int k = 0; k < a.K && ok; ++k) {
            const int grow = k * a.Hout + en.ho;
            int wc = w0;
            for (int c = 0; c < nit && ok; ++c, ++i) {
              const bool cross = wc + 64 > a.Wout;
              const int nbox = kTwoBox && cross ? 2 : 1;
              for (int h = 0; h < nbox; ++h, ++nb) {
                if (nb % kGProducers != who) continue;
                const int g = nb % kGStages;
                if ((nb >= kGStages && !mbar_wait(&emptyA[g], ((nb / kGStages) - 1) & 1, kWaitLimit)) ||
                    *abort_flag) {
                  ok = false;
                  break;
                }
                uint8_t* dst = smem + Cfg::kGOff + g * kBoxBytes;
                mbar_expect_tx(&fullA[g], kBoxBytes);
                if (kTwoBox || !cross) {
                  const int x0 = h == 0 ? wc : wc - a.Wout;  // the second box starts before column 0
                  if (DISCO_IN_BOUNDS(rows_ok && x0 > -64 && x0 < a.Wout))
                    tma_load_3d(dst, &gwide, x0, grow, bc0, &fullA[g]);
                  else
                    mbar_complete_tx(&fullA[g], kBoxBytes);
                } else {
                  for (int q = 0; q < 8; ++q) {
                    const int cn = wrapc(wc + 8 * q, a.Wout);
                    if (DISCO_IN_BOUNDS(rows_ok && cn >= 0 && cn + 8 <= a.Wout))
                      tma_load_3d(dst + q * kNarrowBytes, &gnarrow, cn, grow, bc0, &fullA[g]);
                    else
                      mbar_complete_tx(&fullA[g], kNarrowBytes);
                  }
                }
                done = nb + 1;
              }
              wc = wc + 64 >= a.Wout ? wc + 64 - a.Wout : wc + 64;
            }
          }
        }
        if (!ok) break;
        mbar_arrive(&info_empty[b]);
      }
      if (!ok) {
        btc_flag(kStatusBtcTimeout);
        *abort_flag = 1;
        // let this thread's boxes in flight land before the CTA exits
        for (int lb = done - 1; lb >= 0 && lb >= done - kGStages; --lb)
          if (lb % kGProducers == who) mbar_wait(&fullA[lb % kGStages], (lb / kGStages) & 1, kWaitLimit);
      }
    }
  } else {
    // ----------------------------------------------- epilogue (warps 8-11) --
    const int q = warp & 3;
    // The MMAs accumulate into TMEM that the epilogue leaves zero: cleared here
    // for the first tile, and after reading each tile out for the next one
    // (a tile's entries cover different rows, so no MMA may start a sum).
    for (int col = 0; col < 2 * kN; col += 16) tmem_st16_zero(tmem + ((uint32_t)(q * 32) << 16) + col);
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tmem_empty);
    int tl = 0, npiece = 0;
    for (;; ++tl) {
      const int b = tl & 1;
      // one decision for all 4 epilogue warps: they meet at named barriers below
      bool fin = all_named(mbar_wait(&info_full[b], (tl >> 1) & 1, kWaitLimit) && !*abort_flag, 2, kEpiThreads);
      if (!fin) {
        if (lane == 0) btc_flag(kStatusBtcTimeout);
        *abort_flag = 1;
        break;
      }
      const int tile = tile_id[b];
      if (tile < 0) break;
      fin = all_named(mbar_wait(acc_full, tl & 1, kWaitLimit) && !*abort_flag, 2, kEpiThreads);
      if (!fin) {
        if (lane == 0) btc_flag(kStatusBtcTimeout);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      int qb, bc0, zg;
      tile_coords<S>(a, tile, &qb, &bc0, &zg);
      const int hi0 = zg * kGrpRows;
      const bool any = info_cnt[b] > 0;
      const int er = q * 32 + lane;  // channel row of this thread in a piece
      // 16 pieces of [128 channels x 32 columns] (one row, one column block),
      // each converted into one of two shared-memory buffers and written by a
      // TMA store (rows >= H_in and channels >= B*C are clipped by the store)
      for (int blk = 0; blk < kNT; ++blk)
        for (int r = 0; r < kGrpRows; ++r, ++npiece) {
          uint8_t* ob = outbuf + (npiece & 1) * Cfg::kOutBytes;
          if (tid == 256) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");  // buffer free
          asm volatile("bar.sync 2, 128;" ::: "memory");
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            float v[16];
            if (any) {
              const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + blk * kN + r * 32 + cc * 16;
              tmem_ld16(ta, v);
              tmem_st16_zero(ta);
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] = 0.f;
            }
            uint32_t w32[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              w32[e] = pack2_16(v[2 * e], v[2 * e + 1], a.f16);
            }
            uint4* dst = reinterpret_cast<uint4*>(ob + er * 64 + cc * 32);
            dst[0] = make_uint4(w32[0], w32[1], w32[2], w32[3]);
            dst[1] = make_uint4(w32[4], w32[5], w32[6], w32[7]);
          }
          fence_proxy_async_smem();
          asm volatile("bar.sync 2, 128;" ::: "memory");
          if (tid == 256) {
            const int col = S * (qb + blk * TQ);
            if (col < a.Win && hi0 + r < a.Hin &&  // else the whole piece lies outside gx
                DISCO_IN_BOUNDS(col >= 0 && hi0 + r >= 0 && bc0 >= 0 && bc0 < a.BC))
              asm volatile(
                  "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                      reinterpret_cast<uint64_t>(&gxmap)),
                  "r"(col), "r"(hi0 + r), "r"(bc0), "r"(smem_u32(ob))
                  : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
        }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(tmem_empty);
        mbar_arrive(&info_empty[b]);
      }
    }
    if (tid == 256) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_b() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      n = v;
    else
      n = 1;
  }
  return n;
}

// G as [column][row k*H_out + ho][channel]: in the API layout [BC][K*H_out][W_out]
// (channel rows a K*H_out*W_out slab apart) or, for an intermediate the
// library writes itself, [K*H_out][BC][W_out] (channel rows W_out apart, which
// lets a 128-channel box stream far faster).  Same boxes and coordinates.
int encode_g(CUtensorMap* map, const void* G, const BtcArgs& a, int BC, int boxw, bool swz, bool rows_of_channels) {
  const CUtensorMapDataType dt16 = a.f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  auto enc = encode_fn_b();
  if (!enc) return fail(DISCO_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {(cuuint64_t)a.Wout, (cuuint64_t)a.K * a.Hout, (cuuint64_t)BC};
  cuuint64_t strides[2] = {(cuuint64_t)a.Wout * 2, (cuuint64_t)a.K * a.Hout * a.Wout * 2};
  if (rows_of_channels) {
    strides[0] = (cuuint64_t)BC * a.Wout * 2;
    strides[1] = (cuuint64_t)a.Wout * 2;
  }
  cuuint32_t box[3] = {(cuuint32_t)boxw, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult cr = enc(map, dt16, 3, const_cast<void*>(G), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return fail(DISCO_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)cr);
  return DISCO_OK;
}

template <int S>
int launch_btc(const disco_psi* psi, const void* G, void* gx, int BC, cudaStream_t st, bool roc, bool f16) {
  BtcArgs a;
  a.gx = (__nv_bfloat16*)gx;
  a.grp_ptr = psi->grp_ptr;
  a.grp = psi->grp;
  a.gtab = f16 ? psi->gtab_h : psi->gtab;
  a.f16 = f16 ? 1 : 0;
  a.BC = BC;
  a.Hin = psi->grid_in.nlat;
  a.Win = psi->grid_in.nlon;
  a.Hout = psi->grid_out.nlat;
  a.Wout = psi->grid_out.nlon;
  a.K = psi->K;
  a.ntx = (a.Win + S * kNT * BGeom<S>::TQ - 1) / (S * kNT * BGeom<S>::TQ);
  a.nty = (BC + 127) / 128;
  a.ntz = psi->ngrp;
  a.ngrp_ent = psi->ngrp_ent;
  a.ngtab = psi->ngtab;
  a.launch_id = next_launch_id();
  CUtensorMap wide, narrow, gxm;
  int stt = encode_g(&wide, G, a, BC, 64, true, roc);
  if (stt) return stt;
  if ((stt = encode_g(&narrow, G, a, BC, 8, false, roc))) return stt;
  {
    // gx as the TMA store target: [B*C][H_in][W_in], box 32 columns x 1 row x 128 channels
    cuuint64_t dims[3] = {(cuuint64_t)a.Win, (cuuint64_t)a.Hin, (cuuint64_t)BC};
    cuuint64_t strides[2] = {(cuuint64_t)a.Win * 2, (cuuint64_t)a.Hin * a.Win * 2};
    cuuint32_t box[3] = {32, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult cr = encode_fn_b()(&gxm, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                                gx, dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return fail(DISCO_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)cr);
  }
  auto kern = roc ? bwd_tc_kernel<S, false> : bwd_tc_kernel<S, true>;
  const size_t smem = roc ? BCfg<S, false>::kSmem : BCfg<S, true>::kSmem;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return check_launch("disco_bwd (tensor cores) attribute");
  const long long ntiles = (long long)a.ntx * a.nty * a.ntz;
  const int grid = (int)(ntiles < sm_count() ? ntiles : sm_count());
  if (ntiles + grid > (long long)kSchedCountMask || grid > kSchedMaxCtas)
    return fail(DISCO_ERR_UNSUPPORTED, "problem too large");
  kern<<<grid, kThreads, smem, st>>>(wide, narrow, gxm, a);
  return check_launch("disco_bwd (tensor cores)");
}

}  // namespace

// Leaves in the scheduler word of launch `id` the tag of another launch with
// its counter part-way, as any earlier launch leaves it (diagnostic: launch
// `id` must take the word over and still compute every tile).
cudaError_t btc_sched_plant(unsigned long long id) {
  const unsigned long long w = sched_tag(id + kSchedSlots) | 5ull;  // no active CTA
  return cudaMemcpyToSymbol(g_btc_sched, &w, sizeof(w), (id % kSchedSlots) * sizeof(w));
}

cudaError_t btc_status(int32_t* v, bool clear) {
  int32_t t = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&t, g_btc_status, sizeof(int32_t));
  if (e == cudaSuccess && clear) {
    const int32_t zero = 0;
    e = cudaMemcpyToSymbol(g_btc_status, &zero, sizeof(int32_t));
  }
  *v |= t;
  return e;
}

bool bwd_tc_supported(const disco_psi* psi, int BC) {
  const int Win = psi->grid_in.nlon, Wout = psi->grid_out.nlon, Hin = psi->grid_in.nlat;
  return (psi->s == 1 || psi->s == 2) && Wout % 8 == 0 && Win % 8 == 0 && Wout >= 64 && BC >= 1 &&
         psi->K <= 16 && psi->grp_ptr && psi->grp && psi->gtab && psi->ngrp_ent >= 1 &&
         psi->ngrp == (Hin + kGrpRows - 1) / kGrpRows && psi->grp_max <= kMaxEnt &&
         (long long)psi->K * psi->grid_out.nlat <= (1 << 30);
}

int bwd_tensor_core(const disco_psi* psi, const void* G, void* gx, int BC, cudaStream_t st, bool rows_of_channels,
                    bool f16) {
  if (!bwd_tc_supported(psi, BC) || (f16 && !psi->gtab_h)) return DISCO_ERR_UNSUPPORTED;
  return psi->s == 1 ? launch_btc<1>(psi, G, gx, BC, st, rows_of_channels, f16)
                     : launch_btc<2>(psi, G, gx, BC, st, rows_of_channels, f16);
}

// This unit's word of failed range checks (always 0 outside the bounds-checked build).
DISCO_BOUNDS_READER(btc_bounds)

}  // namespace disco
