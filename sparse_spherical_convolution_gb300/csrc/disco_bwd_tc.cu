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
// per step.  T does not depend on the block, so one T serves both blocks (the
// second block reads the G window TQ columns further on).  The T values come
// from the psi tables by input-row group (disco_psi.gtab), laid out so that a
// 64-column chunk of T is one contiguous block per (ho, k, chunk): every
// builder thread reads 8 consecutive values with no bounds logic.
//
// Operands are K-major in the 128-byte swizzled layout: the G window arrives
// by TMA in boxes of 64 columns x 128 channels (a box that would cross the
// longitude seam is fetched instead as 8 wrapped 8-column boxes in the
// unswizzled layout and read with that layout's descriptor); T is written in
// the same swizzled layout by the builder warps.
//
// Persistent kernel: one CTA per SM; the producer takes the next tile from
// the launch's scheduler counter (disco_sched.cuh), in an order that puts the
// long polar row groups first and keeps the groups that share G rows close;
// the pipeline runs across tile boundaries:
//   warp 0      producer: per tile the tile index and the group's entry list
//               (bulk copy) into one of two info slots, per item (ho, k,
//               chunk) i with i % 3 == 0 the psi block (bulk copy) and 1-2 G
//               boxes (TMA);
//   warp 1      MMA issuer (one thread);
//   warps 2-7   build T;
//   warps 8-11  epilogue: tcgen05.ld, bf16, TMA stores;
//   warps 12-13 the other producers: the copies of items i % 3 == 1, 2 (one
//               thread issuing all 16 KB boxes caps the load rate near 35
//               GB/s per SM; the boxes of G in rows of channels, rows W_out
//               apart, go faster the more threads issue them).
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

constexpr int kProducers = 3;               // warp 0 issues items i % 3 == 0, warps 12, 13 the others
constexpr int kThreads = 384 + 32 * (kProducers - 1);
constexpr int kBuilderThreads = 192;        // warps 2-7
constexpr int kEpiThreads = 128;            // warps 8-11
constexpr int kN = 256;                     // MMA N = 8 rows x 32 columns
constexpr int kNT = 2;                      // column blocks per tile
constexpr int kStages = 3;
// a producer waits on the stage of its own previous item: the ring must be at
// least as deep as the producers' item stride, or it would wait on a phase of
// another producer's item
static_assert(kStages >= kProducers, "one stage per producer at least");
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
struct BCfg {
  static constexpr int TQ = grp_tq(S);
  static constexpr int CW = grp_cw(S);
  static constexpr uint32_t kTabBytes = (uint32_t)grp_block(S) * 2;
  static constexpr uint32_t kTabSlot = (kTabBytes + 1023) & ~1023u;
  // stage: 2 G box slots | T chunk | psi block
  static constexpr uint32_t kStageBytes = 2 * kBoxBytes + kTBytes + kTabSlot;
  static constexpr uint32_t kInfoBytes = 2 * kMaxEnt * sizeof(disco_grp_ent);
  static constexpr uint32_t kOutBytes = 128 * 32 * 2;  // one gx piece: 128 channels x 32 columns
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes + 2 * kOutBytes + kInfoBytes + 256 + 1024;
};

// the z-th row group in processing order: poles first, then inwards, so the
// tiles in flight cover two bands of adjacent groups (which share G rows)
__device__ __forceinline__ int row_group(int z, int nz) { return (z & 1) ? nz - 1 - (z >> 1) : (z >> 1); }

template <int S>
__device__ __forceinline__ void tile_coords(const BtcArgs& a, int tile, int* qb, int* bc0, int* zg) {
  const int x = tile % a.ntx;
  const int rest = tile / a.ntx;
  const int y = rest % a.nty;
  const int z = rest / a.nty;
  *qb = x * (kNT * BCfg<S>::TQ);
  *bc0 = y * 128;
  *zg = row_group(z, a.ntz);
}

// a G box that would cross the longitude seam is fetched as 8 narrow boxes
__device__ __forceinline__ bool box_is_narrow(int col0, int Wout) { return wrapc(col0, Wout) + 64 > Wout; }

template <int S>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap gwide, const __grid_constant__ CUtensorMap gnarrow,
                  const __grid_constant__ CUtensorMap gxmap, const BtcArgs a) {
  using Cfg = BCfg<S>;
  constexpr int TQ = Cfg::TQ, CW = Cfg::CW;
  constexpr int kStep1 = TQ / 16;  // K steps between the two blocks' windows
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled operand tiles
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  disco_grp_ent* infos = reinterpret_cast<disco_grp_ent*>(smem + kStages * Cfg::kStageBytes);
  uint8_t* outbuf = smem + kStages * Cfg::kStageBytes + Cfg::kInfoBytes;  // [2] gx pieces for TMA stores
  uint64_t* bars = reinterpret_cast<uint64_t*>(outbuf + 2 * Cfg::kOutBytes);
  uint64_t* fullA = bars;                         // [kStages] G boxes landed
  uint64_t* fullB = bars + kStages;               // [kStages] T built (192 arrivals)
  uint64_t* empty = bars + 2 * kStages;           // [kStages] MMAs of the stage done (commit)
  uint64_t* info_full = bars + 3 * kStages;       // [2] entry list landed
  uint64_t* info_empty = bars + 3 * kStages + 2;  // [2] entry list released by all readers
  uint64_t* acc_full = bars + 3 * kStages + 4;    // all MMAs of a tile done (commit)
  uint64_t* tmem_empty = bars + 3 * kStages + 5;  // epilogue read TMEM out (128 arrivals)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3 * kStages + 6);
  int32_t* info_cnt = reinterpret_cast<int32_t*>(bars + 3 * kStages + 7);  // [2]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 3 * kStages + 8);
  volatile int* tile_id = reinterpret_cast<volatile int*>(bars + 3 * kStages + 9);  // [2], -1 = no more tiles
  // [kStages] psi block landed: the builders start T while the G boxes are still in flight
  uint64_t* fullT = bars + 3 * kStages + 10;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = a.ntx * a.nty * a.ntz;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&fullA[s], 1);
      mbar_init(&fullT[s], 1);
      mbar_init(&fullB[s], kBuilderThreads);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&info_full[b], 1);
      mbar_init(&info_empty[b], kProducers - 1 + 1 + kBuilderThreads + kEpiThreads);
    }
    mbar_init(acc_full, 1);
    mbar_init(tmem_empty, kEpiThreads);
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

  // Copies of item i (stage i % kStages): the psi block and the 1-2 G boxes.
  // Issued by producer i % kProducers after the stage's previous MMAs completed.
  auto issue_item = [&](int i, const disco_grp_ent& en, int k, int c, int qb, int bc0) -> bool {
    const int s = i % kStages;
    if ((i >= kStages && !mbar_wait(&empty[s], ((i / kStages) - 1) & 1, kWaitLimit)) || *abort_flag)
      return false;
    uint8_t* st = smem + (size_t)s * Cfg::kStageBytes;
    const int nsteps = min(4, (int)en.KB - 4 * c);
    const int nbox = (4 * c + nsteps + kStep1 + 3) / 4 - c;  // 1 or 2
    mbar_expect_tx(&fullT[s], Cfg::kTabBytes);
    const long long toff = (long long)en.off + (long long)(k * en.nch + c) * grp_block(S);
    if (DISCO_IN_BOUNDS(k >= 0 && k < a.K && c >= 0 && c < en.nch && toff >= 0 && toff + grp_block(S) <= a.ngtab))
      bulk_copy(st + 2 * kBoxBytes + kTBytes, a.gtab + toff, Cfg::kTabBytes, &fullT[s]);
    else
      mbar_complete_tx(&fullT[s], Cfg::kTabBytes);
    mbar_expect_tx(&fullA[s], nbox * kBoxBytes);
    const int row = k * a.Hout + en.ho;
    const bool rows_ok = DISCO_IN_BOUNDS(en.ho >= 0 && en.ho < a.Hout && bc0 >= 0 && bc0 < a.BC);
    for (int bb = 0; bb < nbox; ++bb) {
      const int col0 = qb - en.MW + 64 * (c + bb);
      uint8_t* dst = st + bb * kBoxBytes;
      if (!box_is_narrow(col0, a.Wout)) {
        if (DISCO_IN_BOUNDS(rows_ok && wrapc(col0, a.Wout) >= 0))
          tma_load_3d(dst, &gwide, wrapc(col0, a.Wout), row, bc0, &fullA[s]);
        else
          mbar_complete_tx(&fullA[s], kBoxBytes);
      } else {
        for (int g = 0; g < 8; ++g) {
          const int cn = wrapc(col0 + 8 * g, a.Wout);
          if (DISCO_IN_BOUNDS(rows_ok && cn >= 0 && cn + 8 <= a.Wout))
            tma_load_3d(dst + g * kNarrowBytes, &gnarrow, cn, row, bc0, &fullA[s]);
          else
            mbar_complete_tx(&fullA[s], kNarrowBytes);
        }
      }
    }
    return true;
  };
  // after a failure: let this producer's copies in flight land before the CTA
  // exits (n = one past its last issued item)
  auto drain_own = [&](int n, int who) {
    for (int li = n - 1; li >= 0 && li >= n - kProducers * kStages; --li)
      if (li % kProducers == who) {
        mbar_wait(&fullA[li % kStages], (li / kStages) & 1, kWaitLimit);
        mbar_wait(&fullT[li % kStages], (li / kStages) & 1, kWaitLimit);
      }
  };

  if (warp == 0) {
    // ------------------------------------------- producer (items i % 3 == 0) --
    if (lane == 0) {
      int i = 0, tl = 0, done = 0;  // done: one past the last item this thread issued
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
        for (int j = 0; j < ne && ok; ++j) {
          const disco_grp_ent en = info[j];
          for (int k = 0; k < a.K && ok; ++k)
            for (int c = 0; c < en.nch && ok; ++c, ++i)
              if (i % kProducers == 0 && (ok = issue_item(i, en, k, c, qb, bc0))) done = i + 1;
        }
      }
      if (!ok) {
        btc_flag(kStatusBtcTimeout);
        *abort_flag = 1;
        drain_own(done, 0);
      }
      if (slot) sched_leave(slot);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      const uint32_t idesc = idesc_16_f32(128, kN, a.f16 != 0);
      int i = 0, tl = 0;
      bool ok = true;
      for (; ok; ++tl) {
        const int b = tl & 1;
        if (!mbar_wait(&info_full[b], (tl >> 1) & 1, kWaitLimit) || *abort_flag) {
          ok = false;
          break;
        }
        const int tile = tile_id[b];
        if (tile < 0) break;
        if ((tl >= 1 && !mbar_wait(tmem_empty, (tl - 1) & 1, kWaitLimit)) || *abort_flag) {
          ok = false;
          break;
        }
        int qb, bc0, zg;
        tile_coords<S>(a, tile, &qb, &bc0, &zg);
        tc_fence_after();
        const int ne = info_cnt[b];
        const disco_grp_ent* info = infos + b * kMaxEnt;
        bool first = true;
        for (int j = 0; j < ne && ok; ++j) {
          const disco_grp_ent en = info[j];
          for (int k = 0; k < a.K && ok; ++k)
            for (int c = 0; c < en.nch; ++c, ++i) {
              const int s = i % kStages;
              const uint32_t ph = (i / kStages) & 1;
              if (!mbar_wait(&fullA[s], ph, kWaitLimit) || !mbar_wait(&fullB[s], ph, kWaitLimit) ||
                  *abort_flag) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t sbase = smem_u32(smem + (size_t)s * Cfg::kStageBytes);
              const uint32_t tbase = sbase + 2 * kBoxBytes;
              const bool narrow0 = box_is_narrow(qb - en.MW + 64 * c, a.Wout);
              const bool narrow1 = box_is_narrow(qb - en.MW + 64 * (c + 1), a.Wout);
              const int nsteps = min(4, (int)en.KB - 4 * c);
              for (int t = 0; t < nsteps; ++t) {
                const uint64_t bd = smem_desc_sw128(tbase + 32 * t);
                for (int blk = 0; blk < kNT; ++blk) {
                  const int as = t + blk * kStep1;  // K step within the chunk's boxes
                  const int bb = as >> 2, ka = as & 3;
                  const uint32_t slot = sbase + bb * kBoxBytes;
                  const uint64_t ad = (bb ? narrow1 : narrow0)
                                          ? smem_desc(slot + ka * 2 * kNarrowBytes, kNarrowBytes, 128)
                                          : smem_desc_sw128(slot + 32 * ka);
                  umma_bf16(tmem + blk * kN, ad, bd, idesc, (first && t == 0) ? 0u : 1u);
                }
              }
              first = false;
              umma_commit(&empty[s]);
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
        if (i > 0)  // let the MMAs in flight finish before TMEM is freed
          mbar_wait(&empty[(i - 1) % kStages], ((i - 1) / kStages) & 1, kWaitLimit);
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------- T builders (6 warps) --
    const int btid = tid - 64;
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
        const int KB = info[j].KB, nch = info[j].nch;
        for (int k = 0; k < a.K && ok; ++k)
          for (int c = 0; c < nch; ++c, ++i) {
            const int s = i % kStages;
            // the stage's copies are issued only after the MMAs of its previous item
            // completed; T needs only the psi block
            const bool mine = mbar_wait(&fullT[s], (i / kStages) & 1, kWaitLimit) && !*abort_flag;
            ok = all_named(mine, 1, kBuilderThreads);
            if (!ok) break;
            uint8_t* st = smem + (size_t)s * Cfg::kStageBytes;
            uint8_t* T = st + 2 * kBoxBytes;
            const uint16_t* tab = reinterpret_cast<const uint16_t*>(st + 2 * kBoxBytes + kTBytes);
            const int nq = 2 * min(4, KB - 4 * c);  // 16-byte chunks per T row
            // T[(r, t, p), 8 q8 + e] = tab[r][p][8 q8 + TQ - 1 - t + e]: the rows
            // t = 8 g + j (j = 0..7) of one (r, p, q8) read the same 16 table
            // values from the aligned index 8 q8 + TQ - 8 - 8 g on, shifted by
            // 7 - j.  One unit (r, p, g, q8) loads them with two 16-byte loads
            // and writes the 8 rows' chunks q8; q8 varies fastest across lanes
            // (conflict-free loads, and stores that cover all banks)
            constexpr int kG = TQ / 8;  // row groups of 8 t per (r, p)
            for (int u = btid; u < 8 * S * kG * nq; u += kBuilderThreads) {
              const int q8 = u % nq, rest = u / nq;
              const int g = rest % kG, rp = rest / kG;  // rp = r S + p
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
            fence_proxy_async_smem();
            mbar_arrive(&fullB[s]);
          }
      }
      if (!ok) break;
      mbar_arrive(&info_empty[b]);
    }
    if (!ok) {
      btc_flag(kStatusBtcTimeout);
      *abort_flag = 1;
    }
  } else if (warp >= 12) {
    // ----------------------------------- producers of items i % 3 == 1, 2 --
    const int who = warp - 11;
    if (lane == 0) {
      int i = 0, done = 0;
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
          for (int k = 0; k < a.K && ok; ++k)
            for (int c = 0; c < en.nch && ok; ++c, ++i)
              if (i % kProducers == who && (ok = issue_item(i, en, k, c, qb, bc0))) done = i + 1;
        }
        if (!ok) break;
        mbar_arrive(&info_empty[b]);
      }
      if (!ok) {
        btc_flag(kStatusBtcTimeout);
        *abort_flag = 1;
        drain_own(done, who);
      }
    }
  } else {
    // ----------------------------------------------- epilogue (warps 8-11) --
    const int q = warp & 3;
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
              tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + blk * kN + r * 32 + cc * 16, v);
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
      tc_fence_before();
      mbar_arrive(tmem_empty);
      mbar_arrive(&info_empty[b]);
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
  using Cfg = BCfg<S>;
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
  a.ntx = (a.Win + S * kNT * Cfg::TQ - 1) / (S * kNT * Cfg::TQ);
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
  auto kern = bwd_tc_kernel<S>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem) != cudaSuccess)
    return check_launch("disco_bwd (tensor cores) attribute");
  const long long ntiles = (long long)a.ntx * a.nty * a.ntz;
  const int grid = (int)(ntiles < sm_count() ? ntiles : sm_count());
  if (ntiles + grid > (long long)kSchedCountMask || grid > kSchedMaxCtas)
    return fail(DISCO_ERR_UNSUPPORTED, "problem too large");
  kern<<<grid, kThreads, Cfg::kSmem, st>>>(wide, narrow, gxm, a);
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
  static_assert(BCfg<1>::kSmem <= 227 * 1024 && BCfg<2>::kSmem <= 227 * 1024, "shared memory");
  return psi->s == 1 ? launch_btc<1>(psi, G, gx, BC, st, rows_of_channels, f16)
                     : launch_btc<2>(psi, G, gx, BC, st, rows_of_channels, f16);
}

// This unit's word of failed range checks (always 0 outside the bounds-checked build).
DISCO_BOUNDS_READER(btc_bounds)

}  // namespace disco
