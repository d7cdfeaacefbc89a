// disco_fwd_tc.cu -- the forward DISCO contraction on the tensor cores (bf16).
//
// DISCO Kernel Development Guide (torch-harmonics), §Architecture snapshot
// (the forward kernel: the sparse contraction of the input grid into
// X[B,C,K,H,W]) and §kpacked layout
// (psi values of all K side by side, which is what lets a tensor-core tile
// produce all basis functions at once; the page's WGMMA kernel is the Hopper
// form of the same idea).
//
// For one run (output row ho, input row hi) the contraction over the run's
// wrapped column window is a banded Toeplitz product.  For 16 consecutive
// output columns wo = w0 + t,
//
//   X[bc, k, ho, w0 + t] += sum_u x[bc, hi, u0 + u] * T[u, k*16 + t],
//   T[u, k*16 + t] = psi_k(delta = u - S*t - M)   (0 outside the run)
//
// with u0 = S*w0 - M and M = the run's half-width rounded up to 8, so that
// every 8-column group of the window starts on a 16-byte boundary and never
// straddles the longitude wrap.  That is an MMA with M = 128 channels,
// N = 16*K, and a K extent of the window length:
//   A = x window [128 channels x window columns]: TMA, one 2 KB box per
//       8-column group, wrapped column index, rows beyond B*C zero-filled;
//   B = T [16K x window columns], built in shared memory by 6 warps from the
//       psi values of the run (bf16);
//   D = X [128 channels x (k, t)] in TMEM, fp32, accumulated over all runs.
// One CTA owns (ho, 128 channels, NT tiles of 16 columns); the window of NT
// tiles is loaded once per 128-column chunk and shared by the NT MMAs (tile j
// starts S*16*j columns further into it).  Two pipeline stages; roles:
//   warp 0  TMA producer of A chunks (and TMEM owner)
//   warp 1  MMA issuer (one thread)
//   warps 2-7 build B chunks; warps 4-7 also run the epilogue
//             (tcgen05.ld of 16 columns = 16 consecutive wo of one k,
//              bf16 rounding, two 16-byte stores per thread).
// All mbarrier waits are bounded (time-out -> device status flag, abort).

#include <cudaTypedefs.h>

#include <cstring>

#include "disco_bounds.cuh"
#include "disco_internal.cuh"
#include "disco_sched.cuh"
#include "disco_umma.cuh"

namespace disco {

// status word of this translation unit (bit 2: a bounded wait timed out)
__device__ int g_tc_status = 0;

namespace {

constexpr int kThreads = 256;
constexpr int kBuilderThreads = 192;   // warps 2..7
constexpr int kTW = 16;                // output columns per MMA tile
constexpr int kCK = 4;                 // K steps (16 window columns) per chunk
constexpr int kChunkCols = kCK * 16;   // 64
constexpr uint32_t kBoxBytes = 128 * 128;   // one wide TMA box: 128 rows x 64 bf16 (128-byte swizzle)
constexpr uint32_t kNarrowBytes = 128 * 16; // one narrow box: 128 rows x 8 bf16 (no swizzle)
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr int kStatusTcTimeout = 4;

__device__ __forceinline__ void tc_flag(int bit) { atomicOr(&g_tc_status, bit); }

// true in every thread of the named-barrier group iff `pred` holds in all of them
__device__ __forceinline__ bool group_all_b(bool pred, int bar_id, int nthreads) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(bar_id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ int wrap_col(int c, int W) {
  int r = c % W;
  return r < 0 ? r + W : r;
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

struct TcArgs {
  __nv_bfloat16* X;   // [BC][K][Hout][Wout]
  const disco_run* runs;
  const int32_t* run_ptr;
  const int32_t* row_order;
  const int32_t* ftab_off;
  const uint16_t* ftab;  // per run: K rows of TL = roundup8(len + 16), psi_k(delta) at 8 + delta - dlo
  int BC, Hout, Wout, Win;
  int Hin;            // input rows (extent checks of the bounds-checked build)
  int nruns;          // runs, and ftab elements, of psi (the same checks)
  long long nftab;
  int TLB;            // table row capacity (>= every run's row length)
  int tma_store;      // X written by TMA stores (W_out % 8 == 0 and W_out >= one tile's columns)
  int f16;            // x, X and the tables are fp16 (else bf16)
  unsigned long long launch_id;  // selects the scheduler slot of the persistent form
};

__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// geometry of one run for the Toeplitz tiles
struct RunGeom {
  int hi, e0, dlo, len, M, KS, TL;
};

template <int S>
__device__ __forceinline__ RunGeom run_geom(const disco_run& r, int Win) {
  RunGeom g;
  g.hi = r.hi;
  g.e0 = r.e0;
  g.len = r.len;
  g.dlo = (r.len == Win) ? -(Win / 2) : -r.npair;
  g.M = ((-g.dlo) + 7) & ~7;
  const int L = S * (kTW - 1) + 2 * g.M + 1;
  g.KS = (L + 15) >> 4;
  g.TL = (r.len + 16 + 7) & ~7;
  return g;
}

// Builder of one K-chunk of T (the B operand, [16 K rows (k, t)] x [64 window
// columns], 128-byte swizzled): T[(k, t), 8 gi + e] = tab[k][x0 + e] with
// x0 = off + 8 gi - S t, zero where x0 + e lies outside the run's table row
// [0, TL) (the table holds psi_k of offset delta at index 8 + delta - dlo,
// so off = 8 + 64 c - M - dlo for chunk c).  The rows t = 8 g + j
// (j = 0..7) of one (k, gi) read one stretch of the table row starting at
// lo = off + 8 gi - 8 S g - 7 S; lo mod 8 (sh) is the same for the whole run,
// so one unit (k, g, gi) loads the stretch as four aligned 16-byte blocks
// (each wholly inside or outside [0, TL), both multiples of 8) and writes its
// 8 rows with shifts known at compile time, in one of 8 variants picked by
// sh.  gi varies fastest across threads: conflict-free loads and stores.
template <int S, int SH>
__device__ __forceinline__ void t_rows(const uint32_t (&v)[16], uint8_t* sB, int n0, int gi) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int m = SH + S * (7 - j);  // first value of row j within the stretch
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = (m & 1) ? __funnelshift_r(v[m / 2 + e], v[m / 2 + e + 1], 16) : v[m / 2 + e];
    const int n = n0 + j;
    *reinterpret_cast<uint4*>(sB + n * 128 + ((gi ^ (n & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <int K, int S>
__device__ __forceinline__ void build_t_chunk(const uint16_t* tab, int TL, int off, int ngrp, uint8_t* sB,
                                              int btid, int nthreads) {
  const int sh = (off - 7 * S) & 7;
  for (int u = btid; u < K * 2 * ngrp; u += nthreads) {
    const int gi = u % ngrp, kg = u / ngrp;  // kg = 2 k + g
    const int k = kg >> 1, g = kg & 1;
    const int lo = off + 8 * gi - 8 * S * g - 7 * S;
    const int A = lo - sh;  // multiple of 8
    const uint16_t* row = tab + (size_t)k * TL;
    uint32_t v[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int x = A + 8 * q;
      const uint4 b = (x >= 0 && x < TL) ? *reinterpret_cast<const uint4*>(row + x) : make_uint4(0u, 0u, 0u, 0u);
      v[4 * q] = b.x;
      v[4 * q + 1] = b.y;
      v[4 * q + 2] = b.z;
      v[4 * q + 3] = b.w;
    }
    const int n0 = k * 16 + 8 * g;
    switch (sh) {  // the same in every thread
      case 0: t_rows<S, 0>(v, sB, n0, gi); break;
      case 1: t_rows<S, 1>(v, sB, n0, gi); break;
      case 2: t_rows<S, 2>(v, sB, n0, gi); break;
      case 3: t_rows<S, 3>(v, sB, n0, gi); break;
      case 4: t_rows<S, 4>(v, sB, n0, gi); break;
      case 5: t_rows<S, 5>(v, sB, n0, gi); break;
      case 6: t_rows<S, 6>(v, sB, n0, gi); break;
      default: t_rows<S, 7>(v, sB, n0, gi); break;
    }
  }
}

template <int K, int S, int STAGES>
struct TcCfg {
  static constexpr int N = 16 * K;                           // MMA N
  static constexpr uint32_t kBBytes = N * kChunkCols * 2;    // B chunk (128-byte rows)
  static constexpr int NT = (512 / N) < 4 ? (512 / N) : 4;   // tiles per CTA
  // 64-column boxes covering the chunk's window for all NT tiles
  static constexpr int NBOX = (kChunkCols + S * kTW * (NT - 1) + 63) / 64;
  static constexpr uint32_t kABytes = NBOX * kBoxBytes;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;  // multiple of 1024
  static constexpr uint32_t kTmemCols = (NT * N <= 32) ? 32 : (NT * N <= 64) ? 64 : (NT * N <= 128) ? 128
                                        : (NT * N <= 256) ? 256 : 512;
  static constexpr size_t kFixed = (size_t)STAGES * kStageBytes + 256 + 1024;  // + alignment slack
  // the epilogue stages the X tile [K][128 channels][NT*16 columns] (bf16) in
  // the freed pipeline buffers and writes it with TMA stores when it fits
  static constexpr uint32_t kOutRow = NT * kTW * 2;            // bytes of one channel row
  static constexpr uint32_t kOutBytes = (uint32_t)K * 128 * kOutRow;
  static constexpr bool kTmaStore = kOutBytes <= (uint32_t)STAGES * kStageBytes;
  // two psi table buffers (double-buffered across runs): K rows x TLB bf16 each
  __host__ __device__ static size_t tab_bytes(int TLB) { return ((size_t)K * TLB * 2 + 127) & ~(size_t)127; }
  static size_t smem(int TLB) { return kFixed + 2 * tab_bytes(TLB); }
};

template <int K, int S, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap xnarrow,
                  const __grid_constant__ CUtensorMap outmap, const TcArgs a) {
  using Cfg = TcCfg<K, S, STAGES>;
  constexpr int N = Cfg::N, NT = Cfg::NT;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled operand tiles
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * Cfg::kStageBytes);
  uint64_t* fullA = bars;                 // [STAGES] TMA bytes landed
  uint64_t* fullB = bars + STAGES;        // [STAGES] B chunk built (192 arrivals)
  uint64_t* empty = bars + 2 * STAGES;    // [STAGES] MMAs of the stage done (commit)
  uint64_t* done = bars + 3 * STAGES;     // all MMAs done (commit)
  uint64_t* tfull = bars + 3 * STAGES + 1;   // [2] run table landed (bulk copy bytes)
  uint64_t* tempty = bars + 3 * STAGES + 3;  // [2] run table released (192 builder arrivals)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 3 * STAGES + 6);
  // psi tables of two consecutive runs: [2][K][TLB] bf16
  uint8_t* tabs = smem + STAGES * Cfg::kStageBytes + 256;
  const size_t tab_bytes = Cfg::tab_bytes(a.TLB);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int ho = a.row_order[blockIdx.z];
  if (!DISCO_IN_BOUNDS(ho >= 0 && ho < a.Hout)) ho = 0;
  const int bc0 = blockIdx.y * 128;
  const int wc = blockIdx.x * (kTW * NT);
  const int r_begin = a.run_ptr[ho];
  int r_end = a.run_ptr[ho + 1];
  if (!DISCO_IN_BOUNDS(r_begin >= 0 && r_begin <= r_end && r_end <= a.nruns)) r_end = r_begin;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&fullA[s], 1);
      mbar_init(&fullB[s], kBuilderThreads);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kBuilderThreads);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, Cfg::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  // number of work items (run, chunk) of this row
  int items = 0;
  for (int r = r_begin; r < r_end; ++r) items += (run_geom<S>(a.runs[r], a.Win).KS + kCK - 1) / kCK;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int i = 0;
      bool aborted = false;
      for (int r = r_begin; r < r_end && !aborted; ++r) {
        const RunGeom g = run_geom<S>(a.runs[r], a.Win);
        const int u0 = S * wc - g.M;
        {
          // the run's psi table into buffer (run index & 1), once the builders released it
          const int rl = r - r_begin, b = rl & 1;
          if (rl >= 2 && !mbar_wait(&tempty[b], ((rl >> 1) - 1) & 1, kWaitLimit)) {
            tc_flag(kStatusTcTimeout);
            *abort_flag = 1;
            aborted = true;
            break;
          }
          const uint32_t bytes = (uint32_t)K * g.TL * 2;
          mbar_expect_tx(&tfull[b], bytes);
          if (DISCO_IN_BOUNDS(g.TL <= a.TLB && a.ftab_off[r] >= 0 && a.ftab_off[r] + (long long)K * g.TL <= a.nftab))
            bulk_copy(tabs + b * tab_bytes, a.ftab + a.ftab_off[r], bytes, &tfull[b]);
          else
            mbar_complete_tx(&tfull[b], bytes);
        }
        for (int c = 0; c * kCK < g.KS; ++c, ++i) {
          const int s = i % STAGES;
          if ((i >= STAGES && !mbar_wait(&empty[s], ((i / STAGES) - 1) & 1, kWaitLimit)) || *abort_flag) {
            tc_flag(kStatusTcTimeout);
            *abort_flag = 1;
            aborted = true;
            break;
          }
          const int nks = min(kCK, g.KS - c * kCK);
          // boxes holding window columns [64 c, 64 c + 16 nks + S*16*(NT-1))
          const int nbox = (16 * nks + S * kTW * (NT - 1) + 63) / 64;
          uint8_t* sA = smem + s * Cfg::kStageBytes;
          mbar_expect_tx(&fullA[s], nbox * kBoxBytes);
          for (int bb = 0; bb < nbox; ++bb) {
            const int col = wrap_col(u0 + c * kChunkCols + 64 * bb, a.Win);
            [[maybe_unused]] const bool rows_ok = DISCO_IN_BOUNDS(g.hi >= 0 && g.hi < a.Hin && bc0 >= 0 && bc0 < a.BC);
            if (col + 64 <= a.Win) {
              if (DISCO_IN_BOUNDS(rows_ok && col >= 0))
                tma_load_3d(sA + bb * kBoxBytes, &xmap, col, g.hi, bc0, &fullA[s]);
              else
                mbar_complete_tx(&fullA[s], kBoxBytes);
            } else {  // crosses the longitude seam: 8 wrapped narrow boxes
              for (int gi = 0; gi < 8; ++gi) {
                const int cn = wrap_col(col + 8 * gi, a.Win);
                if (DISCO_IN_BOUNDS(rows_ok && cn >= 0 && cn + 8 <= a.Win))
                  tma_load_3d(sA + bb * kBoxBytes + gi * kNarrowBytes, &xnarrow, cn, g.hi, bc0, &fullA[s]);
                else
                  mbar_complete_tx(&fullA[s], kNarrowBytes);
              }
            }
          }
        }
      }
      if (aborted) {
        // let the copies this thread issued land (bounded) before the CTA exits
        for (int back = 1; back <= STAGES && i - back >= 0; ++back) {
          const int li = i - back;
          mbar_wait(&fullA[li % STAGES], (li / STAGES) & 1, kWaitLimit);
        }
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      const uint32_t idesc = idesc_16_f32(128, N, a.f16 != 0);
      int i = 0;
      bool ok = true;
      for (int r = r_begin; r < r_end && ok; ++r) {
        const RunGeom g = run_geom<S>(a.runs[r], a.Win);
        for (int c = 0; c * kCK < g.KS; ++c, ++i) {
          const int s = i % STAGES;
          const uint32_t ph = (i / STAGES) & 1;
          if (!mbar_wait(&fullA[s], ph, kWaitLimit) || !mbar_wait(&fullB[s], ph, kWaitLimit) ||
              *abort_flag) {
            tc_flag(kStatusTcTimeout);
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const int nks = min(kCK, g.KS - c * kCK);
          const uint32_t abase = smem_u32(smem + s * Cfg::kStageBytes);
          const uint32_t bbase = abase + Cfg::kABytes;
          const int u0 = S * wc - g.M;
          bool narrow[Cfg::NBOX];
#pragma unroll
          for (int bb = 0; bb < Cfg::NBOX; ++bb)
            narrow[bb] = wrap_col(u0 + c * kChunkCols + 64 * bb, a.Win) + 64 > a.Win;
          for (int j = 0; j < NT; ++j)
            for (int ks = 0; ks < nks; ++ks) {
              // window column of the K step inside the stage, its box and its step in the box
              const int col = 16 * ks + S * kTW * j;
              const int bb = col >> 6, ka = (col & 63) >> 4;
              bool nb = false;
#pragma unroll
              for (int q = 0; q < Cfg::NBOX; ++q)
                if (q == bb) nb = narrow[q];
              const uint32_t slot = abase + bb * kBoxBytes;
              const uint64_t ad = nb ? smem_desc(slot + ka * 2 * kNarrowBytes, kNarrowBytes, 128)
                                     : smem_desc_sw128(slot + 32 * ka);
              const uint64_t bd = smem_desc_sw128(bbase + 32 * ks);
              umma_bf16(tmem + j * N, ad, bd, idesc, (i > 0 || ks > 0) ? 1u : 0u);
            }
          umma_commit(&empty[s]);
        }
      }
      umma_commit(done);  // arrives when every MMA issued above has completed
    }
  } else {
    // ------------------------------------------------- B builders (6 warps) --
    const int btid = tid - 64;
    int i = 0;
    bool ok = true;
    for (int r = r_begin; r < r_end && ok; ++r) {
      const RunGeom g = run_geom<S>(a.runs[r], a.Win);
      const int rl = r - r_begin, tb = rl & 1;
      const uint16_t* tab = reinterpret_cast<const uint16_t*>(tabs + tb * tab_bytes);
      {
        bool mine = mbar_wait(&tfull[tb], (rl >> 1) & 1, kWaitLimit) && !*abort_flag;
        if (!mine) {
          tc_flag(kStatusTcTimeout);
          *abort_flag = 1;
        }
        ok = group_all_b(mine, 1, kBuilderThreads);
        if (!ok) break;
      }
      for (int c = 0; c * kCK < g.KS; ++c, ++i) {
        const int s = i % STAGES;
        bool mine = true;
        if (i >= STAGES) mine = mbar_wait(&empty[s], ((i / STAGES) - 1) & 1, kWaitLimit);
        mine = mine && !*abort_flag;
        if (!mine) {
          tc_flag(kStatusTcTimeout);
          *abort_flag = 1;
        }
        ok = group_all_b(mine, 1, kBuilderThreads);
        if (!ok) break;
        uint8_t* sB = smem + s * Cfg::kStageBytes + Cfg::kABytes;
        const int nks = min(kCK, g.KS - c * kCK);
        const int ngrp = 2 * nks;  // 8-column groups of this chunk
        build_t_chunk<K, S>(tab, g.TL, 8 + c * kChunkCols - g.M - g.dlo, ngrp, sB, btid, kBuilderThreads);
        fence_proxy_async_smem();
        mbar_arrive(&fullB[s]);
      }
      if (ok) mbar_arrive(&tempty[tb]);  // this run's table is no longer read
    }
    // ------------------------------------------------ epilogue (warps 4-7) --
    if (warp >= 4) {
      const int q = warp & 3;
      bool fin = mbar_wait(done, 0, kWaitLimit);
      fin = __all_sync(0xffffffffu, fin) && !*abort_flag;
      if (!fin) {
        if (lane == 0) tc_flag(kStatusTcTimeout);
      } else if (Cfg::kTmaStore && a.tma_store) {
        tc_fence_after();
        // X tile through shared memory (the pipeline buffers are free once every
        // MMA has completed), then one TMA store per k of [128 channels x NT*16
        // columns]; the store clips columns >= W_out and channels >= B*C
        const int r = q * 32 + lane;
        for (int k = 0; k < K; ++k)
          for (int j = 0; j < NT; ++j) {
            float v[16];
            if (items > 0) {
              tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + j * N + k * 16, v);
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] = 0.f;
            }
            uint32_t w32[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              w32[e] = pack2_16(v[2 * e], v[2 * e + 1], a.f16);
            }
            uint4* dst = reinterpret_cast<uint4*>(smem + ((size_t)k * 128 + r) * Cfg::kOutRow + j * kTW * 2);
            dst[0] = make_uint4(w32[0], w32[1], w32[2], w32[3]);
            dst[1] = make_uint4(w32[4], w32[5], w32[6], w32[7]);
          }
        fence_proxy_async_smem();
        asm volatile("bar.sync 2, 128;" ::: "memory");
        if (warp == 4 && lane == 0) {
          for (int k = 0; k < K; ++k)
            if (DISCO_IN_BOUNDS(wc >= 0 && wc < a.Wout && ho >= 0 && ho < a.Hout && bc0 >= 0 && bc0 < a.BC))
              asm volatile(
                "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                    reinterpret_cast<uint64_t>(&outmap)),
                "r"(wc), "r"(k * a.Hout + ho), "r"(bc0), "r"(smem_u32(smem + (size_t)k * 128 * Cfg::kOutRow))
                : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // shared memory read out
        }
      } else {
        tc_fence_after();
        const int bc = bc0 + q * 32 + lane;
        for (int j = 0; j < NT; ++j) {
          const int wo = wc + j * kTW;
          for (int k = 0; k < K; ++k) {
            float v[16];
            if (items > 0) {
              tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + j * N + k * 16, v);
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] = 0.f;
            }
            if (bc < a.BC && wo < a.Wout) {
              __nv_bfloat16* dst = a.X + (((size_t)bc * K + k) * a.Hout + ho) * a.Wout + wo;
              const int n = min(16, a.Wout - wo);
              // 16-byte stores need 16-byte aligned rows: W_out % 8 == 0 (wo is a multiple of 16)
              if (n == 16 && (a.Wout & 7) == 0) {
                uint32_t w32[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  w32[e] = pack2_16(v[2 * e], v[2 * e + 1], a.f16);
                }
                reinterpret_cast<uint4*>(dst)[0] = make_uint4(w32[0], w32[1], w32[2], w32[3]);
                reinterpret_cast<uint4*>(dst)[1] = make_uint4(w32[4], w32[5], w32[6], w32[7]);
              } else {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  if (e < n) reinterpret_cast<uint16_t*>(dst)[e] = round_16(v[e], a.f16);
              }
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

// ---------------------------------------------------- persistent form --
//
// The same tiles, items and operands, but one CTA per SM takes tile after
// tile (output row in launch order, 128 channels, NT*16 columns) from the
// launch's scheduler counter (disco_sched.cuh) and hands each tile index to
// the other roles through a 4-slot ring in shared memory.  Its pipeline runs
// across tile boundaries: the next tile's x windows and
// psi tables load and its T chunks build while the epilogue writes the
// previous tile.  The epilogue has its own warps (8-11) and writes X one
// basis function at a time ([128 channels x NT*16 columns]) through a
// two-piece shared-memory ring with TMA stores.  The accumulators (NT*N <=
// 512 columns) are single-buffered: a tile's first MMA waits for the
// epilogue to have read the previous tile out.
constexpr int kPThreads = 384;
constexpr int kPEpiThreads = 128;  // warps 8-11
constexpr int kRing = 4;           // tile indices in flight between the producer and the consumers

__device__ unsigned long long g_fwd_sched[kSchedSlots];

// Consumer side of the tile ring: the tl-th tile index (-1 once there are no
// more), or -2 when the wait timed out or the CTA aborts.  Every consumer
// thread arrives on the slot's empty barrier after reading it.
__device__ __forceinline__ int ring_take(uint64_t* full, uint64_t* empty, volatile int* ring, int tl,
                                         volatile int* abort_flag) {
  const int b = tl % kRing;
  if (!mbar_wait(&full[b], (tl / kRing) & 1, kWaitLimit) || *abort_flag) return -2;
  const int t = ring[b];
  mbar_arrive(&empty[b]);
  return t;
}

template <int K, int S>
struct PCfg {
  using C = TcCfg<K, S, 3>;
  static constexpr int kStages = 3;
  static constexpr uint32_t kPiece = 128 * C::kOutRow;  // one basis function of a tile
  static size_t smem(int TLB) {
    return (size_t)kStages * C::kStageBytes + 2 * C::tab_bytes(TLB) + 2 * kPiece + 256 + 1024;
  }
};

template <int K, int S>
__global__ void __launch_bounds__(kPThreads, 1)
    fwd_tcp_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap xnarrow,
                   const __grid_constant__ CUtensorMap outmap, const TcArgs a) {
  using Cfg = TcCfg<K, S, 3>;
  using P = PCfg<K, S>;
  constexpr int STAGES = P::kStages;
  constexpr int N = Cfg::N, NT = Cfg::NT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const size_t tab_bytes = Cfg::tab_bytes(a.TLB);
  uint8_t* tabs = smem + STAGES * Cfg::kStageBytes;          // [2] run tables
  uint8_t* pieces = tabs + 2 * tab_bytes;                     // [2] X pieces for the TMA stores
  uint64_t* bars = reinterpret_cast<uint64_t*>(pieces + 2 * P::kPiece);
  uint64_t* fullA = bars;                    // [STAGES]
  uint64_t* fullB = bars + STAGES;           // [STAGES] (192 arrivals)
  uint64_t* empty = bars + 2 * STAGES;       // [STAGES] (commit)
  uint64_t* tfull = bars + 3 * STAGES;       // [2] run table landed
  uint64_t* tempty = bars + 3 * STAGES + 2;  // [2] run table released (192 arrivals)
  uint64_t* acc_full = bars + 3 * STAGES + 4;   // tile's MMAs done (commit)
  uint64_t* tmem_empty = bars + 3 * STAGES + 5; // epilogue read the tile out (128 arrivals)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 6);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 3 * STAGES + 7);
  uint64_t* ring_full = bars + 3 * STAGES + 8;    // [4] tile index written (producer)
  uint64_t* ring_empty = bars + 3 * STAGES + 12;  // [4] tile index read by every consumer
  volatile int* ring = reinterpret_cast<volatile int*>(bars + 3 * STAGES + 16);  // [4], -1 = no more tiles

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntx = (a.Wout + kTW * NT - 1) / (kTW * NT), nty = (a.BC + 127) / 128;
  const int ntiles = ntx * nty * a.Hout;
  auto coords = [&](int t, int* ho, int* bc0, int* wc) {
    *wc = (t % ntx) * (kTW * NT);
    const int r = t / ntx;
    *bc0 = (r / a.Hout) * 128;
    *ho = a.row_order[r % a.Hout];
    if (!DISCO_IN_BOUNDS(*ho >= 0 && *ho < a.Hout)) *ho = 0;
  };
  // runs of output row ho; every role clips a bad range the same way
  auto row_runs = [&](int ho, int* rb, int* re) {
    *rb = a.run_ptr[ho];
    *re = a.run_ptr[ho + 1];
    if (!DISCO_IN_BOUNDS(*rb >= 0 && *rb <= *re && *re <= a.nruns)) *re = *rb;
  };

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&fullA[s], 1);
      mbar_init(&fullB[s], kBuilderThreads);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kBuilderThreads);
    }
    mbar_init(acc_full, 1);
    mbar_init(tmem_empty, kPEpiThreads);
    for (int b = 0; b < kRing; ++b) {
      mbar_init(&ring_full[b], 1);
      mbar_init(&ring_empty[b], 1 + kBuilderThreads + kPEpiThreads);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, Cfg::kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int i = 0, rl = 0;
      bool ok = true;
      unsigned long long* slot = sched_join(g_fwd_sched, a.launch_id, kWaitLimit);
      if (!slot) tc_flag(kStatusTcTimeout);  // this CTA takes no tile
      for (int tl = 0; ok; ++tl) {
        const int rb = tl % kRing;
        if ((tl >= kRing && !mbar_wait(&ring_empty[rb], ((tl / kRing) - 1) & 1, kWaitLimit)) || *abort_flag) {
          ok = false;
          break;
        }
        const int t = slot ? sched_next(slot) : ntiles;
        ring[rb] = t < ntiles ? t : -1;
        mbar_arrive(&ring_full[rb]);
        if (t >= ntiles) break;
        int ho, bc0, wc;
        coords(t, &ho, &bc0, &wc);
        int r_beg, r_end;
        row_runs(ho, &r_beg, &r_end);
        for (int r = r_beg; r < r_end && ok; ++r, ++rl) {
          const RunGeom g = run_geom<S>(a.runs[r], a.Win);
          const int u0 = S * wc - g.M;
          const int b = rl & 1;
          if ((rl >= 2 && !mbar_wait(&tempty[b], ((rl >> 1) - 1) & 1, kWaitLimit)) || *abort_flag) {
            ok = false;
            break;
          }
          const uint32_t bytes = (uint32_t)K * g.TL * 2;
          mbar_expect_tx(&tfull[b], bytes);
          if (DISCO_IN_BOUNDS(g.TL <= a.TLB && a.ftab_off[r] >= 0 && a.ftab_off[r] + (long long)K * g.TL <= a.nftab))
            bulk_copy(tabs + b * tab_bytes, a.ftab + a.ftab_off[r], bytes, &tfull[b]);
          else
            mbar_complete_tx(&tfull[b], bytes);
          for (int c = 0; c * kCK < g.KS; ++c, ++i) {
            const int s = i % STAGES;
            if ((i >= STAGES && !mbar_wait(&empty[s], ((i / STAGES) - 1) & 1, kWaitLimit)) || *abort_flag) {
              ok = false;  // (the r loop's increment still counts this run's table copy)
              break;
            }
            const int nks = min(kCK, g.KS - c * kCK);
            const int nbox = (16 * nks + S * kTW * (NT - 1) + 63) / 64;
            uint8_t* sA = smem + s * Cfg::kStageBytes;
            mbar_expect_tx(&fullA[s], nbox * kBoxBytes);
            for (int bb = 0; bb < nbox; ++bb) {
              const int col = wrap_col(u0 + c * kChunkCols + 64 * bb, a.Win);
              [[maybe_unused]] const bool rows_ok = DISCO_IN_BOUNDS(g.hi >= 0 && g.hi < a.Hin && bc0 >= 0 && bc0 < a.BC);
              if (col + 64 <= a.Win) {
                if (DISCO_IN_BOUNDS(rows_ok && col >= 0))
                  tma_load_3d(sA + bb * kBoxBytes, &xmap, col, g.hi, bc0, &fullA[s]);
                else
                  mbar_complete_tx(&fullA[s], kBoxBytes);
              } else {
                for (int gi = 0; gi < 8; ++gi) {
                  const int cn = wrap_col(col + 8 * gi, a.Win);
                  if (DISCO_IN_BOUNDS(rows_ok && cn >= 0 && cn + 8 <= a.Win))
                    tma_load_3d(sA + bb * kBoxBytes + gi * kNarrowBytes, &xnarrow, cn, g.hi, bc0, &fullA[s]);
                  else
                    mbar_complete_tx(&fullA[s], kNarrowBytes);
                }
              }
            }
          }
        }
      }
      if (!ok) {
        tc_flag(kStatusTcTimeout);
        *abort_flag = 1;
        for (int back = 1; back <= STAGES && i - back >= 0; ++back) {
          const int li = i - back;
          mbar_wait(&fullA[li % STAGES], (li / STAGES) & 1, kWaitLimit);
        }
        for (int back = 1; back <= 2 && rl - back >= 0; ++back) {
          const int lr = rl - back;
          mbar_wait(&tfull[lr & 1], (lr >> 1) & 1, kWaitLimit);
        }
      }
      if (slot) sched_leave(slot);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      const uint32_t idesc = idesc_16_f32(128, N, a.f16 != 0);
      int i = 0, tl = 0;
      bool ok = true;
      for (; ok; ++tl) {
        const int t = ring_take(ring_full, ring_empty, ring, tl, abort_flag);
        if (t == -1) break;
        if (t < 0) {
          ok = false;
          break;
        }
        int ho, bc0, wc;
        coords(t, &ho, &bc0, &wc);
        if ((tl >= 1 && !mbar_wait(tmem_empty, (tl - 1) & 1, kWaitLimit)) || *abort_flag) {
          ok = false;
          break;
        }
        tc_fence_after();
        bool first = true;
        int r_beg, r_end;
        row_runs(ho, &r_beg, &r_end);
        for (int r = r_beg; r < r_end && ok; ++r) {
          const RunGeom g = run_geom<S>(a.runs[r], a.Win);
          for (int c = 0; c * kCK < g.KS; ++c, ++i) {
            const int s = i % STAGES;
            const uint32_t ph = (i / STAGES) & 1;
            if (!mbar_wait(&fullA[s], ph, kWaitLimit) || !mbar_wait(&fullB[s], ph, kWaitLimit) || *abort_flag) {
              ok = false;
              break;
            }
            tc_fence_after();
            const int nks = min(kCK, g.KS - c * kCK);
            const uint32_t abase = smem_u32(smem + s * Cfg::kStageBytes);
            const uint32_t bbase = abase + Cfg::kABytes;
            const int u0 = S * wc - g.M;
            // descriptors of every (tile block, K step) first, then the MMAs back to back
            uint64_t dbox[Cfg::NBOX];
            bool narrow[Cfg::NBOX];
#pragma unroll
            for (int bb = 0; bb < Cfg::NBOX; ++bb) {
              narrow[bb] = wrap_col(u0 + c * kChunkCols + 64 * bb, a.Win) + 64 > a.Win;
              dbox[bb] = narrow[bb] ? smem_desc(abase + bb * kBoxBytes, kNarrowBytes, 128)
                                    : smem_desc_sw128(abase + bb * kBoxBytes);
            }
            const uint64_t dB = smem_desc_sw128(bbase);
            const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
              for (int ks = 0; ks < kCK; ++ks) {
                // window column of the K step inside the stage: its box and its step in the box
                const int col = 16 * ks + S * kTW * j;
                const int bb = col >> 6, ka = (col & 63) >> 4;
                const uint64_t ad = dbox[bb] + (uint64_t)(narrow[bb] ? ka * (2 * kNarrowBytes >> 4) : ka * 2);
                if (ks < nks)
                  umma_bf16(tmem + j * N, ad, dB + (uint64_t)(ks * 2), idesc, ks == 0 ? acc0 : 1u);
              }
            first = false;
            umma_commit(&empty[s]);
          }
        }
        if (!ok) break;
        // a tile without runs leaves the accumulators unwritten: the epilogue stores zeros
        umma_commit(acc_full);
      }
      if (!ok) {
        tc_flag(kStatusTcTimeout);
        *abort_flag = 1;
        if (i > 0) mbar_wait(&empty[(i - 1) % STAGES], ((i - 1) / STAGES) & 1, kWaitLimit);
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------- B builders (6 warps) --
    const int btid = tid - 64;
    int i = 0, rl = 0;
    bool ok = true;
    for (int tl = 0; ok; ++tl) {
      const int t = ring_take(ring_full, ring_empty, ring, tl, abort_flag);
      ok = group_all_b(t != -2, 1, kBuilderThreads);  // one decision for the 6 warps
      if (!ok || t == -1) break;
      int ho, bc0, wc;
      coords(t, &ho, &bc0, &wc);
      int r_beg, r_end;
      row_runs(ho, &r_beg, &r_end);
      for (int r = r_beg; r < r_end && ok; ++r, ++rl) {
        const RunGeom g = run_geom<S>(a.runs[r], a.Win);
        const int tb = rl & 1;
        const uint16_t* tab = reinterpret_cast<const uint16_t*>(tabs + tb * tab_bytes);
        {
          const bool mine = mbar_wait(&tfull[tb], (rl >> 1) & 1, kWaitLimit) && !*abort_flag;
          ok = group_all_b(mine, 1, kBuilderThreads);
          if (!ok) break;
        }
        for (int c = 0; c * kCK < g.KS; ++c, ++i) {
          const int s = i % STAGES;
          bool mine = true;
          if (i >= STAGES) mine = mbar_wait(&empty[s], ((i / STAGES) - 1) & 1, kWaitLimit);
          ok = group_all_b(mine && !*abort_flag, 1, kBuilderThreads);
          if (!ok) break;
          uint8_t* sB = smem + s * Cfg::kStageBytes + Cfg::kABytes;
          const int nks = min(kCK, g.KS - c * kCK);
          const int ngrp = 2 * nks;
          build_t_chunk<K, S>(tab, g.TL, 8 + c * kChunkCols - g.M - g.dlo, ngrp, sB, btid, kBuilderThreads);
          fence_proxy_async_smem();
          mbar_arrive(&fullB[s]);
        }
        if (!ok) break;
        mbar_arrive(&tempty[tb]);  // this run's table is no longer read
      }
    }
    if (!ok) {
      tc_flag(kStatusTcTimeout);
      *abort_flag = 1;
    }
  } else {
    // ---------------------------------------------- epilogue (warps 8-11) --
    const int q = warp & 3;
    const int er = q * 32 + lane;  // channel row of this thread in a piece
    int npiece = 0;
    for (int tl = 0;; ++tl) {
      const int t = ring_take(ring_full, ring_empty, ring, tl, abort_flag);
      if (!group_all_b(t != -2, 2, kPEpiThreads)) {
        if (lane == 0) tc_flag(kStatusTcTimeout);
        *abort_flag = 1;
        break;
      }
      if (t == -1) break;
      int ho, bc0, wc;
      coords(t, &ho, &bc0, &wc);
      int r_beg, r_end;
      row_runs(ho, &r_beg, &r_end);
      const bool any = r_end > r_beg;
      bool fin = mbar_wait(acc_full, tl & 1, kWaitLimit) && !*abort_flag;
      fin = group_all_b(fin, 2, kPEpiThreads);  // one decision for the 4 warps (named barriers below)
      if (!fin) {
        if (lane == 0) tc_flag(kStatusTcTimeout);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      for (int k = 0; k < K; ++k, ++npiece) {
        uint8_t* pb = pieces + (npiece & 1) * P::kPiece;
        if (tid == 256) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");  // buffer free
        asm volatile("bar.sync 2, 128;" ::: "memory");
        for (int j = 0; j < NT; ++j) {
          float v[16];
          if (any) {
            tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + j * N + k * 16, v);
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = 0.f;
          }
          uint32_t w32[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            w32[e] = pack2_16(v[2 * e], v[2 * e + 1], a.f16);
          }
          uint4* dst = reinterpret_cast<uint4*>(pb + (size_t)er * Cfg::kOutRow + j * kTW * 2);
          dst[0] = make_uint4(w32[0], w32[1], w32[2], w32[3]);
          dst[1] = make_uint4(w32[4], w32[5], w32[6], w32[7]);
        }
        if (k == K - 1) {  // every accumulator read: the next tile's MMAs may start
          tc_fence_before();
          mbar_arrive(tmem_empty);
        }
        fence_proxy_async_smem();
        asm volatile("bar.sync 2, 128;" ::: "memory");
        if (tid == 256) {
          if (DISCO_IN_BOUNDS(wc >= 0 && wc < a.Wout && ho >= 0 && ho < a.Hout && bc0 >= 0 && bc0 < a.BC))
            asm volatile(
              "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                  reinterpret_cast<uint64_t>(&outmap)),
              "r"(wc), "r"(k * a.Hout + ho), "r"(bc0), "r"(smem_u32(pb))
              : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
      }
    }
    if (tid == 256) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

int sm_count_f() {
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

template <int K, int S, int STAGES>
int launch_tc_stages(const disco_psi* psi, const CUtensorMap& map, const CUtensorMap& nmap,
                     const CUtensorMap& omap, TcArgs a, cudaStream_t st) {
  using Cfg = TcCfg<K, S, STAGES>;
  const size_t smem = Cfg::smem(a.TLB);
  auto kern = fwd_tc_kernel<K, S, STAGES>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return check_launch("disco_fwd (tensor cores) attribute");
  dim3 grid((a.Wout + kTW * Cfg::NT - 1) / (kTW * Cfg::NT), (a.BC + 127) / 128, a.Hout);
  kern<<<grid, kThreads, smem, st>>>(map, nmap, omap, a);
  return check_launch("disco_fwd (tensor cores)");
}

template <int K, int S>
int launch_tc(const disco_psi* psi, const void* x, void* X, int BC, cudaStream_t st, bool f16) {
  constexpr size_t kMaxSmem = 227 * 1024;
  const CUtensorMapDataType dt16 = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int Hin = psi->grid_in.nlat, Win = psi->grid_in.nlon;
  TcArgs a;
  a.X = (__nv_bfloat16*)X;
  a.runs = psi->runs;
  a.run_ptr = psi->run_ptr;
  a.row_order = psi->row_order;
  a.ftab_off = psi->ftab_off;
  a.ftab = f16 ? psi->ftab_h : psi->ftab;
  a.f16 = f16 ? 1 : 0;
  a.BC = BC;
  a.Hout = psi->grid_out.nlat;
  a.Wout = psi->grid_out.nlon;
  a.Win = Win;
  a.TLB = (Win + 16 + 7) & ~7;  // a run is at most one ring long
  a.Hin = Hin;
  a.nruns = (int)psi->nruns;
  a.nftab = psi->nftab;
  if (!a.ftab || !psi->ftab_off) return DISCO_ERR_UNSUPPORTED;
  const bool fit3 = TcCfg<K, S, 3>::smem(a.TLB) <= kMaxSmem;
  const bool fit2 = TcCfg<K, S, 2>::smem(a.TLB) <= kMaxSmem;
  if (!fit2) return DISCO_ERR_UNSUPPORTED;
  auto enc = encode_fn();
  if (!enc) return fail(DISCO_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  CUtensorMap map, nmap;
  cuuint64_t dims[3] = {(cuuint64_t)Win, (cuuint64_t)Hin, (cuuint64_t)BC};
  cuuint64_t strides[2] = {(cuuint64_t)Win * 2, (cuuint64_t)Hin * Win * 2};
  cuuint32_t estr[3] = {1, 1, 1};
  for (int m = 0; m < 2; ++m) {
    cuuint32_t box[3] = {m == 0 ? 64u : 8u, 1, 128};
    CUresult cr = enc(m == 0 ? &map : &nmap, dt16, 3, const_cast<void*>(x), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      m == 0 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return fail(DISCO_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)cr);
  }
  // X as the TMA store target: [B*C][K*H_out][W_out], box NT*16 columns x 1 row x 128 channels
  CUtensorMap omap;
  constexpr int NT3 = TcCfg<K, S, 3>::NT;
  a.tma_store = (a.Wout % 8 == 0 && a.Wout >= NT3 * kTW) ? 1 : 0;
  memset(&omap, 0, sizeof(omap));
  if (a.tma_store) {
    cuuint64_t od[3] = {(cuuint64_t)a.Wout, (cuuint64_t)K * a.Hout, (cuuint64_t)BC};
    cuuint64_t os[2] = {(cuuint64_t)a.Wout * 2, (cuuint64_t)K * a.Hout * a.Wout * 2};
    cuuint32_t ob[3] = {(cuuint32_t)(NT3 * kTW), 1, 128};
    CUresult cr = enc(&omap, dt16, 3, X, od, os, ob, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return fail(DISCO_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)cr);
  }
  if (a.tma_store && PCfg<K, S>::smem(a.TLB) <= kMaxSmem) {
    // persistent form: one CTA per SM over all tiles
    const size_t smem = PCfg<K, S>::smem(a.TLB);
    auto kern = fwd_tcp_kernel<K, S>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return check_launch("disco_fwd (tensor cores) attribute");
    const long long ntiles = (long long)((a.Wout + kTW * NT3 - 1) / (kTW * NT3)) * ((BC + 127) / 128) * a.Hout;
    const int grid = (int)(ntiles < sm_count_f() ? ntiles : sm_count_f());
    if (ntiles + grid > (long long)kSchedCountMask || grid > kSchedMaxCtas)
      return fail(DISCO_ERR_UNSUPPORTED, "problem too large");
    a.launch_id = next_launch_id();
    kern<<<grid, kPThreads, smem, st>>>(map, nmap, omap, a);
    return check_launch("disco_fwd (tensor cores)");
  }
  return fit3 ? launch_tc_stages<K, S, 3>(psi, map, nmap, omap, a, st)
              : launch_tc_stages<K, S, 2>(psi, map, nmap, omap, a, st);
}

template <int K, int S>
bool fits_tc(const disco_psi* psi) {
  const int TLB = (psi->grid_in.nlon + 16 + 7) & ~7;
  return TcCfg<K, S, 2>::smem(TLB) <= 227 * 1024;
}

}  // namespace

// Leaves in the scheduler word of launch `id` the tag of another launch with
// its counter part-way, as any earlier launch leaves it (diagnostic: launch
// `id` must take the word over and still compute every tile).
cudaError_t fwd_sched_plant(unsigned long long id) {
  const unsigned long long w = sched_tag(id + kSchedSlots) | 5ull;  // no active CTA
  return cudaMemcpyToSymbol(g_fwd_sched, &w, sizeof(w), (id % kSchedSlots) * sizeof(w));
}

// Reads (and optionally clears) this unit's status word; the caller has
// synchronised the device.
cudaError_t tc_status(int32_t* v, bool clear) {
  int32_t t = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&t, g_tc_status, sizeof(int32_t));
  if (e == cudaSuccess && clear) {
    const int32_t zero = 0;
    e = cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int32_t));
  }
  *v |= t;
  return e;
}

// True when fwd_tensor_core takes this psi and channel count.
bool fwd_tc_supported(const disco_psi* psi, int BC) {
  if (psi->grid_in.nlon % 8 != 0 || psi->grid_in.nlon < 64 || (psi->s != 1 && psi->s != 2) || BC < 1 ||
      BC > 65535 * 128 ||
      !psi->ftab || !psi->ftab_off || psi->K < 1 || psi->K > 9)
    return false;
#define DISCO_TFIT(KK) \
  if (psi->K == KK) return psi->s == 1 ? fits_tc<KK, 1>(psi) : fits_tc<KK, 2>(psi);
  DISCO_TFIT(1)
  DISCO_TFIT(2)
  DISCO_TFIT(3)
  DISCO_TFIT(4)
  DISCO_TFIT(5)
  DISCO_TFIT(6)
  DISCO_TFIT(7)
  DISCO_TFIT(8)
  DISCO_TFIT(9)
#undef DISCO_TFIT
  return false;
}

// Forward contraction on the tensor cores; returns DISCO_ERR_UNSUPPORTED
// (without launching) for shapes this path does not take.
int fwd_tensor_core(const disco_psi* psi, const void* x, void* X, int BC, cudaStream_t st, bool f16) {
  if (!fwd_tc_supported(psi, BC) || (f16 && !psi->ftab_h)) return DISCO_ERR_UNSUPPORTED;
  const int K = psi->K;
#define DISCO_TCASE(KK)                                                               \
  if (K == KK) return psi->s == 1 ? launch_tc<KK, 1>(psi, x, X, BC, st, f16)         \
                                  : launch_tc<KK, 2>(psi, x, X, BC, st, f16);
  DISCO_TCASE(1)
  DISCO_TCASE(2)
  DISCO_TCASE(3)
  DISCO_TCASE(4)
  DISCO_TCASE(5)
  DISCO_TCASE(6)
  DISCO_TCASE(7)
  DISCO_TCASE(8)
  DISCO_TCASE(9)
#undef DISCO_TCASE
  return DISCO_ERR_UNSUPPORTED;
}

// This unit's word of failed range checks (always 0 outside the bounds-checked build).
DISCO_BOUNDS_READER(tc_bounds)

}  // namespace disco
