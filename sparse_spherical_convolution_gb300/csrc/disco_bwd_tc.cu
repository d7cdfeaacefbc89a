// disco_bwd_tc.cu -- the transpose DISCO contraction on the tensor cores (bf16).
//
// DISCO Kernel Development Guide (torch-harmonics), §Architecture snapshot
// ("backward: CSR transpose contraction (B,C,K,H,W) -> inp") and §Backward
// direction (gather direction, each input pixel accumulates from its
// neighbourhood, no atomics; this kernel owns its output rows outright).
//
// Polyphase form: with input column j = S q + p and offset delta = S e + p,
//
//   gx[bc, hi, S q + p] = sum_{ho} sum_k sum_e psi_k^{(ho,hi)}(S e + p) G[bc, k, ho, q - e].
//
// For a tile of TQ decimated positions q = qb + t and a window of G columns
// w = qb - MW + i, this is, per (ho, k), an MMA
//
//   D[bc, (r, t, p)] += sum_i G[bc, k, ho, qb - MW + i] * T[(r, t, p), i],
//   T[(r, t, p), i] = psi_k^{(ho, hi0 + r)}(S (t - i + MW) + p),
//
// with M = 128 channels, N = 4 rows x S phases x TQ = 256 (ordered so that
// the N columns of row r are its output columns in order), and the window i
// as the K extent.  One CTA owns 4 consecutive input rows (they share most
// of their output-row neighbourhood, so every G window is loaded once for
// all four), 128 channels and 2 column tiles (TMEM: 2 x 256 columns).
// Per (ho, k, 64-column chunk) one pipeline stage holds
//   A  the G window, by TMA (8-column boxes of 128 channels, wrapped column),
//   tables  the 4 runs' bf16 polyphase tables of psi (bulk copies),
//   B  T built from the tables by 6 warps.
// Roles: warp 0 TMA/bulk producer and TMEM owner, warp 1 MMA issuer, warps
// 2-7 builders; all 8 warps run the epilogue.  All mbarrier waits are bounded.

#include <cudaTypedefs.h>

#include "disco_internal.cuh"
#include "disco_umma.cuh"

namespace disco {

__device__ int g_btc_status = 0;

namespace {

constexpr int kThreads = 256;
constexpr int kBuilderThreads = 192;
constexpr int kNR = 4;                      // input rows per CTA
constexpr int kNT = 2;                      // column tiles per CTA
constexpr int kN = 256;                     // MMA N = kNR * S * TQ
constexpr int kCK = 4;                      // K steps per chunk
constexpr int kChunkW = kCK * 16;           // 64 window columns
constexpr int kStages = 3;
constexpr uint32_t kGroupBytes = 128 * 16;  // one TMA box: 128 channels x 8 columns
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr int kStatusBtcTimeout = 8;

__device__ __forceinline__ void btc_flag(int bit) { atomicOr(&g_btc_status, bit); }

__device__ __forceinline__ int wrapc(int c, int W) {
  int r = c % W;
  return r < 0 ? r + W : r;
}
__device__ __forceinline__ int fdiv(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

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
  const disco_run* runs;
  const int32_t* trun_ptr;
  const int32_t* truns;
  const int32_t* btab_off;
  const uint16_t* btab;
  int BC, Hin, Win, Hout, Wout, K;
  int TLB;  // table row capacity (>= every run's row length, multiple of 8)
};

// per-run polyphase geometry
struct RunP {
  int EH;   // floor(dhi / S)
  int E;    // max |e| over the run
  int TL;   // table row length
};

template <int S>
__device__ __forceinline__ RunP run_p(const disco_run& r, int Win) {
  const int dlo = (r.len == Win) ? -(Win / 2) : -r.npair;
  const int dhi = dlo + r.len - 1;
  RunP g;
  g.EH = fdiv(dhi, S);
  const int EL = -fdiv(-(dlo - S + 1), S);  // ceil((dlo - S + 1) / S)
  g.E = max(g.EH, -EL);
  g.TL = (g.EH - EL + 1 + 16 + 7) & ~7;
  return g;
}

// run of (ho, hi) or -1, from hi's transposed list (ascending ho, contiguous)
__device__ __forceinline__ int find_run(const BtcArgs& a, int hi, int ho) {
  const int b = a.trun_ptr[hi], e = a.trun_ptr[hi + 1];
  if (b == e) return -1;
  const int first = a.runs[a.truns[b]].ho;
  const int pos = b + (ho - first);
  if (pos >= b && pos < e && a.runs[a.truns[pos]].ho == ho) return a.truns[pos];
  for (int i = b; i < e; ++i)
    if (a.runs[a.truns[i]].ho == ho) return a.truns[i];
  return -1;
}

template <int S>
struct BCfg {
  static constexpr int TQ = kN / (kNR * S);                         // decimated positions per tile
  static constexpr int AG = (TQ * (kNT - 1) + kChunkW) / 8;        // A groups per stage
  static constexpr uint32_t kABytes = AG * kGroupBytes;
  static constexpr uint32_t kBBytes = kN * kChunkW * 2;
  static constexpr uint32_t kSBOB = (kChunkW / 8) * 128;            // 1024
  __host__ __device__ static uint32_t tab_bytes(int TLB) { return (uint32_t)kNR * S * TLB * 2; }
  // stages start on 1 KB boundaries (TMA destinations need 128-byte alignment)
  __host__ __device__ static uint32_t stage_bytes(int TLB) {
    return (kABytes + kBBytes + tab_bytes(TLB) + 1023) & ~1023u;
  }
  __host__ __device__ static size_t smem(int TLB) { return (size_t)kStages * stage_bytes(TLB) + 256; }
};

// ho range of the CTA: union of the rows' neighbourhoods
__device__ __forceinline__ void ho_range(const BtcArgs& a, int hi0, int* lo, int* hi_) {
  int l = 1 << 30, h = -1;
  for (int r = 0; r < kNR; ++r) {
    const int hi = hi0 + r;
    if (hi >= a.Hin) break;
    const int b = a.trun_ptr[hi], e = a.trun_ptr[hi + 1];
    if (b == e) continue;
    l = min(l, a.runs[a.truns[b]].ho);
    h = max(h, a.runs[a.truns[e - 1]].ho);
  }
  *lo = l;
  *hi_ = h;
}

template <int S>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap gmap, const BtcArgs a) {
  using Cfg = BCfg<S>;
  constexpr int TQ = Cfg::TQ;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t stage_bytes = Cfg::stage_bytes(a.TLB);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * stage_bytes);
  uint64_t* fullA = bars;
  uint64_t* fullT = bars + kStages;
  uint64_t* fullB = bars + 2 * kStages;
  uint64_t* empty = bars + 3 * kStages;
  uint64_t* done = bars + 4 * kStages;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 4 * kStages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 4 * kStages + 2);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qb = blockIdx.x * (kNT * TQ);
  const int bc0 = blockIdx.y * 128;
  const int hi0 = blockIdx.z * kNR;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&fullA[s], 1);
      mbar_init(&fullT[s], 1);
      mbar_init(&fullB[s], kBuilderThreads);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
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

  int ho_lo, ho_hi;
  ho_range(a, hi0, &ho_lo, &ho_hi);

  // the per-ho window half-width MW and K steps KS, shared by all roles
  auto ho_geom = [&](int ho, int* rid, RunP* rp, int* MW, int* KS) {
    int E = 0;
    for (int r = 0; r < kNR; ++r) {
      rid[r] = (hi0 + r < a.Hin) ? find_run(a, hi0 + r, ho) : -1;
      if (rid[r] >= 0) {
        rp[r] = run_p<S>(a.runs[rid[r]], a.Win);
        E = max(E, rp[r].E);
      }
    }
    *MW = (E + 7) & ~7;
    *KS = (TQ + 2 * *MW + 15) >> 4;
  };

  if (warp == 0) {
    // ---------------------------------------------- TMA / bulk producer --
    if (lane == 0) {
      int i = 0;
      bool aborted = false;
      for (int ho = ho_lo; ho <= ho_hi && !aborted; ++ho) {
        int rid[kNR];
        RunP rp[kNR];
        int MW, KS;
        ho_geom(ho, rid, rp, &MW, &KS);
        for (int k = 0; k < a.K && !aborted; ++k)
          for (int c = 0; c * kCK < KS; ++c, ++i) {
            const int s = i % kStages;
            if ((i >= kStages && !mbar_wait(&empty[s], ((i / kStages) - 1) & 1, kWaitLimit)) ||
                *abort_flag) {
              btc_flag(kStatusBtcTimeout);
              *abort_flag = 1;
              aborted = true;
              break;
            }
            uint8_t* st = smem + (size_t)s * stage_bytes;
            uint8_t* tab = st + Cfg::kABytes + Cfg::kBBytes;
            uint32_t tbytes = 0;
            for (int r = 0; r < kNR; ++r)
              if (rid[r] >= 0) tbytes += S * rp[r].TL * 2;
            mbar_expect_tx(&fullT[s], tbytes);
            for (int r = 0; r < kNR; ++r)
              if (rid[r] >= 0)
                bulk_copy(tab + (size_t)r * S * a.TLB * 2,
                          a.btab + a.btab_off[rid[r]] + (size_t)k * S * rp[r].TL, S * rp[r].TL * 2,
                          &fullT[s]);
            const int nks = min(kCK, KS - c * kCK);
            const int ng = (TQ * (kNT - 1) + 16 * nks) / 8;
            mbar_expect_tx(&fullA[s], ng * kGroupBytes);
            const int w0 = qb - MW + c * kChunkW;
            for (int gi = 0; gi < ng; ++gi)
              tma_load_3d(st + gi * kGroupBytes, &gmap, wrapc(w0 + 8 * gi, a.Wout), k * a.Hout + ho,
                          bc0, &fullA[s]);
          }
      }
      if (aborted) {
        for (int back = 1; back <= kStages && i - back >= 0; ++back) {
          const int li = i - back;
          mbar_wait(&fullA[li % kStages], (li / kStages) & 1, kWaitLimit);
          mbar_wait(&fullT[li % kStages], (li / kStages) & 1, kWaitLimit);
        }
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, kN);
      int i = 0;
      bool ok = true;
      for (int ho = ho_lo; ho <= ho_hi && ok; ++ho) {
        int rid[kNR];
        RunP rp[kNR];
        int MW, KS;
        ho_geom(ho, rid, rp, &MW, &KS);
        for (int k = 0; k < a.K && ok; ++k)
          for (int c = 0; c * kCK < KS; ++c, ++i) {
            const int s = i % kStages;
            const uint32_t ph = (i / kStages) & 1;
            if (!mbar_wait(&fullA[s], ph, kWaitLimit) || !mbar_wait(&fullB[s], ph, kWaitLimit) ||
                *abort_flag) {
              btc_flag(kStatusBtcTimeout);
              *abort_flag = 1;
              ok = false;
              break;
            }
            tc_fence_after();
            const int nks = min(kCK, KS - c * kCK);
            const uint32_t abase = smem_u32(smem + (size_t)s * stage_bytes);
            const uint32_t bbase = abase + Cfg::kABytes;
            for (int j = 0; j < kNT; ++j)
              for (int ks = 0; ks < nks; ++ks) {
                const uint64_t ad = smem_desc(abase + (uint32_t)(j * TQ / 8 + 2 * ks) * kGroupBytes,
                                              kGroupBytes, 128);
                const uint64_t bd = smem_desc(bbase + ks * 256, 128, Cfg::kSBOB);
                umma_bf16(tmem + j * kN, ad, bd, idesc, (i > 0 || ks > 0) ? 1u : 0u);
              }
            umma_commit(&empty[s]);
          }
      }
      umma_commit(done);
    }
  } else {
    // ------------------------------------------------- B builders (6 warps) --
    const int btid = tid - 64;
    int i = 0;
    bool ok = true;
    for (int ho = ho_lo; ho <= ho_hi && ok; ++ho) {
      int rid[kNR];
      RunP rp[kNR];
      int MW, KS;
      ho_geom(ho, rid, rp, &MW, &KS);
      for (int k = 0; k < a.K && ok; ++k)
        for (int c = 0; c * kCK < KS; ++c, ++i) {
          const int s = i % kStages;
          const uint32_t ph = (i / kStages) & 1;
          bool mine = true;
          if (i >= kStages) mine = mbar_wait(&empty[s], ((i / kStages) - 1) & 1, kWaitLimit);
          mine = mine && mbar_wait(&fullT[s], ph, kWaitLimit) && !*abort_flag;
          if (!mine) {
            btc_flag(kStatusBtcTimeout);
            *abort_flag = 1;
          }
          ok = all_named(mine, 1, kBuilderThreads);
          if (!ok) break;
          uint8_t* st = smem + (size_t)s * stage_bytes;
          uint8_t* sB = st + Cfg::kABytes;
          const uint16_t* tab = reinterpret_cast<const uint16_t*>(st + Cfg::kABytes + Cfg::kBBytes);
          const int nks = min(kCK, KS - c * kCK);
          const int ngrp = 2 * nks;
          for (int idx = btid; idx < kN * ngrp; idx += kBuilderThreads) {
            const int n = idx % kN, gi = idx / kN;
            const int r = n / (S * TQ), rem = n - r * (S * TQ);
            const int t = rem / S, p = rem - t * S;
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            if (rid[r] >= 0) {
              // table index of window column c*64 + 8*gi + j is x0 + j
              const int TL = rp[r].TL;
              const int x0 = 8 + rp[r].EH - MW - t + c * kChunkW + 8 * gi;
              const uint16_t* row = tab + (size_t)r * S * a.TLB + (size_t)p * TL;
              if (x0 + 7 >= 0 && x0 < TL) {
                uint16_t v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const int x = x0 + j;
                  v[j] = (x >= 0 && x < TL) ? row[x] : (uint16_t)0;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) w[j] = (uint32_t)v[2 * j] | ((uint32_t)v[2 * j + 1] << 16);
              }
            }
            *reinterpret_cast<uint4*>(sB + (n >> 3) * Cfg::kSBOB + gi * 128 + (n & 7) * 16) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();
          mbar_arrive(&fullB[s]);
        }
    }
  }

  // ----------------------------------------------------- epilogue (8 warps) --
  {
    bool fin = mbar_wait(done, 0, kWaitLimit);
    fin = __all_sync(0xffffffffu, fin) && !*abort_flag;
    const bool any = ho_lo <= ho_hi;
    if (!fin) {
      if (lane == 0) btc_flag(kStatusBtcTimeout);
    } else {
      tc_fence_after();
      const int q = warp & 3, j = warp >> 2 ? 0 : 1;  // warps 4-7: tile 0, warps 0-3: tile 1
      const int bc = bc0 + q * 32 + lane;
      for (int r = 0; r < kNR; ++r) {
        const int hi = hi0 + r;
        for (int cc = 0; cc < (S * TQ) / 16; ++cc) {
          float v[16];
          if (any) {
            tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + j * kN + r * (S * TQ) + cc * 16, v);
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = 0.f;
          }
          const int col = S * (qb + j * TQ) + cc * 16;
          if (hi < a.Hin && bc < a.BC && col < a.Win) {
            __nv_bfloat16* dst = a.gx + ((size_t)bc * a.Hin + hi) * a.Win + col;
            const int n = min(16, a.Win - col);
            if (n == 16) {
              uint32_t w32[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                __nv_bfloat162 p2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                w32[e] = *reinterpret_cast<uint32_t*>(&p2);
              }
              reinterpret_cast<uint4*>(dst)[0] = make_uint4(w32[0], w32[1], w32[2], w32[3]);
              reinterpret_cast<uint4*>(dst)[1] = make_uint4(w32[4], w32[5], w32[6], w32[7]);
            } else {
              for (int e = 0; e < n; ++e) dst[e] = __float2bfloat16_rn(v[e]);
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

template <int S>
int launch_btc(const disco_psi* psi, const void* G, void* gx, int BC, cudaStream_t st) {
  using Cfg = BCfg<S>;
  BtcArgs a;
  a.gx = (__nv_bfloat16*)gx;
  a.runs = psi->runs;
  a.trun_ptr = psi->trun_ptr;
  a.truns = psi->truns;
  a.btab_off = psi->btab_off;
  a.btab = psi->btab;
  a.BC = BC;
  a.Hin = psi->grid_in.nlat;
  a.Win = psi->grid_in.nlon;
  a.Hout = psi->grid_out.nlat;
  a.Wout = psi->grid_out.nlon;
  a.K = psi->K;
  // a run spans at most one ring: EH - EL + 1 <= (W_in - 1 + S)/S + 1
  a.TLB = ((a.Win - 1 + S) / S + 1 + 1 + 16 + 7) & ~7;
  const size_t smem = Cfg::smem(a.TLB);
  if (smem > 227 * 1024) return DISCO_ERR_UNSUPPORTED;
  auto enc = encode_fn_b();
  if (!enc) return fail(DISCO_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  CUtensorMap map;
  cuuint64_t dims[3] = {(cuuint64_t)a.Wout, (cuuint64_t)a.K * a.Hout, (cuuint64_t)BC};
  cuuint64_t strides[2] = {(cuuint64_t)a.Wout * 2, (cuuint64_t)a.K * a.Hout * a.Wout * 2};
  cuuint32_t box[3] = {8, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult cr = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(G), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return fail(DISCO_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)cr);
  auto kern = bwd_tc_kernel<S>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return check_launch("disco_bwd (tensor cores) attribute");
  dim3 grid((a.Win + S * kNT * Cfg::TQ - 1) / (S * kNT * Cfg::TQ), (BC + 127) / 128,
            (a.Hin + kNR - 1) / kNR);
  kern<<<grid, kThreads, smem, st>>>(map, a);
  return check_launch("disco_bwd (tensor cores)");
}

}  // namespace

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

int bwd_tensor_core(const disco_psi* psi, const void* G, void* gx, int BC, cudaStream_t st) {
  if (psi->grid_out.nlon % 8 != 0 || psi->grid_in.nlon % 8 != 0 || (psi->s != 1 && psi->s != 2) ||
      BC > 65535 * 128 || psi->K > 16 || !psi->btab || !psi->btab_off)
    return DISCO_ERR_UNSUPPORTED;
  return psi->s == 1 ? launch_btc<1>(psi, G, gx, BC, st) : launch_btc<2>(psi, G, gx, BC, st);
}

}  // namespace disco
