// disco_fused.cu -- fused DISCO convolution and its input gradient on the
// sm_100-family tensor cores (tcgen05 MMA, fp32 accumulators in TMEM).
//
// DISCO Kernel Development Guide (torch-harmonics), §Architecture snapshot
// (the fused kernel: the contraction followed by the einsum).  The
// einsum y[b,o,ho,wo] = sum_{c,k} W[o,c,k] X[b,c,k,ho,wo] is a dense
// contraction over C*K, so it runs on the tensor cores; the contraction that
// produces X stays the CUDA-core gather of disco_fwd and X never reaches
// global memory.
//
// disco_fused_conv: one CTA per (batch, output row, 64 output columns).
//   warps 0-7  gather 16 input channels at a time (all K basis functions, 64
//              columns) into fp32 registers, round to bf16 and write the
//              chunk to shared memory as the MMA's B operand (K-major);
//   warp 8     streams the matching W chunk (A operand, K-major, all output
//              channels) into shared memory with cp.async and issues the
//              tcgen05.mma chain into TMEM (one 128-row M tile per 128 output
//              channels, N = 64 columns, K = 16 * K_basis per chunk).
//   The W load of chunk i+1 overlaps the gather of chunk i+1; the gather
//   warps only wait for the MMA of chunk i before overwriting its B tile.
//   Epilogue: tcgen05.ld of the accumulators, bf16 rounding, coalesced
//   row stores of y.
//
// disco_fused_conv_bwd_input: dX = W^T dy on the tensor cores (M = 128
//   pixels, N = 128 of the C*K rows, K = output channels in chunks of 64,
//   two-stage shared-memory pipeline), dX kept as bf16 in the caller's
//   workspace, then the transpose contraction gx = psi^T dX (disco_bwd).
//
// Every wait on an mbarrier is bounded; on time-out the kernel records a flag
// in a device status word (read by disco_device_status), stops issuing work,
// waits (bounded) for MMAs in flight and frees its TMEM before returning.

#include <mutex>

#include "disco_gather.cuh"
#include "disco_sched.cuh"
#include "disco_umma.cuh"

namespace disco {

__device__ int g_device_status = 0;

namespace {

constexpr uint32_t kWaitLimit = 1u << 24;  // polls before an mbarrier wait gives up
enum : int { kStatusFusedTimeout = 1, kStatusGemmTimeout = 2, kStatusWaitCheck = 16 };

__device__ __forceinline__ void flag_status(int bit) { atomicOr(&g_device_status, bit); }

// ------------------------------------------------------------ fused fwd --

constexpr int kFGatherThreads = 256;   // warps 0-7
constexpr int kFThreads = 288;         // + warp 8 (W loads, MMA issue, TMEM owner)
constexpr int kFNW = 64;               // output columns per CTA = MMA N
constexpr int kFTW = 4;                // output columns per gather thread
constexpr int kFCC = 16;               // input channels per chunk

struct FusedArgs {
  const __nv_bfloat16* x;
  const __nv_bfloat16* W;
  __nv_bfloat16* y;
  int B, Cin, Cout, Hin, Win, Hout, Wout, Kp, MT;
  const int32_t* run_ptr;
  const disco_run* runs;
  const float* hval;
  const int32_t* row_order;
  int nruns;        // runs and hval rows of psi (extent checks of the
  long long nhval;  // bounds-checked build)
};

template <int K, int S, bool ANISO>
struct FusedCfg {
  using G = RowGather<__nv_bfloat16, K, S, ANISO, kFCC, kFTW, kFNW, kFGatherThreads>;
  static constexpr int KD = kFCC * K;                // MMA K extent per chunk (multiple of 16)
  static constexpr uint32_t SBO = KD / 8 * 128;      // bytes per 8-row band of an operand
  static constexpr int kMTileBytes = 128 * KD * 2;   // one 128-row A tile
  static constexpr int kXBytes = kFNW * KD * 2;      // B tile
  static size_t smem_bytes(int MT) {
    return (size_t)MT * kMTileBytes + kXBytes + (size_t)G::kSmemFloats * 4 + 64;
  }
};

__host__ __device__ constexpr uint32_t tmem_cols_for(int ncols) {
  return ncols <= 32 ? 32 : ncols <= 64 ? 64 : ncols <= 128 ? 128 : ncols <= 256 ? 256 : 512;
}

template <int K, int S, bool ANISO>
__global__ void __launch_bounds__(kFThreads, 2) fused_fwd_kernel(const FusedArgs a) {
  using Cfg = FusedCfg<K, S, ANISO>;
  using G = typename Cfg::G;
  constexpr int KD = Cfg::KD;
  constexpr uint32_t SBO = Cfg::SBO;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sW = smem;
  uint8_t* sX = smem + (size_t)a.MT * Cfg::kMTileBytes;
  float* sG = reinterpret_cast<float*>(sX + Cfg::kXBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sG + G::kSmemFloats);
  uint64_t* bar_x = bars;      // gather -> MMA: B tile written (256 arrivals)
  uint64_t* bar_mma = bars + 1;  // MMA -> all: chunk's MMAs complete (commit)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 3);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z;
  int ho = a.row_order[blockIdx.y];
  if (!DISCO_IN_BOUNDS(ho >= 0 && ho < a.Hout)) ho = 0;
  const int wo_blk = blockIdx.x * kFNW;
  const int NC = a.Cin / kFCC;
  const uint32_t ncols = tmem_cols_for(a.MT * kFNW);

  // A-tile rows beyond Cout are never loaded: zero them once
  for (int i = tid; i < (a.MT * 128 - a.Cout) * (KD / 8); i += kFThreads) {
    const int o = a.Cout + i / (KD / 8), j = i % (KD / 8);
    *reinterpret_cast<uint4*>(sW + (size_t)(o >> 7) * Cfg::kMTileBytes +
                              kmajor_off(o & 127, 8 * j, SBO)) = make_uint4(0, 0, 0, 0);
  }
  if (tid == 0) {
    mbar_init(bar_x, kFGatherThreads);
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(tslot, ncols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 8) {
    // ---------------------------------------------- W loads + MMA issue --
    const size_t wrow = (size_t)a.Cin * K;
    auto load_w = [&](int ci) {
      const int pieces = a.Cout * (KD / 8);
      for (int i = lane; i < pieces; i += 32) {
        const int o = i / (KD / 8), j = i - o * (KD / 8);
        const __nv_bfloat16* src = a.W + (size_t)o * wrow + (size_t)ci * KD + 8 * j;
        cp_async16(sW + (size_t)(o >> 7) * Cfg::kMTileBytes + kmajor_off(o & 127, 8 * j, SBO), src);
      }
      cp_async_wait_all();
      fence_proxy_async_smem();
      __syncwarp();
    };
    constexpr uint32_t idesc = idesc_bf16_f32(128, kFNW);
    load_w(0);
    int pending = -1;  // chunk whose MMAs were issued but not yet seen complete
    for (int ci = 0; ci < NC; ++ci) {
      const bool got_x = __shfl_sync(0xffffffffu, mbar_wait(bar_x, ci & 1, kWaitLimit), 0);
      if (!got_x || *abort_flag) {
        if (lane == 0) flag_status(kStatusFusedTimeout);
        *abort_flag = 1;
        break;
      }
      if (lane == 0) {
        tc_fence_after();
        const uint32_t wbase = smem_u32(sW), xbase = smem_u32(sX);
        for (int mt = 0; mt < a.MT; ++mt)
#pragma unroll
          for (int ks = 0; ks < KD / 16; ++ks) {
            const uint64_t ad = smem_desc(wbase + mt * Cfg::kMTileBytes + ks * 256, 128, SBO);
            const uint64_t bd = smem_desc(xbase + ks * 256, 128, SBO);
            umma_bf16(tmem + mt * kFNW, ad, bd, idesc, (ci > 0 || ks > 0) ? 1u : 0u);
          }
        umma_commit(bar_mma);
      }
      __syncwarp();
      pending = ci;
      const bool done = __shfl_sync(0xffffffffu, mbar_wait(bar_mma, ci & 1, kWaitLimit), 0);
      if (!done) {
        if (lane == 0) flag_status(kStatusFusedTimeout);
        *abort_flag = 1;
        break;
      }
      pending = -1;
      if (ci + 1 < NC) load_w(ci + 1);
    }
    if (pending >= 0) {
      // give MMAs still in flight a bounded chance to finish before TMEM is freed
      mbar_wait(bar_mma, pending & 1, kWaitLimit);
    }
  } else {
    // ------------------------------------------------------- gather warps --
    const int ch = lane & 15, h = lane >> 4;
    constexpr int dg = 4 / S;  // half-warps 16 floats apart in the window: conflict-free
    const int g = (warp / dg) * 2 * dg + (warp % dg) + h * dg;
    const int o0 = g * kFTW;
    typename G::Args ga;
    ga.x = a.x;
    ga.BC = a.B * a.Cin;
    ga.Hin = a.Hin;
    ga.W = a.Win;
    ga.run_ptr = a.run_ptr;
    ga.runs = a.runs;
    ga.hval = a.hval;
    ga.Kp = a.Kp;
    ga.nruns = a.nruns;
    ga.nhval = a.nhval;
    bool ok = true;
    for (int ci = 0; ci < NC && ok; ++ci) {
      ga.bc0 = b * a.Cin + ci * kFCC;
      float acc[K][kFTW];
      G::run(acc, sG, ga, ho, wo_blk, ch, o0, tid, 1);
      bool mine = true;
      if (ci > 0) mine = mbar_wait(bar_mma, (ci - 1) & 1, kWaitLimit);
      mine = mine && !*abort_flag;
      ok = group_all(mine, 1, kFGatherThreads);  // uniform across the gather warps
      if (!ok) {
        if (tid == 0) flag_status(kStatusFusedTimeout);
        break;
      }
#pragma unroll
      for (int k = 0; k < K; ++k)
#pragma unroll
        for (int t = 0; t < kFTW; ++t)
          *reinterpret_cast<__nv_bfloat16*>(sX + kmajor_off(o0 + t, ch * K + k, SBO)) =
              __float2bfloat16_rn(acc[k][t]);
      fence_proxy_async_smem();
      mbar_arrive(bar_x);
    }
    bool fin = ok && mbar_wait(bar_mma, (NC - 1) & 1, kWaitLimit) && !*abort_flag;
    fin = group_all(fin, 1, kFGatherThreads);
    if (!fin && ok && tid == 0) flag_status(kStatusFusedTimeout);
    if (fin) {
      tc_fence_after();
      const int q = warp & 3, mt = warp >> 2;
      if (mt < a.MT) {
        const int o = mt * 128 + q * 32 + lane;
        const int wo0 = wo_blk;
#pragma unroll
        for (int j = 0; j < kFNW / 16; ++j) {
          float v[16];
          tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + mt * kFNW + j * 16, v);
          if (o < a.Cout) {
            __nv_bfloat16* dst = a.y + (((size_t)b * a.Cout + o) * a.Hout + ho) * a.Wout + wo0 + j * 16;
            const int n = min(16, a.Wout - (wo0 + j * 16));
            if (n == 16 && (a.Wout % 8) == 0) {
              uint4 u[2];
              uint32_t* w32 = reinterpret_cast<uint32_t*>(u);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                __nv_bfloat162 p2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                w32[i] = *reinterpret_cast<uint32_t*>(&p2);
              }
              reinterpret_cast<uint4*>(dst)[0] = u[0];
              reinterpret_cast<uint4*>(dst)[1] = u[1];
            } else {
              for (int i = 0; i < n; ++i) dst[i] = __float2bfloat16_rn(v[i]);
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    // every MMA this CTA issued was seen complete, or given a bounded drain wait
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

template <int K, int S, bool ANISO>
int launch_fused(const FusedArgs& a, cudaStream_t st) {
  auto kern = fused_fwd_kernel<K, S, ANISO>;
  const size_t smem = FusedCfg<K, S, ANISO>::smem_bytes(a.MT);
  if (smem > 227 * 1024) return fail(DISCO_ERR_UNSUPPORTED, "fused tile needs %zu bytes of shared memory", smem);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return check_launch("disco_fused_conv attribute");
  dim3 grid((a.Wout + kFNW - 1) / kFNW, a.Hout, a.B);
  kern<<<grid, kFThreads, smem, st>>>(a);
  return check_launch("disco_fused_conv");
}

template <int S>
int dispatch_fused(int kind, int K, const FusedArgs& a, cudaStream_t st) {
#define DISCO_FCASE(KK, AN) \
  if (K == KK && (kind == 1) == AN) return launch_fused<KK, S, AN>(a, st);
  DISCO_FCASE(1, false)
  DISCO_FCASE(2, false)
  DISCO_FCASE(3, false)
  DISCO_FCASE(4, false)
  DISCO_FCASE(5, false)
  DISCO_FCASE(6, false)
  DISCO_FCASE(7, false)
  DISCO_FCASE(8, false)
  DISCO_FCASE(3, true)
  DISCO_FCASE(6, true)
  DISCO_FCASE(9, true)
#undef DISCO_FCASE
  return fail(DISCO_ERR_UNSUPPORTED, "K = %d (kind %d) has no fused kernel", K, kind);
}

// --------------------------------------------------------- dX = W^T dy --
//
// D[p, n] = sum_o dy[b, o, p] * W[o, n]   (p = pixel, n = c*K + k)
// A = dy^T tile [128 pixels x 64 o], B = W^T tile [128 n x 64 o], both
// transposed into K-major shared-memory tiles by the loading threads.

constexpr int kGThreads = 256;
constexpr int kGM = 128;   // pixels per CTA
constexpr int kGN = 128;   // C*K rows per CTA
constexpr int kGK = 64;    // output channels per pipeline stage
constexpr uint32_t kGSBO = kGK / 8 * 128;       // 1024
constexpr int kGTileA = kGM * kGK * 2;          // 16 KB
constexpr int kGTileB = kGN * kGK * 2;          // 16 KB
constexpr int kGStage = kGTileA + kGTileB;
constexpr size_t kGSmem = 2 * (size_t)kGStage + 64;

struct GemmArgs {
  const __nv_bfloat16* dy;  // [B][Cout][P]
  const __nv_bfloat16* W;   // [Cout][CK]
  __nv_bfloat16* dX;        // [B][CK][P]
  int Cout, CK;
  int64_t P;
};

__global__ void __launch_bounds__(kGThreads, 2) dx_gemm_kernel(const GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kGStage);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // C*K tiles vary fastest so consecutive CTAs reuse one dy tile from L2
  const int64_t p0 = (int64_t)blockIdx.y * kGM;
  const int n0 = blockIdx.x * kGN;
  const int b = blockIdx.z;
  const int nk = (a.Cout + kGK - 1) / kGK;
  const __nv_bfloat16* dyb = a.dy + (size_t)b * a.Cout * a.P;

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, kGN);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  bool ok = true;

  for (int kc = 0; kc < nk; ++kc) {
    const int s = kc & 1;
    uint8_t* sA = smem + s * kGStage;
    uint8_t* sB = sA + kGTileA;
    if (kc >= 2) {  // stage s was read by the MMAs of chunk kc-2
      if (!mbar_wait(&bars[s], ((kc - 2) >> 1) & 1, kWaitLimit)) {
        if (tid == 0) flag_status(kStatusGemmTimeout);
        ok = false;
      }
    }
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }
    const int o_base = kc * kGK;
    // A: (row p, k o) <- dy[o][p].  A thread gathers 8 consecutive o of one
    // pixel (lanes on consecutive pixels: coalesced 2-byte loads) and writes
    // them as one 16-byte core-matrix row.
    for (int i = tid; i < kGM * (kGK / 8); i += kGThreads) {
      const int pl = i % kGM, og = i / kGM;
      const int64_t p = p0 + pl;
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const int o = o_base + og * 8 + e;
        __nv_bfloat16 v0 = __float2bfloat16_rn(0.f), v1 = v0;
        if (p < a.P) {
          if (o < a.Cout) v0 = dyb[(size_t)o * a.P + p];
          if (o + 1 < a.Cout) v1 = dyb[(size_t)(o + 1) * a.P + p];
        }
        __nv_bfloat162 p2;
        p2.x = v0;
        p2.y = v1;
        w[e >> 1] = *reinterpret_cast<uint32_t*>(&p2);
      }
      *reinterpret_cast<uint4*>(sA + kmajor_off(pl, og * 8, kGSBO)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    // B: (row n, k o) <- W[o][n], same scheme along n
    for (int i = tid; i < kGN * (kGK / 8); i += kGThreads) {
      const int nl = i % kGN, og = i / kGN;
      const int n = n0 + nl;
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const int o = o_base + og * 8 + e;
        __nv_bfloat16 v0 = __float2bfloat16_rn(0.f), v1 = v0;
        if (n < a.CK) {
          if (o < a.Cout) v0 = a.W[(size_t)o * a.CK + n];
          if (o + 1 < a.Cout) v1 = a.W[(size_t)(o + 1) * a.CK + n];
        }
        __nv_bfloat162 p2;
        p2.x = v0;
        p2.y = v1;
        w[e >> 1] = *reinterpret_cast<uint32_t*>(&p2);
      }
      *reinterpret_cast<uint4*>(sB + kmajor_off(nl, og * 8, kGSBO)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_bf16_f32(kGM, kGN);
#pragma unroll
      for (int ks = 0; ks < kGK / 16; ++ks) {
        const uint64_t ad = smem_desc(smem_u32(sA) + ks * 256, 128, kGSBO);
        const uint64_t bd = smem_desc(smem_u32(sB) + ks * 256, 128, kGSBO);
        umma_bf16(tmem, ad, bd, idesc, (kc > 0 || ks > 0) ? 1u : 0u);
      }
      umma_commit(&bars[s]);
    }
  }
  // wait for the last chunk's MMAs (its commit covers all earlier ones)
  {
    const int last = nk - 1;
    bool done = mbar_wait(&bars[last & 1], (last >> 1) & 1, kWaitLimit);
    done = __syncthreads_and(done) != 0;
    if (!done && tid == 0) flag_status(kStatusGemmTimeout);
    ok = ok && done;
  }
  tc_fence_after();
  if (ok && warp < 4) {
    const int64_t p = p0 + warp * 32 + lane;
#pragma unroll 1
    for (int j = 0; j < kGN / 16; ++j) {
      float v[16];
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + j * 16, v);
      if (p < a.P) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int n = n0 + j * 16 + i;
          if (n < a.CK) a.dX[((size_t)b * a.CK + n) * a.P + p] = __float2bfloat16_rn(v[i]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kGN);
  }
}

// ------------------------------------------------------ y = W X (einsum) --
//
// D[p, o] = sum_ck X[b, ck, p] * W[o, ck]   (p = pixel ho*W_out + wo, ck = c*K + k)
// M = 128 pixels, N = Cout (<= 256, one tile), K = Cin*K in chunks of 64,
// two-stage pipeline.  A = X^T tile: each thread gathers 8 consecutive ck of
// one pixel (lanes on consecutive pixels) into one 16-byte core-matrix row;
// B = W tile: 16-byte rows of W[o][ck] as they are (already K-major).
// Epilogue: lane = pixel, so each column store of y is coalesced.

constexpr int kEN = 256;                        // max Cout per tile
constexpr int kETileB = kEN * kGK * 2;          // 32 KB
constexpr int kEStage = kGTileA + kETileB;
constexpr size_t kESmem = 2 * (size_t)kEStage + 64;

struct EinArgs {
  const __nv_bfloat16* X;   // [B][CK][P]
  const __nv_bfloat16* W;   // [Cout][CK]
  __nv_bfloat16* y;         // [B][Cout][P]
  int Cout, CK, Npad;       // Npad: Cout rounded up to 16
  int64_t P;
};

__global__ void __launch_bounds__(kGThreads, 2) einsum_gemm_kernel(const EinArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kEStage);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t p0 = (int64_t)blockIdx.x * kGM;
  const int b = blockIdx.y;
  const int nk = (a.CK + kGK - 1) / kGK;
  const __nv_bfloat16* Xb = a.X + (size_t)b * a.CK * a.P;

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, kEN);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  bool ok = true;
  const bool vec_w = (a.CK % 8) == 0;

  for (int kc = 0; kc < nk; ++kc) {
    const int s = kc & 1;
    uint8_t* sA = smem + s * kEStage;
    uint8_t* sB = sA + kGTileA;
    if (kc >= 2) {
      if (!mbar_wait(&bars[s], ((kc - 2) >> 1) & 1, kWaitLimit)) {
        if (tid == 0) flag_status(kStatusGemmTimeout);
        ok = false;
      }
    }
    if (!__syncthreads_and(ok)) {
      ok = false;
      break;
    }
    const int c_base = kc * kGK;
    // A: (row p, k ck) <- X[ck][p]
    for (int i = tid; i < kGM * (kGK / 8); i += kGThreads) {
      const int pl = i % kGM, cg = i / kGM;
      const int64_t p = p0 + pl;
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const int ck = c_base + cg * 8 + e;
        __nv_bfloat16 v0 = __float2bfloat16_rn(0.f), v1 = v0;
        if (p < a.P) {
          if (ck < a.CK) v0 = Xb[(size_t)ck * a.P + p];
          if (ck + 1 < a.CK) v1 = Xb[(size_t)(ck + 1) * a.P + p];
        }
        __nv_bfloat162 p2;
        p2.x = v0;
        p2.y = v1;
        w[e >> 1] = *reinterpret_cast<uint32_t*>(&p2);
      }
      *reinterpret_cast<uint4*>(sA + kmajor_off(pl, cg * 8, kGSBO)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    // B: (row o, k ck) <- W[o][ck], 16-byte pieces
    for (int i = tid; i < a.Npad * (kGK / 8); i += kGThreads) {
      const int o = i / (kGK / 8), cg = i % (kGK / 8);
      const int ck = c_base + cg * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (o < a.Cout) {
        if (vec_w && ck + 8 <= a.CK) {
          v = *reinterpret_cast<const uint4*>(a.W + (size_t)o * a.CK + ck);
        } else {
          __align__(16) __nv_bfloat16 t[8];
          for (int e = 0; e < 8; ++e)
            t[e] = (ck + e < a.CK) ? a.W[(size_t)o * a.CK + ck + e] : __float2bfloat16_rn(0.f);
          v = *reinterpret_cast<uint4*>(t);
        }
      }
      *reinterpret_cast<uint4*>(sB + kmajor_off(o, cg * 8, kGSBO)) = v;
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(kGM, a.Npad);
#pragma unroll
      for (int ks = 0; ks < kGK / 16; ++ks) {
        const uint64_t ad = smem_desc(smem_u32(sA) + ks * 256, 128, kGSBO);
        const uint64_t bd = smem_desc(smem_u32(sB) + ks * 256, 128, kGSBO);
        umma_bf16(tmem, ad, bd, idesc, (kc > 0 || ks > 0) ? 1u : 0u);
      }
      umma_commit(&bars[s]);
    }
  }
  {
    const int last = nk - 1;
    bool done = mbar_wait(&bars[last & 1], (last >> 1) & 1, kWaitLimit);
    done = __syncthreads_and(done) != 0;
    if (!done && tid == 0) flag_status(kStatusGemmTimeout);
    ok = ok && done;
  }
  tc_fence_after();
  if (ok) {
    // 8 warps: lane quarter = warp % 4, column half = warp / 4
    const int q = warp & 3, half = warp >> 2;
    const int64_t p = p0 + q * 32 + lane;
    const int ncols = a.Npad / 2;
#pragma unroll 1
    for (int j = 0; j < ncols / 16; ++j) {
      float v[16];
      const int c0 = half * ncols + j * 16;
      tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
      if (p < a.P) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int o = c0 + i;
          if (o < a.Cout) a.y[((size_t)b * a.Cout + o) * a.P + p] = __float2bfloat16_rn(v[i]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kEN);
  }
}

int check_fused_common(const disco_psi* psi, const void* a, const void* W, const void* out,
                       int32_t B, int32_t Cin, int32_t Cout, disco_dtype dtype) {
  int st = check_psi(psi);
  if (st) return st;
  if ((st = check_device())) return st;
  if (!a || !W || !out) return fail(DISCO_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(a) || !aligned16(W) || !aligned16(out))
    return fail(DISCO_ERR_ALIGNMENT, "tensors must be 16-byte aligned");
  if ((st = check_dev_ptr(a, "input")) || (st = check_dev_ptr(W, "W")) || (st = check_dev_ptr(out, "output")))
    return st;
  if (dtype != DISCO_BF16 && dtype != DISCO_F16) return fail(DISCO_ERR_UNSUPPORTED, "fused paths take bf16 or fp16");
  if (B < 1 || Cin < 1 || Cout < 1) return fail(DISCO_ERR_INVALID_ARG, "B, Cin, Cout must be >= 1");
  if (B > 65535) return fail(DISCO_ERR_UNSUPPORTED, "B > 65535");
  if (psi->s != 1 && psi->s != 2)
    return fail(DISCO_ERR_UNSUPPORTED, "W_in / W_out = %d (1 and 2 supported)", psi->s);
  return DISCO_OK;
}

}  // namespace
}  // namespace disco

using namespace disco;

// Tensor-core path of disco_fused_conv: X = contraction into the workspace
// (bf16), then the einsum on the tensor cores.
static int fused_tc(const disco_psi* psi, const void* x, const void* W, void* y, int32_t B, int32_t Cin,
                    int32_t Cout, void* X, cudaStream_t s, bool f16) {
  const int64_t P = (int64_t)psi->grid_out.nlat * psi->grid_out.nlon;
  if (f16 && !gemm_tc_supported(P, Cin * psi->K, Cout))
    return fail(DISCO_ERR_UNSUPPORTED, "fp16 fused conv: needs the tensor-core einsum shape "
                "(H_out*W_out, Cin*K, Cout multiples of 8, Cin*K >= 64, Cout >= 16)");
  int st = fwd_tensor_core(psi, x, X, B * Cin, s, f16);
  if (st) return st;
  st = einsum_tensor_core(X, W, y, B, Cin * psi->K, Cout, P, s, f16);
  if (st != DISCO_ERR_UNSUPPORTED) return st;
  EinArgs e;
  e.X = (const __nv_bfloat16*)X;
  e.W = (const __nv_bfloat16*)W;
  e.y = (__nv_bfloat16*)y;
  e.Cout = Cout;
  e.CK = Cin * psi->K;
  e.Npad = (Cout + 31) / 32 * 32;  // the epilogue splits N into two halves of 16-column steps
  e.P = (int64_t)psi->grid_out.nlat * psi->grid_out.nlon;
  if (cudaFuncSetAttribute(einsum_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kESmem) !=
      cudaSuccess)
    return check_launch("einsum attribute");
  dim3 grid((unsigned)((e.P + kGM - 1) / kGM), B);
  if (grid.x > 0x7fffffffu || B > 65535) return fail(DISCO_ERR_UNSUPPORTED, "problem too large");
  einsum_gemm_kernel<<<grid, kGThreads, kESmem, s>>>(e);
  return check_launch("einsum");
}

extern "C" size_t disco_fused_conv_workspace_bytes(const disco_psi* psi, int32_t B, int32_t Cin, int32_t Cout,
                                                   disco_dtype dtype) {
  if (!psi || B < 1 || Cin < 1 || Cout < 1 || (dtype != DISCO_BF16 && dtype != DISCO_F16) ||
      !fwd_tc_supported(psi, B * Cin))
    return 0;
  return (size_t)B * Cin * psi->K * psi->grid_out.nlat * psi->grid_out.nlon * 2;
}

extern "C" int disco_fused_conv(const disco_psi* psi, const void* x, const void* W, void* y,
                                int32_t B, int32_t Cin, int32_t Cout, disco_dtype dtype,
                                void* workspace, size_t workspace_bytes, void* stream) {
  disco::NvtxScope nvtx_scope("disco_fused_conv");
  int st = check_fused_common(psi, x, W, y, B, Cin, Cout, dtype);
  if (st) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t need = disco_fused_conv_workspace_bytes(psi, B, Cin, Cout, dtype);
  if (need > 0) {
    if (!workspace || workspace_bytes < need)
      return fail(DISCO_ERR_WORKSPACE, "workspace needs %zu bytes", need);
    if (!aligned16(workspace)) return fail(DISCO_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
    if ((st = check_dev_ptr(workspace, "workspace"))) return st;
    return fused_tc(psi, x, W, y, B, Cin, Cout, workspace, s, dtype == DISCO_F16);
  }
  if (dtype == DISCO_F16)
    return fail(DISCO_ERR_UNSUPPORTED, "fp16 fused conv: needs the tensor-core forward shape (W_in % 8 == 0, "
                "W_in >= 64, K <= 9)");
  // shapes the tensor-core contraction does not take: X built on chip by the
  // CUDA-core gather, einsum on the tensor cores
  if (Cout > 256) return fail(DISCO_ERR_UNSUPPORTED, "Cout must be <= 256 on the CUDA-core gather path");
  if (Cin % kFCC != 0) return fail(DISCO_ERR_UNSUPPORTED, "Cin must be a multiple of %d", kFCC);
  FusedArgs a;
  a.x = (const __nv_bfloat16*)x;
  a.W = (const __nv_bfloat16*)W;
  a.y = (__nv_bfloat16*)y;
  a.B = B;
  a.Cin = Cin;
  a.Cout = Cout;
  a.Hin = psi->grid_in.nlat;
  a.Win = psi->grid_in.nlon;
  a.Hout = psi->grid_out.nlat;
  a.Wout = psi->grid_out.nlon;
  a.Kp = psi->K_pad;
  a.MT = (Cout + 127) / 128;
  a.run_ptr = psi->run_ptr;
  a.runs = psi->runs;
  a.hval = psi->hval;
  a.row_order = psi->row_order;
  a.nruns = (int)psi->nruns;
  a.nhval = psi->nhval;
  return psi->s == 1 ? dispatch_fused<1>(psi->basis.kind, psi->K, a, s)
                     : dispatch_fused<2>(psi->basis.kind, psi->K, a, s);
}

extern "C" size_t disco_fused_conv_bwd_input_workspace_bytes(const disco_psi* psi, int32_t B,
                                                             int32_t Cin, disco_dtype dtype) {
  if (!psi || B < 1 || Cin < 1 || (dtype != DISCO_BF16 && dtype != DISCO_F16)) return 0;
  return (size_t)B * Cin * psi->K * psi->grid_out.nlat * psi->grid_out.nlon * 2;
}

// The input gradient with dX in `workspace`; the caller has checked the
// arguments and the workspace (a caller buffer or the library's own scratch).
static int fused_bwd_input(const disco_psi* psi, const void* dy, const void* W, void* gx, int32_t B,
                           int32_t Cin, int32_t Cout, disco_dtype dtype, void* workspace, void* stream);

extern "C" int disco_fused_conv_bwd_input(const disco_psi* psi, const void* dy, const void* W,
                                          void* gx, int32_t B, int32_t Cin, int32_t Cout,
                                          disco_dtype dtype, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  disco::NvtxScope nvtx_scope("disco_fused_conv_bwd_input");
  int st = check_fused_common(psi, dy, W, gx, B, Cin, Cout, dtype);
  if (st) return st;
  size_t need = disco_fused_conv_bwd_input_workspace_bytes(psi, B, Cin, dtype);
  if (!workspace || workspace_bytes < need)
    return fail(DISCO_ERR_WORKSPACE, "workspace needs %zu bytes", need);
  if (!aligned16(workspace)) return fail(DISCO_ERR_ALIGNMENT, "workspace must be 16-byte aligned");
  if ((st = check_dev_ptr(workspace, "workspace"))) return st;
  return fused_bwd_input(psi, dy, W, gx, B, Cin, Cout, dtype, workspace, stream);
}

static int fused_bwd_input(const disco_psi* psi, const void* dy, const void* W, void* gx, int32_t B,
                           int32_t Cin, int32_t Cout, disco_dtype dtype, void* workspace, void* stream) {
  int st = DISCO_OK;
  GemmArgs g;
  g.dy = (const __nv_bfloat16*)dy;
  g.W = (const __nv_bfloat16*)W;
  g.dX = (__nv_bfloat16*)workspace;
  g.Cout = Cout;
  g.CK = Cin * psi->K;
  g.P = (int64_t)psi->grid_out.nlat * psi->grid_out.nlon;
  cudaStream_t s = (cudaStream_t)stream;
  const bool f16 = dtype == DISCO_F16;
  if (dx_tensor_core_supported(Cout, g.CK, g.P) && bwd_tc_supported(psi, B * Cin)) {
    // both on the tensor cores: dX goes through the workspace as
    // [K*H_out][B*Cin][W_out], whose 128-channel boxes the transpose streams
    // much faster than boxes of the [B*Cin][K][H_out][W_out] layout
    const int roc[4] = {psi->K, psi->grid_out.nlat, psi->grid_out.nlon, Cin};
    st = dx_tensor_core(dy, W, workspace, B, Cout, g.CK, g.P, s, roc, f16);
    if (st) return st;
    return bwd_tensor_core(psi, workspace, gx, B * Cin, s, true, f16);
  }
  if (f16)
    return fail(DISCO_ERR_UNSUPPORTED, "fp16 fused input gradient: needs the tensor-core shapes (dX GEMM: "
                "H_out*W_out, Cout multiples of 8, Cout >= 64, Cin*K multiple of 64; transpose: W_out % 8 == 0, "
                "W_out >= 64, s <= 2)");
  st = dx_tensor_core(dy, W, workspace, B, Cout, g.CK, g.P, s);
  if (st == DISCO_ERR_UNSUPPORTED) {
    if (cudaFuncSetAttribute(dx_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kGSmem) != cudaSuccess)
      return check_launch("dX gemm attribute");
    dim3 grid((g.CK + kGN - 1) / kGN, (unsigned)((g.P + kGM - 1) / kGM), B);
    if (grid.y > 65535) return fail(DISCO_ERR_UNSUPPORTED, "H_out * W_out too large");
    dx_gemm_kernel<<<grid, kGThreads, kGSmem, s>>>(g);
    st = check_launch("dX gemm");
  }
  if (st) return st;
  return contract(false, psi, workspace, gx, B, Cin, dtype, stream, false);
}

static size_t align256z(size_t v) { return (v + 255) & ~(size_t)255; }

extern "C" size_t disco_fused_conv_bwd_weight_workspace_bytes(const disco_psi* psi, int32_t B, int32_t Cin,
                                                              int32_t Cout, disco_dtype dtype) {
  if (!psi || B < 1 || Cin < 1 || Cout < 1 || (dtype != DISCO_BF16 && dtype != DISCO_F16) ||
      !fwd_tc_supported(psi, B * Cin))
    return 0;
  const int64_t P = (int64_t)psi->grid_out.nlat * psi->grid_out.nlon;
  const int CK = Cin * psi->K;
  if (!dw_tensor_core_supported(B, Cout, CK, P)) return 0;
  return align256z((size_t)B * CK * P * 2) + dw_partial_bytes(B, Cout, CK, P);
}

extern "C" int disco_fused_conv_bwd_weight(const disco_psi* psi, const void* x, const void* dy, void* dW,
                                           int32_t B, int32_t Cin, int32_t Cout, disco_dtype dtype,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  disco::NvtxScope nvtx_scope("disco_fused_conv_bwd_weight");
  int st = check_fused_common(psi, x, dy, dW, B, Cin, Cout, dtype);
  if (st) return st;
  const size_t need = disco_fused_conv_bwd_weight_workspace_bytes(psi, B, Cin, Cout, dtype);
  if (need == 0)
    return fail(DISCO_ERR_UNSUPPORTED,
                "weight gradient: needs the tensor-core forward shape (bf16 or fp16, W_in % 8 == 0, W_in >= 64, "
                "K <= 9) with H_out*W_out, Cin*K and Cout multiples of 8, Cin*K >= 64, Cout >= 16");
  if (!workspace || workspace_bytes < need) return fail(DISCO_ERR_WORKSPACE, "workspace needs %zu bytes", need);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(DISCO_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if ((st = check_dev_ptr(workspace, "workspace"))) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const int64_t P = (int64_t)psi->grid_out.nlat * psi->grid_out.nlon;
  const int CK = Cin * psi->K;
  // X = the forward contraction (bf16) in the first part of the workspace
  const bool f16 = dtype == DISCO_F16;
  if ((st = fwd_tensor_core(psi, x, workspace, B * Cin, s, f16))) return st;
  void* part = (char*)workspace + align256z((size_t)B * CK * P * 2);
  return dw_tensor_core(dy, workspace, dW, part, B, Cout, CK, P, s, f16);
}

// One thread waits, with the bounded wait of the tensor-core kernels, on the
// first phase of an mbarrier that nothing arrives on; when the wait runs out
// it records that in the status word and returns.
__global__ void wait_check_kernel(uint32_t limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (!mbar_wait(&bar, 0, limit)) flag_status(kStatusWaitCheck);
}

extern "C" int disco_check_wait_timeout(uint32_t limit, void* stream) {
  int st = check_device();
  if (st) return st;
  if (limit < 1 || limit > (1u << 24)) return fail(DISCO_ERR_INVALID_ARG, "limit must be in [1, 2^24]");
  wait_check_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(limit);
  return check_launch("wait check");
}

extern "C" int disco_device_status(int32_t* flags, int32_t clear) {
  if (!flags) return fail(DISCO_ERR_INVALID_ARG, "flags is null");
  int st = check_device();
  if (st) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(flags, g_device_status, sizeof(int32_t));
  if (e == cudaSuccess && clear) {
    const int32_t zero = 0;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int32_t));
  }
  if (e == cudaSuccess) e = tc_status(flags, clear != 0);
  if (e == cudaSuccess) e = btc_status(flags, clear != 0);
  if (e == cudaSuccess) e = gemm_status(flags, clear != 0);
  int32_t bounds = 0;
  for (auto fn : {contract_bounds, psi_bounds, tc_bounds, btc_bounds, gemm_bounds, fused_bounds})
    if (e == cudaSuccess) e = fn(&bounds, clear != 0);
  *flags |= bounds;
  if (e != cudaSuccess) return fail(DISCO_ERR_CUDA, "device status: %s", cudaGetErrorString(e));
  if (bounds & kStatusBounds)
    return fail(DISCO_ERR_DEVICE_BOUNDS, "a range check of the bounds-checked build failed (access skipped)");
  return DISCO_OK;
}

extern "C" int32_t disco_build_flags(void) {
#ifdef DISCO_DEBUG_BOUNDS
  return DISCO_BUILD_DEBUG_BOUNDS;
#else
  return 0;
#endif
}

namespace disco {
namespace {

// One thread walks the scheduler protocol (disco_sched.cuh) on a private word,
// playing the CTAs of two launches; ids are multiples of kSchedSlots so the
// word is entry 0 of the one-entry table.
__device__ unsigned long long g_sched_walk[1];
__device__ int g_sched_walk_out[9];

__global__ void sched_walk_kernel() {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  constexpr unsigned long long L1 = 1 * kSchedSlots, L2 = 2 * kSchedSlots;
  unsigned long long* const t = g_sched_walk;
  t[0] = sched_tag(4 * kSchedSlots) | 7ull;  // left by an earlier launch, no active CTA
  int* o = g_sched_walk_out;
  unsigned long long* a = sched_join(t, L1, 4);       // launch 1 takes the word
  o[0] = a != nullptr;                                // 1
  o[1] = a ? sched_next(a) : -1;                      // 0
  o[2] = a ? sched_next(a) : -1;                      // 1
  unsigned long long* b = sched_join(t, L1, 4);       // a sibling joins
  o[3] = b ? sched_next(b) : -1;                      // 2
  o[4] = sched_join(t, L2, 4) == nullptr;             // launch 2 waits while launch 1 draws: 1
  if (a) sched_leave(a);
  if (b) sched_leave(b);
  unsigned long long* c = sched_join(t, L2, 4);       // launch 1 gone: launch 2 takes the word
  o[5] = c ? sched_next(c) : -1;                      // 0
  o[6] = sched_join(t, L1, 4) == nullptr;             // a late CTA of launch 1 waits: 1
  if (c) sched_leave(c);
  unsigned long long* d = sched_join(t, L1, 4);       // ... and takes the word back once free
  o[7] = d ? sched_next(d) : -1;                      // 0
  if (d) sched_leave(d);
  o[8] = t[0] == (sched_tag(L1) | 1ull);              // no active CTA left: 1
}

}  // namespace
}  // namespace disco

extern "C" int disco_check_sched_takeover(void) {
  int st = check_device();
  if (st) return st;
  sched_walk_kernel<<<1, 32>>>();
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  int got[9];
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(got, g_sched_walk_out, sizeof(got));
  if (e != cudaSuccess) return fail(DISCO_ERR_CUDA, "scheduler walk: %s", cudaGetErrorString(e));
  const int want[9] = {1, 0, 1, 2, 1, 0, 1, 0, 1};
  for (int k = 0; k < 9; ++k)
    if (got[k] != want[k])
      return fail(DISCO_ERR_CUDA, "scheduler walk: step %d drew %d, expected %d", k, got[k], want[k]);
  const unsigned long long id = peek_launch_id();
  e = fwd_sched_plant(id);
  if (e == cudaSuccess) e = btc_sched_plant(id);
  if (e != cudaSuccess) return fail(DISCO_ERR_CUDA, "scheduler word: %s", cudaGetErrorString(e));
  return DISCO_OK;
}

// ------------------------------------------------ allocation-free variant --
//
// disco_fused_conv_bwd_input_noalloc: the same computation as
// disco_fused_conv_bwd_input, for callers that cannot allocate device memory
// themselves (for example a host runtime whose allocator owns all device
// memory from start-up, or a hot loop that must not risk the implicit device
// synchronisation cudaMalloc can cause).  Its dX scratch is the fixed array
// below, which the CUDA runtime creates on every device that loads this
// library and keeps until the process exits.  Host code cannot use the
// array's name as a device address, so the address is looked up once per
// device with cudaGetSymbolAddress (on the first call on that device, with
// that device current) and cached.

namespace disco {
namespace {

constexpr size_t kNoAllocScratchBytes = DISCO_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
// per device: the context the address was looked up in, and the address
struct NoAllocAddr {
  void* ctx = nullptr;
  void* ptr = nullptr;
};
NoAllocAddr g_noalloc[kMaxDevices];

int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DISCO_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(DISCO_ERR_UNSUPPORTED, "device index %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocAddr& c = g_noalloc[dev];
  void* ctx = current_context();
  // the cached address holds only for the context it was taken in: after a
  // device reset the array lives at a new address of a new context
  if (!c.ptr || !ctx || ctx != c.ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return fail(DISCO_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    c.ptr = p;
    c.ctx = current_context();  // the lookup made the device's context current
  }
  *out = c.ptr;
  return DISCO_OK;
}

}  // namespace
// This unit's word of failed range checks (always 0 outside the bounds-checked build).
DISCO_BOUNDS_READER(fused_bounds)

}  // namespace disco

extern "C" int disco_fused_conv_bwd_input_noalloc(const disco_psi* psi, const void* dy, const void* W,
                                                  void* gx, int32_t B, int32_t Cin, int32_t Cout,
                                                  disco_dtype dtype, void* stream) {
  disco::NvtxScope nvtx_scope("disco_fused_conv_bwd_input_noalloc");
  int st = check_fused_common(psi, dy, W, gx, B, Cin, Cout, dtype);
  if (st) return st;
  const size_t need = disco_fused_conv_bwd_input_workspace_bytes(psi, B, Cin, dtype);
  if (need > kNoAllocScratchBytes)
    return fail(DISCO_ERR_WORKSPACE,
                "disco_fused_conv_bwd_input_noalloc: this problem needs %zu bytes of scratch, "
                "the fixed scratch holds %zu (use disco_fused_conv_bwd_input with a workspace)",
                need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch))) return st;
  // dX is fully rewritten by the GEMM before the transpose reads it, so
  // nothing left in the scratch by an earlier call needs clearing.
  return fused_bwd_input(psi, dy, W, gx, B, Cin, Cout, dtype, scratch, stream);
}
