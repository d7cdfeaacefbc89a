// disco_gemm_tc.cu -- the dense contractions of the fused paths on the tensor
// cores: the channel/basis einsum of the fused convolution and the dX GEMM of
// its input gradient.
//
// DISCO Kernel Development Guide (torch-harmonics), §Architecture snapshot
// (the fused kernel: the contraction followed by an einsum): after the S2
// contraction, y[b,o,ho,wo] = sum_{c,k} W[o,c,k] X[b,c,k,ho,wo].  Both GEMMs
// here have the form
//
//   out[b, n, p] = sum_j A[b, j, p] * Bop(j, n)        (p = pixel ho*W_out + wo)
//
//   einsum: A = X  [B][C*K][P],   Bop(j, n) = W[n][j]   (n = o,  j = c*K + k)
//   dX:     A = dy [B][Cout][P],  Bop(j, n) = W[j][n]   (n = c*K + k, j = o)
//
// as one tcgen05 GEMM per tile of 128 pixels x N (<= 256) outputs: M = 128
// pixels, accumulators in TMEM.  A is read by TMA straight from its natural
// layout as "MN-major" tiles (pixels contiguous; two 64-pixel boxes of 64
// j-rows per stage, 128-byte swizzle); Bop is K-major (einsum: W rows) or
// MN-major (dX: W rows are j), also by TMA.  Persistent kernel, 4-stage
// load ring, two TMEM accumulators so the epilogue of one tile overlaps the
// main loop of the next:
//   warp 0  TMA producer (one thread),
//   warp 1  MMA issuer (one thread, TMEM owner),
//   warps 2-9 epilogue: tcgen05.ld, bf16, stores coalesced along pixels
//            (two warps per TMEM lane quadrant, alternate 16-output steps).
// The dW kernel below keeps four epilogue warps (warps 2-5).
// All mbarrier waits are bounded (time-out -> status flag, abort).

#include <cudaTypedefs.h>

#include "disco_bounds.cuh"
#include "disco_internal.cuh"
#include "disco_umma.cuh"

namespace disco {

__device__ int g_gemm_status = 0;

namespace {

constexpr int kThreads = 224;           // dw_gemm_kernel: producer, MMA, 4 epilogue warps, second producer
constexpr int kEpiThreads = 128;
constexpr int kDProducers = 2;          // dw_gemm_kernel: warp 0 (items i % 2 == 0) and warp 6 (i % 2 == 1)
// gemm_tc_kernel: producer, MMA and 8 epilogue warps, two per TMEM lane
// quadrant, taking alternate 16-output steps (its epilogue, not the MMA,
// bounds the dX GEMM, whose tiles have a short reduction)
constexpr int kGEpiWarps = 8;
constexpr int kGThreads = 64 + 32 * kGEpiWarps;
constexpr int kGEpiThreads = 32 * kGEpiWarps;
constexpr int kBM = 128;                  // pixels per tile
constexpr int kBK = 64;                   // j per stage
constexpr int kStages = 4;
constexpr uint32_t kABytes = kBM * kBK * 2;   // 16 KB: two 64-pixel boxes
constexpr uint32_t kBMax = 256 * kBK * 2;     // 32 KB: up to 256 outputs
constexpr uint32_t kStageBytes = kABytes + kBMax;
constexpr uint32_t kEpiStage = 16 * 32 * 2;      // per epilogue warp: 16 outputs x 32 pixels bf16
constexpr size_t kSmem = (size_t)kStages * kStageBytes + kGEpiWarps * kEpiStage + 256 + 1024;
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr int kStatusGemmTimeout = 2;

__device__ __forceinline__ void gemm_flag() { atomicOr(&g_gemm_status, kStatusGemmTimeout); }

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
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

// 128-byte swizzled operand tile descriptor with explicit LBO / SBO (bytes)
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;
  d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// kind::f16 instruction descriptor, bf16 A and B, fp32 D; A MN-major, B as given
__host__ __device__ constexpr uint32_t idesc_mn(int M, int N, bool b_mn, bool half) {
  return idesc_16_f32(M, N, half) | (1u << 15) | ((b_mn ? 1u : 0u) << 16);
}

struct GemmTcArgs {
  __nv_bfloat16* out;  // [B][Nt][P], or the row-of-channels form below when ctK > 0
  // Row-of-channels output (dX of the input gradient, n = c*K + k, p = ho*W + wo):
  //   out[(k*ctH + ho)][b*ctC + c][wo]
  // so that a TMA box of 128 channels x 64 columns of one row (k, ho) reads
  // rows W*2 bytes apart instead of a channel slab apart.
  int ctK, ctH, ctW, ctC;
  int f16;             // operands and out are fp16 (else bf16)
  uint32_t bbytes;     // bytes of the B boxes of one stage
  int64_t P;           // pixels
  int Kt;              // reduction length j
  int Nt;              // outputs n
  int NB;              // outputs per tile (multiple of 16, <= 256)
  int mt, nt, B;       // tiles along pixels, along n, batch
};

template <bool kBMN>
__global__ void __launch_bounds__(kGThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                   const GemmTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint16_t* epi_stage = reinterpret_cast<uint16_t*>(smem + kStages * kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes + kGEpiWarps * kEpiStage);
  uint64_t* full = bars;                   // [kStages]
  uint64_t* empty = bars + kStages;        // [kStages]
  uint64_t* accf = bars + 2 * kStages;     // [2] accumulator complete (commit)
  uint64_t* acce = bars + 2 * kStages + 2; // [2] accumulator drained (128 arrivals)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kStages + 5);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = a.mt * a.nt * a.B;
  const int nk = (a.Kt + kBK - 1) / kBK;
  const uint32_t bbytes = a.bbytes;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], kGEpiThreads);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  // tile t: n tiles fastest (consecutive CTAs share the A tile in L2), then pixels, then batch
  auto coords = [&](int t, int* p0, int* n0, int* b) {
    *n0 = (t % a.nt) * a.NB;
    const int r = t / a.nt;
    *p0 = (r % a.mt) * kBM;
    *b = r / a.mt;
  };

  if (warp == 0) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      int i = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        int p0, n0, b;
        coords(t, &p0, &n0, &b);
        for (int kc = 0; kc < nk; ++kc, ++i) {
          const int s = i % kStages;
          if ((i >= kStages && !mbar_wait(&empty[s], ((i / kStages) - 1) & 1, kWaitLimit)) || *abort_flag) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * kStageBytes;
          uint8_t* sb = sa + kABytes;
          mbar_expect_tx(&full[s], kABytes + bbytes);
          // the tile's origin lies inside the operands (boxes past the ends of a
          // ragged tail are read as zeros by the copy engine, by design)
          if (!DISCO_IN_BOUNDS(p0 >= 0 && p0 < a.P && kc * kBK < a.Kt && b >= 0 && b < a.B && n0 >= 0 &&
                               n0 < a.Nt)) {
            mbar_complete_tx(&full[s], kABytes + bbytes);
            continue;
          }
          tma_load_3d(sa, &amap, p0, kc * kBK, b, &full[s]);
          tma_load_3d(sa + kABytes / 2, &amap, p0 + 64, kc * kBK, b, &full[s]);
          if (kBMN) {
            for (int q = 0; q < a.NB / 64; ++q)  // W rows j, 64 outputs per box
              tma_load_2d(sb + q * (64 * kBK * 2), &bmap, n0 + 64 * q, kc * kBK, &full[s]);
          } else {
            tma_load_2d(sb, &bmap, kc * kBK, n0, &full[s]);  // NB W rows of 64 j
          }
        }
      }
      if (!ok) {
        gemm_flag();
        *abort_flag = 1;
        for (int back = 1; back <= kStages && i - back >= 0; ++back) {
          const int li = i - back;
          mbar_wait(&full[li % kStages], (li / kStages) & 1, kWaitLimit);
        }
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      const uint32_t idesc = idesc_mn(kBM, a.NB, kBMN, a.f16 != 0);
      int i = 0, tl = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++tl) {
        const int ab = tl & 1;  // accumulator buffer
        if (tl >= 2 && !mbar_wait(&acce[ab], ((tl >> 1) - 1) & 1, kWaitLimit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + ab * 256;
        for (int kc = 0; kc < nk; ++kc, ++i) {
          const int s = i % kStages;
          if (!mbar_wait(&full[s], (i / kStages) & 1, kWaitLimit) || *abort_flag) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks) {
            // A: 16 j-rows = two 8-row groups (SBO 1024) further; second pixel half at LBO 8 KB
            const uint64_t ad = desc_sw128(sa + ks * 2048, kABytes / 2, 1024);
            const uint64_t bd = kBMN ? desc_sw128(sb + ks * 2048, 64 * kBK * 2, 1024)
                                     : desc_sw128(sb + ks * 32, 16, 1024);
            umma_bf16(d, ad, bd, idesc, (kc > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&accf[ab]);
      }
      if (!ok) {
        gemm_flag();
        *abort_flag = 1;
        if (i > 0) mbar_wait(&empty[(i - 1) % kStages], ((i - 1) / kStages) & 1, kWaitLimit);
      }
    }
  } else {
    // ------------------------------------------------- epilogue (warps 2-9) --
    const int q = warp & 3;             // TMEM lanes 32q .. 32q+31
    const int half = (warp - 2) >> 2;   // output steps c0 = 16 half + 32 j
    int tl = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tl) {
      const int ab = tl & 1;
      bool fin = mbar_wait(&accf[ab], (tl >> 1) & 1, kWaitLimit);
      fin = __all_sync(0xffffffffu, fin) && !*abort_flag;
      if (!fin) {
        if (lane == 0) gemm_flag();
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      int p0, n0, b;
      coords(t, &p0, &n0, &b);
      // 16 outputs x 32 pixels at a time through shared memory, so that each
      // lane then stores 16 consecutive bytes (8 pixels) of one output row
      const int64_t pw = p0 + q * 32;  // this warp's first pixel
      uint16_t* stg = epi_stage + (warp - 2) * (kEpiStage / 2);
      __nv_bfloat16* ob = a.out + (size_t)b * a.Nt * a.P;
      // row-of-channels form: this lane's pixel segment (row ho, column wo) is
      // fixed for the tile; its two outputs per step, n = n0 + c0 + lane/4 + 8h,
      // advance by 16 per step, so (c, k) = divmod(n, K) is carried along
      const int64_t BC = (int64_t)a.B * a.ctC;
      int64_t rho = 0, rwo = 0;
      int rc[2] = {0, 0}, rk[2] = {0, 0}, dc = 0, dk = 0;
      if (a.ctK > 0) {
        const int64_t pp = pw + (lane & 3) * 8;
        rho = pp / a.ctW;
        rwo = pp - rho * a.ctW;
        dc = 32 / a.ctK;
        dk = 32 - dc * a.ctK;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int n = n0 + 16 * half + (lane >> 2) + 8 * h;
          rc[h] = n / a.ctK;
          rk[h] = n - rc[h] * a.ctK;
        }
      }
      for (int c0 = 16 * half; c0 < a.NB; c0 += 32) {
        float v[16];
        tmem_ld16(tmem + ab * 256 + ((uint32_t)(q * 32) << 16) + c0, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) stg[e * 32 + lane] = round_16(v[e], a.f16);
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int idx = lane + 32 * h, row = idx >> 2, seg = idx & 3;
          const int n = n0 + c0 + row;
          const int64_t pp = pw + seg * 8;  // P % 8 == 0: a segment is all in or all out
          if (n < a.Nt && pp < a.P) {
            __nv_bfloat16* dst;
            bool inside;
            if (a.ctK > 0) {  // W % 8 == 0: the 8 pixels lie in one row
              dst = a.out + (((int64_t)rk[h] * a.ctH + rho) * BC + (int64_t)b * a.ctC + rc[h]) * a.ctW + rwo;
              inside = DISCO_IN_BOUNDS(rk[h] >= 0 && rk[h] < a.ctK && rho >= 0 && rho < a.ctH && rc[h] >= 0 &&
                                       rc[h] < a.ctC && b < a.B && rwo >= 0 && rwo + 8 <= a.ctW);
            } else {
              dst = ob + (size_t)n * a.P + pp;
              inside = DISCO_IN_BOUNDS(b >= 0 && b < a.B && pp >= 0 && pp + 8 <= a.P);
            }
            if (inside) *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(stg + row * 32 + seg * 8);
          }
        }
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // next step: n += 32
          rc[h] += dc;
          rk[h] += dk;
          if (rk[h] >= a.ctK) {
            rk[h] -= a.ctK;
            ++rc[h];
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acce[ab]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------- dW = sum_p dy X^T --
//
// Weight gradient of the fused convolution, y = einsum(W, X):
//   dW[o, n] = sum_b sum_p dy[b, o, p] X[b, n, p]          (n = c*K + k)
// Both operands are K-major with the pixels as the reduction (dy rows o, X
// rows n, pixels contiguous), one TMA box each per 64 pixels.  Tiles of 128 o
// x NB n; the reduction over (b, pixel chunks) is split across CTAs
// (deterministic: each split writes fp32 partial sums, a second kernel adds
// them in split order and rounds to bf16).

struct DwArgs {
  float* part;         // [nsplit][mt*128][nt*NB] fp32 partial sums
  uint32_t abytes, bbytes;  // bytes of one A / B box (rows clipped to the tensor)
  int64_t P;
  int Cout, Nt, NB;    // rows o, columns n, columns per tile
  int mt, nt, nsplit;  // tiles along o, along n, reduction splits
  int nkp, B;          // 64-pixel chunks per image, images
  int f16;             // dy and X are fp16 (else bf16)
};

__global__ void __launch_bounds__(kThreads, 1)
    dw_gemm_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                   const DwArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes + 4 * kEpiStage);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* accf = bars + 2 * kStages;
  uint64_t* acce = bars + 2 * kStages + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kStages + 5);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = a.mt * a.nt * a.nsplit;
  const int nq = a.nkp * a.B;  // (image, pixel chunk) reduction steps

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], kEpiThreads);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  // tile t: split fastest, then n, then o; split sp reduces steps [q0, q1)
  auto coords = [&](int t, int* o0, int* n0, int* sp, int* q0, int* q1) {
    *sp = t % a.nsplit;
    const int r = t / a.nsplit;
    *n0 = (r % a.nt) * a.NB;
    *o0 = (r / a.nt) * kBM;
    *q0 = (int)((long long)nq * *sp / a.nsplit);
    *q1 = (int)((long long)nq * (*sp + 1) / a.nsplit);
  };

  if (warp == 0 || warp == 6) {
    // producers: item i (one reduction step of a tile) by warp 0 when i is
    // even, by warp 6 when odd; with kStages a multiple of kDProducers a
    // stage always serves the same producer, which waits only on its own
    // earlier items (boxes of dy and X rows P apart are issued faster by
    // two threads than by one)
    static_assert(kStages % kDProducers == 0, "a stage stays with one producer");
    const int who = warp == 0 ? 0 : 1;
    if (lane == 0) {
      int i = 0, done = 0;  // done: one past the last item this thread issued
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        int o0, n0, sp, q0, q1;
        coords(t, &o0, &n0, &sp, &q0, &q1);
        for (int q = q0; q < q1; ++q, ++i) {
          if (i % kDProducers != who) continue;
          const int s = i % kStages;
          if ((i >= kStages && !mbar_wait(&empty[s], ((i / kStages) - 1) & 1, kWaitLimit)) || *abort_flag) {
            ok = false;
            break;
          }
          const int b = q / a.nkp, p0 = (q - b * a.nkp) * kBK;
          uint8_t* sa = smem + s * kStageBytes;
          // rows of a box past the tensor (o >= Cout, n >= Nt) keep stale values:
          // they only reach accumulator rows / columns that are never reduced
          mbar_expect_tx(&full[s], a.abytes + a.bbytes);
          if (DISCO_IN_BOUNDS(p0 >= 0 && p0 < a.P && o0 >= 0 && o0 < a.Cout && n0 >= 0 && n0 < a.Nt && b >= 0 &&
                              b < a.B)) {
            tma_load_3d(sa, &amap, p0, o0, b, &full[s]);
            tma_load_3d(sa + kABytes, &bmap, p0, n0, b, &full[s]);
          } else {
            mbar_complete_tx(&full[s], a.abytes + a.bbytes);
          }
          done = i + 1;
        }
      }
      if (!ok) {
        gemm_flag();
        *abort_flag = 1;
        for (int li = done - 1; li >= 0 && li >= done - kDProducers * kStages; --li)
          if (li % kDProducers == who) mbar_wait(&full[li % kStages], (li / kStages) & 1, kWaitLimit);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_16_f32(kBM, a.NB, a.f16 != 0);
      int i = 0, tl = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++tl) {
        int o0, n0, sp, q0, q1;
        coords(t, &o0, &n0, &sp, &q0, &q1);
        const int ab = tl & 1;
        if (tl >= 2 && !mbar_wait(&acce[ab], ((tl >> 1) - 1) & 1, kWaitLimit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + ab * 256;
        for (int q = q0; q < q1; ++q, ++i) {
          const int s = i % kStages;
          if (!mbar_wait(&full[s], (i / kStages) & 1, kWaitLimit) || *abort_flag) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks)
            umma_bf16(d, desc_sw128(sa + ks * 32, 16, 1024), desc_sw128(sb + ks * 32, 16, 1024), idesc,
                      (q > q0 || ks > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&accf[ab]);
      }
      if (!ok) {
        gemm_flag();
        *abort_flag = 1;
        if (i > 0) mbar_wait(&empty[(i - 1) % kStages], ((i - 1) / kStages) & 1, kWaitLimit);
      }
    }
  } else {
    const int q4 = warp & 3;
    int tl = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++tl) {
      const int ab = tl & 1;
      bool fin = mbar_wait(&accf[ab], (tl >> 1) & 1, kWaitLimit);
      fin = __all_sync(0xffffffffu, fin) && !*abort_flag;
      if (!fin) {
        if (lane == 0) gemm_flag();
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      int o0, n0, sp, q0, q1;
      coords(t, &o0, &n0, &sp, &q0, &q1);
      const bool empty_split = q1 <= q0;  // no reduction steps: the partial is zero
      const int row = o0 + q4 * 32 + lane;
      float* dst = a.part + ((size_t)sp * a.mt * kBM + row) * ((size_t)a.nt * a.NB) + n0;
      const bool inside = DISCO_IN_BOUNDS(sp >= 0 && sp < a.nsplit && row >= 0 && row < a.mt * kBM && n0 >= 0 &&
                                          n0 + a.NB <= a.nt * a.NB);
      for (int c0 = 0; c0 < a.NB && inside; c0 += 16) {
        float v[16];
        if (!empty_split) {
          tmem_ld16(tmem + ab * 256 + ((uint32_t)(q4 * 32) << 16) + c0, v);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0.f;
        }
#pragma unroll
        for (int g = 0; g < 4; ++g)
          reinterpret_cast<float4*>(dst + c0)[g] = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
      }
      tc_fence_before();
      mbar_arrive(&acce[ab]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// dW[o][n] = bf16 or fp16 (sum over splits, in split order, of the partials)
__global__ void dw_reduce_kernel(const float* part, uint16_t* dW, int Cout, int Nt, int rows, int cols,
                                 int nsplit, int f16) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)Cout * Nt) return;
  const int o = (int)(i / Nt), n = (int)(i - (int64_t)o * Nt);
  float acc = 0.f;
  if (!DISCO_IN_BOUNDS(o < rows && n < cols)) return;
  for (int sp = 0; sp < nsplit; ++sp) acc += part[((size_t)sp * rows + o) * cols + n];
  dW[i] = round_16(acc, f16);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_g() {
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

int encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
           const cuuint32_t* box, bool f16) {
  auto enc = encode_fn_g();
  if (!enc) return fail(DISCO_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult cr = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
                    const_cast<void*>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return fail(DISCO_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)cr);
  return DISCO_OK;
}

int sm_count_g() {
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

// out[b][n][p] = sum_j A[b][j][p] * Bop(j, n); W is [Nt][Kt] (kBMN false) or [Kt][Nt] (true)
template <bool kBMN>
int launch_gemm(const void* A, const void* W, void* out, int B, int Kt, int Nt, int64_t P, cudaStream_t st,
                const int* ct, bool f16) {
  GemmTcArgs g;
  g.f16 = f16 ? 1 : 0;
  g.out = (__nv_bfloat16*)out;
  g.ctK = ct ? ct[0] : 0;
  g.ctH = ct ? ct[1] : 0;
  g.ctW = ct ? ct[2] : 0;
  g.ctC = ct ? ct[3] : 0;
  g.P = P;
  g.Kt = Kt;
  g.Nt = Nt;
  // outputs per tile: at most 256 (one TMEM accumulator); more outputs take
  // more tiles along n
  g.NB = kBMN ? (Nt >= 256 ? 256 : (Nt + 63) / 64 * 64) : (Nt >= 256 ? 256 : (Nt + 15) / 16 * 16);
  g.mt = (int)((P + kBM - 1) / kBM);
  g.nt = (Nt + g.NB - 1) / g.NB;
  g.B = B;
  // K-major B rows past Nt are not loaded (stale smem feeds only unstored columns)
  g.bbytes = kBMN ? (uint32_t)g.NB * kBK * 2 : (uint32_t)(Nt < g.NB ? Nt : g.NB) * kBK * 2;
  CUtensorMap amap, bmap;
  {
    cuuint64_t dims[3] = {(cuuint64_t)P, (cuuint64_t)Kt, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)P * 2, (cuuint64_t)Kt * P * 2};
    cuuint32_t box[3] = {64, kBK, 1};
    int s = encode(&amap, A, 3, dims, strides, box, f16);
    if (s) return s;
  }
  {
    cuuint64_t dims[2] = {kBMN ? (cuuint64_t)Nt : (cuuint64_t)Kt, kBMN ? (cuuint64_t)Kt : (cuuint64_t)Nt};
    cuuint64_t strides[1] = {(kBMN ? (cuuint64_t)Nt : (cuuint64_t)Kt) * 2};
    cuuint32_t box[2] = {64, kBMN ? (cuuint32_t)kBK : (cuuint32_t)(Nt < g.NB ? Nt : g.NB)};
    int s = encode(&bmap, W, 2, dims, strides, box, f16);
    if (s) return s;
  }
  auto kern = gemm_tc_kernel<kBMN>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) != cudaSuccess)
    return check_launch("tensor-core GEMM attribute");
  const long long ntiles = (long long)g.mt * g.nt * B;
  if (ntiles > 0x7fffffffLL) return fail(DISCO_ERR_UNSUPPORTED, "problem too large");
  const int grid = (int)(ntiles < sm_count_g() ? ntiles : sm_count_g());
  kern<<<grid, kGThreads, kSmem, st>>>(amap, bmap, g);
  return check_launch("tensor-core GEMM");
}

}  // namespace

bool gemm_tc_supported(int64_t P, int Kt, int Nt) {
  return P % 8 == 0 && P >= 128 && Kt % 8 == 0 && Kt >= kBK && Nt % 8 == 0 && Nt >= 16;
}

int einsum_tensor_core(const void* X, const void* W, void* y, int B, int CK, int Cout, int64_t P, cudaStream_t st,
                       bool f16) {
  if (!gemm_tc_supported(P, CK, Cout)) return DISCO_ERR_UNSUPPORTED;
  return launch_gemm<false>(X, W, y, B, CK, Cout, P, st, nullptr, f16);
}

bool dx_tensor_core_supported(int Cout, int CK, int64_t P) { return gemm_tc_supported(P, Cout, CK) && CK % 64 == 0; }

int dx_tensor_core(const void* dy, const void* W, void* dX, int B, int Cout, int CK, int64_t P, cudaStream_t st,
                   const int* rows_of_channels, bool f16) {
  if (!dx_tensor_core_supported(Cout, CK, P)) return DISCO_ERR_UNSUPPORTED;
  if (rows_of_channels) {
    const int K = rows_of_channels[0], H = rows_of_channels[1], W_ = rows_of_channels[2], C = rows_of_channels[3];
    if (K < 1 || C < 1 || W_ % 8 != 0 || (int64_t)K * C != CK || (int64_t)H * W_ != P) return DISCO_ERR_UNSUPPORTED;
  }
  return launch_gemm<true>(dy, W, dX, B, Cout, CK, P, st, rows_of_channels, f16);
}

namespace {
struct DwPlan {
  int mt, nt, NB, nsplit, nkp;
};
DwPlan dw_plan(int B, int Cout, int CK, int64_t P) {
  DwPlan d;
  d.NB = CK >= 256 ? 256 : (CK + 15) / 16 * 16;
  d.mt = (Cout + kBM - 1) / kBM;
  d.nt = (CK + d.NB - 1) / d.NB;
  d.nkp = (int)((P + kBK - 1) / kBK);
  const long long steps = (long long)d.nkp * B;
  long long ns = (2LL * sm_count_g() + (long long)d.mt * d.nt - 1) / ((long long)d.mt * d.nt);
  if (ns > steps) ns = steps;
  if (ns < 1) ns = 1;
  d.nsplit = (int)ns;
  return d;
}
}  // namespace

bool dw_tensor_core_supported(int B, int Cout, int CK, int64_t P) {
  return B >= 1 && gemm_tc_supported(P, CK, Cout) && Cout >= 16 && CK >= 16;
}

size_t dw_partial_bytes(int B, int Cout, int CK, int64_t P) {
  const DwPlan d = dw_plan(B, Cout, CK, P);
  return (size_t)d.nsplit * d.mt * kBM * ((size_t)d.nt * d.NB) * 4;
}

int dw_tensor_core(const void* dy, const void* X, void* dW, void* partials, int B, int Cout, int CK, int64_t P,
                   cudaStream_t st, bool f16) {
  if (!dw_tensor_core_supported(B, Cout, CK, P)) return DISCO_ERR_UNSUPPORTED;
  const DwPlan d = dw_plan(B, Cout, CK, P);
  DwArgs g;
  g.part = (float*)partials;
  g.P = P;
  g.Cout = Cout;
  g.Nt = CK;
  g.NB = d.NB;
  g.mt = d.mt;
  g.nt = d.nt;
  g.nsplit = d.nsplit;
  g.nkp = d.nkp;
  g.B = B;
  g.f16 = f16 ? 1 : 0;
  const int arows = Cout < kBM ? Cout : kBM, brows = CK < d.NB ? CK : d.NB;
  g.abytes = (uint32_t)arows * kBK * 2;
  g.bbytes = (uint32_t)brows * kBK * 2;
  CUtensorMap amap, bmap;
  {
    cuuint64_t dims[3] = {(cuuint64_t)P, (cuuint64_t)Cout, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)P * 2, (cuuint64_t)Cout * P * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)arows, 1};
    int s = encode(&amap, dy, 3, dims, strides, box, f16);
    if (s) return s;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)P, (cuuint64_t)CK, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)P * 2, (cuuint64_t)CK * P * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)brows, 1};
    int s = encode(&bmap, X, 3, dims, strides, box, f16);
    if (s) return s;
  }
  if (cudaFuncSetAttribute(dw_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) !=
      cudaSuccess)
    return check_launch("dW GEMM attribute");
  const long long ntiles = (long long)d.mt * d.nt * d.nsplit;
  const int grid = (int)(ntiles < sm_count_g() ? ntiles : sm_count_g());
  dw_gemm_kernel<<<grid, kThreads, kSmem, st>>>(amap, bmap, g);
  int s = check_launch("dW GEMM");
  if (s) return s;
  const long long n = (long long)Cout * CK;
  dw_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(
      (const float*)partials, (uint16_t*)dW, Cout, CK, d.mt * kBM, d.nt * d.NB, d.nsplit, f16 ? 1 : 0);
  return check_launch("dW reduce");
}

cudaError_t gemm_status(int32_t* v, bool clear) {
  int32_t t = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&t, g_gemm_status, sizeof(int32_t));
  if (e == cudaSuccess && clear) {
    const int32_t zero = 0;
    e = cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof(int32_t));
  }
  *v |= t;
  return e;
}

// This unit's word of failed range checks (always 0 outside the bounds-checked build).
DISCO_BOUNDS_READER(gemm_bounds)

}  // namespace disco
