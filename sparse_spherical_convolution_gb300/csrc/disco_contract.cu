// disco_contract.cu -- forward and transpose DISCO contractions on CUDA cores.
//
// DISCO Kernel Development Guide (torch-harmonics):
//  * §Architecture snapshot: forward = CSR sparse contraction inp -> (B,C,K,H,W),
//    backward = CSR transpose contraction (B,C,K,H,W) -> inp.
//  * §Backward direction: both run in the gather direction (each output
//    element reads a bounded neighbourhood), with no atomics; the scatter
//    backward was retired because of atomic contention.
//  * §BC_TILE optimization: one thread block serves many channels so each
//    psi index/value load is amortised over them.
//
// Design (sm_103a):
//  * psi is walked as runs: for output row ho and input row hi the support
//    is one wrapped window of columns, symmetric about offset 0.  The basis
//    values of offset -delta equal those of +delta for the {1, cos} parts and
//    are negated for the sin part, so every run is processed as mirrored
//    pairs: p = x[+d] + x[-d], q = x[+d] - x[-d], acc += w * (p or q).  The
//    pair weights (halved for the self-mirrored offsets) come from psi.hval.
//  * A block owns 32 channels (one per lane) x 64 output columns (8 per
//    thread) of one output row (forward) or input row (transpose).  The
//    wrapped window of the current run is staged in shared memory as fp32
//    with an odd row pitch (lane = channel -> conflict-free), and each thread
//    keeps K x 8 fp32 accumulators in registers.
//  * Blocks of the forward are launched heaviest output rows first (psi.row_order).

#include "disco_gather.cuh"

namespace disco {
namespace {

constexpr int kThreads = 256;  // 8 warps
constexpr int kTW = 8;         // output columns per thread
constexpr int kTile = 64;      // output columns per block

struct ContractArgs {
  const void* in;
  void* out;
  int BC, Hin, Win, Hout, Wout, Kp;
  const int32_t* run_ptr;
  const disco_run* runs;
  const int32_t* trun_ptr;
  const int32_t* truns;
  const float* hval;
  const int32_t* row_order;
  int vec_ok;  // output rows are 16-byte aligned
};

template <typename T>
__device__ __forceinline__ float ld_in(const T* p) {
  return to_f32(p[0]);
}

// Stores 8 consecutive outputs (acc[t], t = 0..7) at dst[0..7], n valid.
template <typename T>
__device__ __forceinline__ void store8(T* dst, const float* v, int n, bool vec);
template <>
__device__ __forceinline__ void store8<float>(float* dst, const float* v, int n, bool vec) {
  if (vec && n == 8) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    for (int t = 0; t < n; ++t) dst[t] = v[t];
  }
}
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* dst, const float* v, int n,
                                                     bool vec) {
  if (vec && n == 8) {
    __nv_bfloat162 p0 = __floats2bfloat162_rn(v[0], v[1]);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(v[2], v[3]);
    __nv_bfloat162 p2 = __floats2bfloat162_rn(v[4], v[5]);
    __nv_bfloat162 p3 = __floats2bfloat162_rn(v[6], v[7]);
    uint4 u;
    u.x = *reinterpret_cast<uint32_t*>(&p0);
    u.y = *reinterpret_cast<uint32_t*>(&p1);
    u.z = *reinterpret_cast<uint32_t*>(&p2);
    u.w = *reinterpret_cast<uint32_t*>(&p3);
    reinterpret_cast<uint4*>(dst)[0] = u;
  } else {
    for (int t = 0; t < n; ++t) dst[t] = __float2bfloat16_rn(v[t]);
  }
}

// ------------------------------------------------------------- forward --
//
// X[bc,k,ho,wo] = sum_runs sum_{delta=0..D} w_k(delta) * (x[hi, S wo + delta] +/- x[hi, S wo - delta])
// Lane = channel (32 per block), warp = 8 consecutive output columns.
template <typename T, int K, int S, bool ANISO>
using FwdGather = RowGather<T, K, S, ANISO, 32, kTW, kTile, kThreads>;

template <typename T, int K, int S, bool ANISO>
__global__ void __launch_bounds__(kThreads, 2) fwd_kernel(const ContractArgs a) {
  extern __shared__ float sm[];
  using G = FwdGather<T, K, S, ANISO>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ho = a.row_order[blockIdx.z];
  const int bc0 = blockIdx.y * 32;
  const int wo_blk = blockIdx.x * kTile;
  const int o0 = warp * kTW;
  typename G::Args ga;
  ga.x = reinterpret_cast<const T*>(a.in);
  ga.bc0 = bc0;
  ga.BC = a.BC;
  ga.Hin = a.Hin;
  ga.W = a.Win;
  ga.run_ptr = a.run_ptr;
  ga.runs = a.runs;
  ga.hval = a.hval;
  ga.Kp = a.Kp;
  float acc[K][kTW];
  G::run(acc, sm, ga, ho, wo_blk, lane, o0, threadIdx.x, 0);

  const int bc = bc0 + lane;
  const int wo = wo_blk + o0;
  if (bc >= a.BC || wo >= a.Wout) return;
  const int n = min(kTW, a.Wout - wo);
  T* X = reinterpret_cast<T*>(a.out);
#pragma unroll
  for (int k = 0; k < K; ++k) {
    T* dst = X + (((size_t)bc * K + k) * a.Hout + ho) * a.Wout + wo;
    store8<T>(dst, acc[k], n, a.vec_ok != 0);
  }
}

// ----------------------------------------------------------- transpose --
//
// gx[bc,hi,wi] = sum_{runs reading hi} sum_k sum_{delta=0..D} w_k(delta) *
//                (G_k[ho, (wi - delta)/S] +/- G_k[ho, (wi + delta)/S])
// (terms only where S divides wi -/+ delta).  One block owns 32 channels x
// 64 columns of input row hi; the runs that read hi come from psi.truns.
template <int S>
struct TWin {
  static constexpr int kSingle = (kTile - 1 + 2 * kDCMax) / S + 1;
  static constexpr int kDouble = (kTile - 1 + kDCMax) / S + 1;
  static constexpr int kLen = (kSingle > 2 * kDouble) ? kSingle : 2 * kDouble;
};

template <typename T, int K, int S, bool ANISO>
__global__ void __launch_bounds__(kThreads, 2) bwd_kernel(const ContractArgs a) {
  extern __shared__ float sm[];
  constexpr int kPitch = TWin<S>::kLen | 1;
  float* win = sm;
  float* wts = sm + 32 * kPitch;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int hi = blockIdx.z;
  const int bc0 = blockIdx.y * 32;
  const int wi_blk = blockIdx.x * kTile;  // multiple of S
  const int o0 = warp * kTW;              // multiple of S
  const T* G = reinterpret_cast<const T*>(a.in);
  const int Wo = a.Wout;

  float acc[kTW];
#pragma unroll
  for (int t = 0; t < kTW; ++t) acc[t] = 0.f;

  const int t_begin = a.trun_ptr[hi], t_end = a.trun_ptr[hi + 1];
  for (int tr = t_begin; tr < t_end; ++tr) {
    const disco_run run = a.runs[a.truns[tr]];
    const int steps = run.D + 1;
    const int dc = min(kDCMax, (steps + 7) & ~7);
    for (int k = 0; k < K; ++k) {
      const T* Gk = G + ((size_t)k * a.Hout + run.ho) * Wo;
      const size_t plane = (size_t)K * a.Hout * Wo;
      for (int da = 0; da < steps; da += dc) {
        const int nd = min(dc, steps - da);
        const bool single = (da == 0);
        // minus side: wo = (wi - delta)/S = start_m + (o - u + offm)/S
        // plus side:  wo = (wi + delta)/S = start_p + (o + u + offp)/S
        const int len_p = single ? (kTile - 1 + 2 * dc) / S + 1 : (kTile - 1 + dc) / S + 1;
        const int start_m = (wi_blk - da - dc) / S;  // exact: all terms multiples of S
        const int start_p = single ? start_m : (wi_blk + da) / S;
        const int offm = dc;
        const int offp = single ? dc : 0;
        float* wm = win;
        float* wp = single ? win : win + len_p;
        __syncthreads();
        {
          // one warp per window row (channel x side), lanes along the columns
          const int nrows = 32 * (single ? 1 : 2);
          const int smn = imod(start_m, Wo), sp = imod(start_p, Wo);
          for (int row = threadIdx.x >> 5; row < nrows; row += kThreads / 32) {
            const int w2 = row >= 32;
            const int c = row - w2 * 32;
            const int bc = bc0 + c;
            const int base = w2 ? sp : smn;
            float* dst = win + c * kPitch + w2 * len_p;
            const T* src = Gk + bc * plane;
            for (int j = lane; j < len_p; j += 32) {
              int col = base + j;
              if (col >= Wo) col %= Wo;
              dst[j] = (bc < a.BC) ? ld_in(src + col) : 0.f;
            }
          }
          for (int i = threadIdx.x; i < dc; i += kThreads)
            wts[i] = (i < nd) ? a.hval[(size_t)(run.hoff + da + i) * a.Kp + k] : 0.f;
        }
        __syncthreads();
        const bool neg = ANISO && (k % 3 == 2);
        for (int ub = 0; ub < nd; ub += 8) {
          // o0, ub, offm, offp are multiples of S, so both bases are exact and
          // the per-(t, u) offsets below are compile-time constants
          const float* bm = wm + lane * kPitch + (o0 - ub + offm) / S;
          const float* bp = wp + lane * kPitch + (o0 + ub + offp) / S;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float w = wts[ub + u];
#pragma unroll
            for (int t = 0; t < kTW; ++t) {
              if ((t - u) % S != 0) continue;  // S must divide wi -/+ delta
              const float gm = bm[(t - u) / S];
              const float gp = bp[(t + u) / S];
              acc[t] = fmaf(w, neg ? gm - gp : gm + gp, acc[t]);
            }
          }
        }
      }
    }
  }

  const int bc = bc0 + lane;
  const int wi = wi_blk + o0;
  if (bc >= a.BC || wi >= a.Win) return;
  const int n = min(kTW, a.Win - wi);
  T* gx = reinterpret_cast<T*>(a.out);
  store8<T>(gx + ((size_t)bc * a.Hin + hi) * a.Win + wi, acc, n, a.vec_ok != 0);
}

template <typename T, int K, int S, bool ANISO>
constexpr size_t fwd_smem() {
  return (size_t)FwdGather<T, K, S, ANISO>::kSmemFloats * sizeof(float);
}
template <int S>
constexpr size_t bwd_smem() {
  return (size_t)(32 * (TWin<S>::kLen | 1) + kDCMax) * sizeof(float);
}

template <typename T, int K, int S, bool ANISO>
int launch_fwd(const ContractArgs& a, cudaStream_t st) {
  auto kern = fwd_kernel<T, K, S, ANISO>;
  size_t smem = fwd_smem<T, K, S, ANISO>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return check_launch("disco_fwd attribute");
  dim3 grid((a.Wout + kTile - 1) / kTile, (a.BC + 31) / 32, a.Hout);
  kern<<<grid, kThreads, smem, st>>>(a);
  return check_launch("disco_fwd");
}

template <typename T, int K, int S, bool ANISO>
int launch_bwd(const ContractArgs& a, cudaStream_t st) {
  auto kern = bwd_kernel<T, K, S, ANISO>;
  size_t smem = bwd_smem<S>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return check_launch("disco_bwd attribute");
  dim3 grid((a.Win + kTile - 1) / kTile, (a.BC + 31) / 32, a.Hin);
  kern<<<grid, kThreads, smem, st>>>(a);
  return check_launch("disco_bwd");
}

template <typename T, int S>
int dispatch(bool fwd, int kind, int K, const ContractArgs& a, cudaStream_t st) {
#define DISCO_CASE(KK, AN)                                                    \
  if (K == KK && (kind == 1) == AN)                                           \
    return fwd ? launch_fwd<T, KK, S, AN>(a, st) : launch_bwd<T, KK, S, AN>(a, st);
  DISCO_CASE(1, false)
  DISCO_CASE(2, false)
  DISCO_CASE(3, false)
  DISCO_CASE(4, false)
  DISCO_CASE(5, false)
  DISCO_CASE(6, false)
  DISCO_CASE(7, false)
  DISCO_CASE(8, false)
  DISCO_CASE(3, true)
  DISCO_CASE(6, true)
  DISCO_CASE(9, true)
#undef DISCO_CASE
  return fail(DISCO_ERR_UNSUPPORTED, "K = %d (kind %d) has no contraction kernel", K, kind);
}

int contract(bool fwd, const disco_psi* psi, const void* in, void* out, int32_t B, int32_t C,
             disco_dtype dtype, void* stream) {
  int st = check_psi(psi);
  if (st) return st;
  if ((st = check_device())) return st;
  if (!in || !out) return fail(DISCO_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(in) || !aligned16(out)) return fail(DISCO_ERR_ALIGNMENT, "tensors must be 16-byte aligned");
  if (B < 1 || C < 1) return fail(DISCO_ERR_INVALID_ARG, "B and C must be >= 1");
  if ((int64_t)B * C > (int64_t)65535 * 32) return fail(DISCO_ERR_UNSUPPORTED, "B*C too large");
  if (dtype != DISCO_F32 && dtype != DISCO_BF16) return fail(DISCO_ERR_UNSUPPORTED, "dtype");
  if (psi->s != 1 && psi->s != 2)
    return fail(DISCO_ERR_UNSUPPORTED, "W_in / W_out = %d (contractions support 1 and 2)", psi->s);
  ContractArgs a;
  a.in = in;
  a.out = out;
  a.BC = B * C;
  a.Hin = psi->grid_in.nlat;
  a.Win = psi->grid_in.nlon;
  a.Hout = psi->grid_out.nlat;
  a.Wout = psi->grid_out.nlon;
  a.Kp = psi->K_pad;
  a.run_ptr = psi->run_ptr;
  a.runs = psi->runs;
  a.trun_ptr = psi->trun_ptr;
  a.truns = psi->truns;
  a.hval = psi->hval;
  a.row_order = psi->row_order;
  int elems16 = dtype == DISCO_F32 ? 4 : 8;
  a.vec_ok = ((fwd ? a.Wout : a.Win) % elems16) == 0;
  cudaStream_t s = (cudaStream_t)stream;
  int kind = psi->basis.kind, K = psi->K;
  if (fwd && dtype == DISCO_BF16) {
    // bf16 forward: the tensor-core Toeplitz kernel where its shape rules hold
    const int tst = fwd_tensor_core(psi, in, out, a.BC, s);
    if (tst != DISCO_ERR_UNSUPPORTED) return tst;
  }
  if (dtype == DISCO_F32)
    return psi->s == 1 ? dispatch<float, 1>(fwd, kind, K, a, s) : dispatch<float, 2>(fwd, kind, K, a, s);
  return psi->s == 1 ? dispatch<__nv_bfloat16, 1>(fwd, kind, K, a, s)
                     : dispatch<__nv_bfloat16, 2>(fwd, kind, K, a, s);
}

}  // namespace
}  // namespace disco

extern "C" int disco_fwd(const disco_psi* psi, const void* x, void* X, int32_t B, int32_t C,
                         disco_dtype dtype, void* stream) {
  return disco::contract(true, psi, x, X, B, C, dtype, stream);
}

extern "C" int disco_bwd(const disco_psi* psi, const void* G, void* gx, int32_t B, int32_t C,
                         disco_dtype dtype, void* stream) {
  return disco::contract(false, psi, G, gx, B, C, dtype, stream);
}
