// disco_contract.cu -- forward and transpose DISCO contractions on CUDA cores.
//
// DISCO Kernel Development Guide (torch-harmonics):
//  * §Architecture snapshot: the forward kernel contracts the input grid with
//    the sparse psi into the [B, C, K, H_out, W_out] tensor; the backward
//    kernel applies the transpose of that map, back to the input grid.
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
  const float* hval_full;  // union layout values [nnz][Kp] (signed offsets)
  const int32_t* row_order;
  int vec_ok;  // output rows are 16-byte aligned
  int nruns;                // runs, hval rows and union entries of psi
  long long nhval, nnz;     // (extent checks of the bounds-checked build)
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
template <>
__device__ __forceinline__ void store8<__half>(__half* dst, const float* v, int n, bool vec) {
  if (vec && n == 8) {
    __half2 p0 = __floats2half2_rn(v[0], v[1]);
    __half2 p1 = __floats2half2_rn(v[2], v[3]);
    __half2 p2 = __floats2half2_rn(v[4], v[5]);
    __half2 p3 = __floats2half2_rn(v[6], v[7]);
    uint4 u;
    u.x = *reinterpret_cast<uint32_t*>(&p0);
    u.y = *reinterpret_cast<uint32_t*>(&p1);
    u.z = *reinterpret_cast<uint32_t*>(&p2);
    u.w = *reinterpret_cast<uint32_t*>(&p3);
    reinterpret_cast<uint4*>(dst)[0] = u;
  } else {
    for (int t = 0; t < n; ++t) dst[t] = __float2half_rn(v[t]);
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
  int ho = a.row_order[blockIdx.z];
  if (!DISCO_IN_BOUNDS(ho >= 0 && ho < a.Hout)) ho = 0;
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
  ga.nruns = a.nruns;
  ga.nhval = a.nhval;
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
// gx[bc,hi,j] = sum_{runs (ho, hi)} sum_k sum_{delta in run} psi_k(delta) * G_k[ho, (j - delta)/S]
// (terms only where S divides j - delta).  Polyphase form: with j = S q + p
// and delta = S e + p, gx[S q + p] = sum psi_k(S e + p) G_k[q - e], i.e. a
// correlation per phase p on the decimated index q.
//
// One block owns input row hi, 32 channels (one per lane) and 64 decimated
// positions (S * 64 input columns); a thread owns 8 positions x S phases.
// Per run and chunk of up to kBDC offsets the block stages the G windows of
// ALL K planes (bf16, pitch = 2 mod 4 elements so the 32 lanes hit 32 banks)
// and the run's psi values for the chunk, then every thread accumulates
// K x (offsets) x 8 terms per phase in registers.  For S = 2 both phases
// read the same 11 staged values per block of 8 offsets.
constexpr int kBQ = 64;     // decimated positions per block
constexpr int kBT = 8;      // decimated positions per thread
constexpr int kBDC = 32;    // offsets per staged chunk (multiple of 8)

// staged G window element: bf16 bits for bf16 inputs (exact), fp32 for fp32
template <typename T>
struct BwdStage {
  using E = uint16_t;
  __device__ static E put(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
  __device__ static float get(E e) { return __uint_as_float((uint32_t)e << 16); }
};
template <>
struct BwdStage<float> {
  using E = float;
  __device__ static E put(float v) { return v; }
  __device__ static float get(E e) { return e; }
};

template <typename T, int S>
struct BwdWin {
  static constexpr int kLen = kBQ + kBDC / S + 2;  // G window per k and channel
  // row pitch in elements: 32 lanes (channels) must hit 32 different banks
  static constexpr int kPitch = sizeof(typename BwdStage<T>::E) == 2 ? ((kLen + 1) / 4) * 4 + 2
                                                                      : (kLen | 1);
};

template <typename T, int K, int S>
constexpr size_t bwd_smem() {
  return (size_t)K * 32 * BwdWin<T, S>::kPitch * sizeof(typename BwdStage<T>::E) +
         (size_t)K * kBDC * sizeof(float);
}

template <typename T, int K, int S, bool ANISO>
__global__ void __launch_bounds__(kThreads, 2) bwd_kernel(const ContractArgs a) {
  extern __shared__ __align__(16) uint8_t bsm[];
  using St = BwdStage<T>;
  using E = typename St::E;
  constexpr int kPitch = BwdWin<T, S>::kPitch;
  E* sG = reinterpret_cast<E*>(bsm);                                            // [K][32][kPitch]
  float* sW = reinterpret_cast<float*>(bsm + (size_t)K * 32 * kPitch * sizeof(E));  // [K][kBDC]

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int hi = blockIdx.z;
  const int bc0 = blockIdx.y * 32;
  const int qb = blockIdx.x * kBQ;
  const int q0 = warp * kBT;  // first decimated position of this thread inside the block
  const T* G = reinterpret_cast<const T*>(a.in);
  const int Wo = a.Wout;
  const size_t plane = (size_t)K * a.Hout * Wo;

  float acc[S][kBT];
#pragma unroll
  for (int p = 0; p < S; ++p)
#pragma unroll
    for (int t = 0; t < kBT; ++t) acc[p][t] = 0.f;

  const int t_begin = a.trun_ptr[hi];
  int t_end = a.trun_ptr[hi + 1];
  if (!DISCO_IN_BOUNDS(t_begin >= 0 && t_begin <= t_end && t_end <= a.nruns)) t_end = t_begin;
  for (int tr = t_begin; tr < t_end; ++tr) {
    const int ri = a.truns[tr];
    if (!DISCO_IN_BOUNDS(ri >= 0 && ri < a.nruns)) continue;  // the whole block skips it alike
    const disco_run run = a.runs[ri];
    const int dlo = (run.len == a.Win) ? -(a.Win / 2) : -run.npair;
    const int dhi = dlo + run.len - 1;
    if (!DISCO_IN_BOUNDS(run.ho >= 0 && run.ho < a.Hout && run.len >= 1 && run.e0 >= 0 &&
                         run.e0 + (long long)run.len <= a.nnz))
      continue;
    const int dstart = (dlo >= 0) ? (dlo & ~7) : -(((-dlo) + 7) & ~7);  // multiple of 8, <= dlo
    for (int da = dstart; da <= dhi; da += kBDC) {
      // decimated G index of (j, delta) is (j - delta)/S; over the block and chunk
      // it runs from gs = (S*qb - da - kBDC)/S upward (exact: all multiples of S)
      const int gs = (S * qb - da - kBDC) / S;
      __syncthreads();
      // stage G windows of all K planes: one warp per (k, channel) row
      const int g0 = imod(gs, Wo);
      for (int row = warp; row < K * 32; row += kThreads / 32) {
        const int k = row >> 5, c = row & 31;
        const int bc = bc0 + c;
        const T* src = G + (size_t)bc * plane + ((size_t)k * a.Hout + run.ho) * Wo;
        E* dst = sG + (size_t)row * kPitch;
        for (int i = lane; i < BwdWin<T, S>::kLen; i += 32) {
          int col = g0 + i;
          if (col >= Wo) col %= Wo;
          dst[i] = St::put((bc < a.BC && DISCO_IN_BOUNDS(col >= 0 && col < Wo)) ? to_f32(src[col]) : 0.f);
        }
      }
      // psi values of the chunk, signed offsets, zero outside the run
      for (int i = threadIdx.x; i < K * kBDC; i += kThreads) {
        const int k = i / kBDC, u = i - k * kBDC;
        const int d = da + u;
        sW[i] = (d >= dlo && d <= dhi) ? a.hval_full[(size_t)(run.e0 + d - dlo) * a.Kp + k] : 0.f;
      }
      __syncthreads();
      const int nub = min(kBDC, dhi - da + 1);
#pragma unroll 1
      for (int k = 0; k < K; ++k) {
        const E* gk = sG + ((size_t)k * 32 + lane) * kPitch;
        const float* wk = sW + k * kBDC;
        for (int ub = 0; ub < nub; ub += 8) {
          // window index of (position qb + q0 + t, delta = da + ub + u, phase p):
          //   qb + q0 + t - (da + ub)/S + (p - u)/S - gs,  and qb - gs = (da + kBDC)/S,
          //   so it is base + t + (p - u)/S with base = q0 + (kBDC - ub)/S,
          //   which stays in [1, kBQ - 1 + kBDC/S] < the staged window length
          const int base = q0 + (kBDC - ub) / S;
          float w[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) w[u] = wk[ub + u];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
#pragma unroll
            for (int p = 0; p < S; ++p) {
              if (((p - u) % S + S) % S != 0) continue;
#pragma unroll
              for (int t = 0; t < kBT; ++t) {
                const float gv = St::get(gk[base + t + (p - u) / S]);
                acc[p][t] = fmaf(w[u], gv, acc[p][t]);
              }
            }
          }
        }
      }
    }
  }

  const int bc = bc0 + lane;
  if (bc >= a.BC) return;
  T* gx = reinterpret_cast<T*>(a.out);
  T* row = gx + ((size_t)bc * a.Hin + hi) * a.Win;
  // output columns j = S*(qb + q0 + t) + p
  float v[S * kBT];
#pragma unroll
  for (int t = 0; t < kBT; ++t)
#pragma unroll
    for (int p = 0; p < S; ++p) v[t * S + p] = acc[p][t];
  const int j0 = S * (qb + q0);
  if (j0 >= a.Win) return;
#pragma unroll
  for (int h = 0; h < S; ++h) {
    const int jj = j0 + h * 8;
    if (jj < a.Win) store8<T>(row + jj, v + h * 8, min(8, a.Win - jj), a.vec_ok != 0);
  }
}

template <typename T, int K, int S, bool ANISO>
constexpr size_t fwd_smem() {
  return (size_t)FwdGather<T, K, S, ANISO>::kSmemFloats * sizeof(float);
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
  size_t smem = bwd_smem<T, K, S>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return check_launch("disco_bwd attribute");
  dim3 grid((a.Win + S * kBQ - 1) / (S * kBQ), (a.BC + 31) / 32, a.Hin);
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

}  // namespace

int contract(bool fwd, const disco_psi* psi, const void* in, void* out, int32_t B, int32_t C,
             disco_dtype dtype, void* stream, bool check_ptrs) {
  int st = check_psi(psi);
  if (st) return st;
  if ((st = check_device())) return st;
  if (!in || !out) return fail(DISCO_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(in) || !aligned16(out)) return fail(DISCO_ERR_ALIGNMENT, "tensors must be 16-byte aligned");
  if (check_ptrs && ((st = check_dev_ptr(in, fwd ? "x" : "G")) || (st = check_dev_ptr(out, fwd ? "X" : "gx"))))
    return st;
  if (B < 1 || C < 1) return fail(DISCO_ERR_INVALID_ARG, "B and C must be >= 1");
  if ((int64_t)B * C > (int64_t)65535 * 32) return fail(DISCO_ERR_UNSUPPORTED, "B*C too large");
  if (dtype != DISCO_F32 && dtype != DISCO_BF16 && dtype != DISCO_F16) return fail(DISCO_ERR_UNSUPPORTED, "dtype");
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
  a.hval_full = psi->val;
  a.nruns = (int)psi->nruns;
  a.nhval = psi->nhval;
  a.nnz = psi->nnz;
  a.row_order = psi->row_order;
  int elems16 = dtype == DISCO_F32 ? 4 : 8;
  a.vec_ok = ((fwd ? a.Wout : a.Win) % elems16) == 0;
  cudaStream_t s = (cudaStream_t)stream;
  int kind = psi->basis.kind, K = psi->K;
  if (dtype != DISCO_F32) {
    // bf16 / fp16: the tensor-core Toeplitz kernels where their shape rules hold
    const bool f16 = dtype == DISCO_F16;
    const int tst = fwd ? fwd_tensor_core(psi, in, out, a.BC, s, f16)
                        : bwd_tensor_core(psi, in, out, a.BC, s, false, f16);
    if (tst != DISCO_ERR_UNSUPPORTED) return tst;
  }
  if (dtype == DISCO_F32)
    return psi->s == 1 ? dispatch<float, 1>(fwd, kind, K, a, s) : dispatch<float, 2>(fwd, kind, K, a, s);
  if (dtype == DISCO_F16)
    return psi->s == 1 ? dispatch<__half, 1>(fwd, kind, K, a, s) : dispatch<__half, 2>(fwd, kind, K, a, s);
  return psi->s == 1 ? dispatch<__nv_bfloat16, 1>(fwd, kind, K, a, s)
                     : dispatch<__nv_bfloat16, 2>(fwd, kind, K, a, s);
}

// This unit's word of failed range checks (always 0 outside the bounds-checked build).
DISCO_BOUNDS_READER(contract_bounds)

}  // namespace disco

extern "C" int disco_fwd(const disco_psi* psi, const void* x, void* X, int32_t B, int32_t C,
                         disco_dtype dtype, void* stream) {
  disco::NvtxScope nvtx_scope("disco_fwd");
  return disco::contract(true, psi, x, X, B, C, dtype, stream, true);
}

extern "C" int disco_bwd(const disco_psi* psi, const void* G, void* gx, int32_t B, int32_t C,
                         disco_dtype dtype, void* stream) {
  disco::NvtxScope nvtx_scope("disco_bwd");
  return disco::contract(false, psi, G, gx, B, C, dtype, stream, true);
}
