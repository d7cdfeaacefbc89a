// disco_gather.cuh -- the forward gather of one output-row tile, shared by
// disco_fwd and disco_fused_conv.
//
// For output row ho, a tile of TILE output columns starting at wo_blk and NCH
// channels starting at bc0, each thread accumulates, for its channel `ch` and
// its TW output columns o0 .. o0+TW-1 of the tile,
//
//   acc[k][t] = sum_{runs (ho, hi)} sum_{delta = 0..D} w_k(delta) *
//               (x[hi, S (wo_blk + o0 + t) + delta]  +/-  x[hi, S (wo_blk + o0 + t) - delta])
//
// (minus for the sin component of an anisotropic basis).  This is the CSR
// gather of the DISCO Kernel Development Guide, §Backward direction (every
// output pixel reads only its own bounded neighbourhood), walked run by run with
// mirrored offsets paired.  The NT threads of the group stage the wrapped
// window of the current run in shared memory (fp32, row pitch = 1 mod 32)
// and the pair weights next to it; the group synchronises on named barrier
// `bar_id`.  Offsets are processed in chunks of up to kDCMax pair steps: the
// first chunk of a run uses one window holding both sides, later chunks one
// window per side.
#pragma once

#include "disco_bounds.cuh"
#include "disco_internal.cuh"

namespace disco {

constexpr int kDCMax = 32;  // pair steps per staged chunk

__device__ __forceinline__ void group_sync(int bar_id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(nthreads) : "memory");
}

// true in every thread of the named-barrier group iff `pred` holds in all of them
__device__ __forceinline__ bool group_all(bool pred, int bar_id, int nthreads) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(bar_id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ int imod(int a, int m) {
  int r = a % m;
  return r < 0 ? r + m : r;
}

template <typename T, int K, int S, bool ANISO, int NCH, int TW, int TILE, int NT>
struct RowGather {
  static constexpr int kSingle = S * (TILE - 1) + 2 * kDCMax - 1;  // first chunk: both sides
  static constexpr int kDouble = S * (TILE - 1) + kDCMax;          // later chunks: per side
  static constexpr int kLen = (kSingle > 2 * kDouble) ? kSingle : 2 * kDouble;
  static constexpr int kPitch = (kLen + 31) / 32 * 32 + 1;          // = 1 (mod 32)
  static constexpr int kSmemFloats = NCH * kPitch + kDCMax * K;

  struct Args {
    const T* x;  // [BC][Hin][Win]
    int bc0, BC, Hin, W;
    const int32_t* run_ptr;
    const disco_run* runs;
    const float* hval;
    int Kp;
    int nruns;        // runs and hval rows of psi (extent checks of the
    long long nhval;  // bounds-checked build)
  };

  __device__ static void run(float (&acc)[K][TW], float* sm, const Args& a, int ho, int wo_blk,
                             int ch, int o0, int tid, int bar_id) {
    float* win = sm;
    float* wts = sm + NCH * kPitch;
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
      for (int t = 0; t < TW; ++t) acc[k][t] = 0.f;
    const int P0 = S * wo_blk;
    const int W = a.W;
    const int r_begin = a.run_ptr[ho];
    int r_end = a.run_ptr[ho + 1];
    if (!DISCO_IN_BOUNDS(r_begin >= 0 && r_begin <= r_end && r_end <= a.nruns)) r_end = r_begin;
    for (int r = r_begin; r < r_end; ++r) {
      const disco_run run = a.runs[r];
      // (every thread of the group reads the same run and skips it alike)
      if (!DISCO_IN_BOUNDS(run.hi >= 0 && run.hi < a.Hin && run.D >= 0 && run.hoff >= 0 &&
                           run.hoff + (long long)run.D + 1 <= a.nhval))
        continue;
      const int steps = run.D + 1;
      const int dc = min(kDCMax, (steps + 7) & ~7);
      const T* xrow = a.x + (size_t)run.hi * W;
      for (int da = 0; da < steps; da += dc) {
        const int nd = min(dc, steps - da);
        const bool single = (da == 0);
        const int len_p = single ? S * (TILE - 1) + 2 * dc - 1 : S * (TILE - 1) + dc;
        const int start_p = single ? P0 - (dc - 1) : P0 + da;
        const int start_m = P0 - da - (dc - 1);
        const int offp = single ? dc - 1 : 0;
        const int offm = dc - 1;
        group_sync(bar_id, NT);
        {
          // one warp per window row (channel x side), lanes along the columns:
          // coalesced loads, no integer division
          const int nrows = NCH * (single ? 1 : 2);
          const int sp = imod(start_p, W), smn = imod(start_m, W);
          for (int row = tid >> 5; row < nrows; row += NT / 32) {
            const int w2 = row >= NCH;
            const int c = row - w2 * NCH;
            const int bc = a.bc0 + c;
            const int base = w2 ? smn : sp;
            float* dst = win + c * kPitch + w2 * len_p;
            const T* src = xrow + (size_t)bc * a.Hin * W;
            for (int j = tid & 31; j < len_p; j += 32) {
              int col = base + j;
              if (col >= W) col %= W;
              dst[j] = (bc < a.BC && DISCO_IN_BOUNDS(col >= 0 && col < W)) ? to_f32(src[col]) : 0.f;
            }
          }
          for (int i = tid; i < dc * K; i += NT) {
            const int u = i / K, k = i - u * K;
            wts[i] = (u < nd) ? a.hval[(size_t)(run.hoff + da + u) * a.Kp + k] : 0.f;
          }
        }
        group_sync(bar_id, NT);
        const float* bp = win + (single ? 0 : 0) + ch * kPitch + S * o0 + offp;
        const float* bm = win + (single ? 0 : len_p) + ch * kPitch + S * o0 + offm;
        for (int ub = 0; ub < nd; ub += 8) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            float w[K];
#pragma unroll
            for (int k = 0; k < K; ++k) w[k] = wts[(ub + u) * K + k];
#pragma unroll
            for (int t = 0; t < TW; ++t) {
              const float xp = bp[ub + S * t + u];
              const float xm = bm[-ub + S * t - u];
              const float pp = xp + xm;
              if (ANISO) {
                const float qq = xp - xm;
#pragma unroll
                for (int k = 0; k < K; ++k)
                  acc[k][t] = fmaf(w[k], (k % 3 == 2) ? qq : pp, acc[k][t]);
              } else {
#pragma unroll
                for (int k = 0; k < K; ++k) acc[k][t] = fmaf(w[k], pp, acc[k][t]);
              }
            }
          }
        }
      }
    }
  }
};

}  // namespace disco
