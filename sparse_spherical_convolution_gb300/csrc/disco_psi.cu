// disco_psi.cu -- device construction of the DISCO filter tensor psi.
//
// DISCO Kernel Development Guide (torch-harmonics), §kpacked layout: psi is
// converted once at init into a neighbour list shared across the K basis
// functions, with the values of all k side by side (K padded to K_PAD =
// ceil(K/8)*8).  Here the whole build runs on the GPU in fp64:
//
//   count   (one block per output row)  for each input row hi, the half-width
//           m of the union support (the support of one input row is a
//           contiguous window symmetric about offset 0, because the distance
//           grows with |longitude offset|), per-ring structural counts and
//           per-ring sums of hat * quadrature;
//   plan    per-row totals are copied to the host to size the buffers;
//   scan    row pointers, CSR row pointers, run and pair-weight offsets;
//   fill    indices, fp32 values (union layout, CSR layout, pair weights),
//           run table;
//   trans   the transposed run list (runs grouped by input row) for the
//           gather-direction transpose contraction.
//
// Definitions (the page names the operations but not the basis, so these are
// the plainest readings of the workload text):
//   colatitude  (i + 1/2) pi / H, or i pi / (H - 1) on a pole grid (pi exactly at i = H-1)
//   distance    haversine great-circle distance, longitude offset 2 pi delta / W_in
//   hats        width w = cutoff / R, h_r(d) = max(0, 1 - |d - r w| / w)
//   bearing     atan2(sin dphi sin th_i, sin th_o cos th_i - cos th_o sin th_i cos dphi)
//   quadrature  sin(colatitude), exactly 0 on the pole rows of a pole grid
//   support     h_r > 1e-9 and quadrature > 0
//   value       h_r * {1, cos beta, sin beta}[a] * q / N(r, ho), N = sum of h_r q over ring r
// All fp64 arithmetic uses explicitly rounded operations (no fused
// multiply-add), so the index structures are bit-exact and the values agree
// with a plain fp64 evaluation to the last fp32 bit in all but rare ties.

#include <stdio.h>
#include <string.h>

#include <vector>

#include "disco_bounds.cuh"
#include "disco_internal.cuh"

namespace disco {
namespace {

constexpr double kPi = 3.14159265358979323846;
constexpr double kTauSupport = 1e-9;
constexpr double kCoincident = 1e-12;
constexpr int kMaxRad = 8;

struct PsiGeom {
  int Hin, Win, pin, Hout, Wout, pout;  // pin / pout: 0 midpoint, 1 poles, 2 Legendre-Gauss
  int kind, R, K, Kp;
  double cutoff, width;
  const double* lg;  // workspace table [theta_in (Hin) | w_in (Hin) | theta_out (Hout)] for Legendre-Gauss grids
};

__device__ double colat(int H, int poles, int i) {
  if (poles) {
    if (i == H - 1) return kPi;
    return __ddiv_rn(__dmul_rn((double)i, kPi), (double)(H - 1));
  }
  return __ddiv_rn(__dmul_rn(__dadd_rn((double)i, 0.5), kPi), (double)H);
}

__device__ double quadw(int H, int poles, int i) {
  if (poles && (i == 0 || i == H - 1)) return 0.0;
  return sin(colat(H, poles, i));
}

// Legendre-Gauss node i of order n (descending x): Newton's method on P_n
// from cos(pi (i + 3/4) / (n + 1/2)), P_n and P_n' by the three-term
// recurrence; the weight 2 / ((1 - x^2) P_n'(x)^2).
__device__ void gauss_node(int n, int i, double* x_out, double* w_out) {
  double x = cos(kPi * ((double)i + 0.75) / ((double)n + 0.5));
  double pn = 0.0, pm = 0.0;
  for (int it = 0; it < 100; ++it) {
    pm = 1.0;
    pn = x;
    for (int j = 1; j < n; ++j) {
      const double nx = ((2.0 * j + 1.0) * x * pn - (double)j * pm) / ((double)j + 1.0);
      pm = pn;
      pn = nx;
    }
    const double dp = (double)n * (x * pn - pm) / -((1.0 - x) * (1.0 + x));
    const double dx = pn / dp;
    x -= dx;
    if (fabs(dx) <= 1e-15) break;
  }
  pm = 1.0;
  pn = x;
  for (int j = 1; j < n; ++j) {
    const double nx = ((2.0 * j + 1.0) * x * pn - (double)j * pm) / ((double)j + 1.0);
    pm = pn;
    pn = nx;
  }
  const double dp = (double)n * (x * pn - pm) / -((1.0 - x) * (1.0 + x));
  *x_out = x;
  *w_out = 2.0 / ((1.0 - x) * (1.0 + x) * dp * dp);
}

// Colatitude and quadrature weight of a row of the input / output grid.
__device__ double th_in(const PsiGeom& g, int i) { return g.pin == 2 ? g.lg[i] : colat(g.Hin, g.pin, i); }
__device__ double q_in(const PsiGeom& g, int i) { return g.pin == 2 ? g.lg[g.Hin + i] : quadw(g.Hin, g.pin, i); }
__device__ double th_out(const PsiGeom& g, int i) {
  return g.pout == 2 ? g.lg[2 * g.Hin + i] : colat(g.Hout, g.pout, i);
}

// distance and bearing from (th_o, 0) to (th_i, 2 pi delta / W)
__device__ void geometry(double th_o, double th_i, int delta, int W, double* d, double* beta) {
  int ad = delta < 0 ? -delta : delta;
  double half = __ddiv_rn(__dmul_rn(kPi, (double)ad), (double)W);
  double s1 = sin(__dmul_rn(0.5, __dsub_rn(th_i, th_o)));
  double s2 = sin(half);
  double so = sin(th_o), si = sin(th_i), co = cos(th_o), ci = cos(th_i);
  double hav = __dadd_rn(__dmul_rn(s1, s1), __dmul_rn(__dmul_rn(so, si), __dmul_rn(s2, s2)));
  if (hav > 1.0) hav = 1.0;
  *d = __dmul_rn(2.0, asin(sqrt(hav)));
  double twice = __dmul_rn(2.0, half);
  double sdp = sin(twice), cdp = cos(twice);
  if (delta < 0) sdp = -sdp;
  *beta = atan2(__dmul_rn(sdp, si), __dsub_rn(__dmul_rn(so, ci), __dmul_rn(__dmul_rn(co, si), cdp)));
}

__device__ double hat(double d, int r, double width) {
  double v = __dsub_rn(1.0, __ddiv_rn(fabs(__dsub_rn(d, __dmul_rn((double)r, width))), width));
  return v > 0.0 ? v : 0.0;
}

// largest |delta| of one ring (W/2 for even W: the antipodal column)
__device__ __host__ inline int half_ring(int W) { return W / 2; }

// union support at |delta| = ad; fills hats and structural flags
__device__ bool support_at(const PsiGeom& g, double th_o, double th_i, double q, int ad,
                           double* h, bool* st, double* d, double* beta) {
  geometry(th_o, th_i, ad, g.Win, d, beta);
  bool any = false;
  for (int r = 0; r < g.R; ++r) {
    h[r] = hat(*d, r, g.width);
    st[r] = (h[r] > kTauSupport) && (q > 0.0);
    any |= st[r];
  }
  return any;
}

// entries of a run with |delta| = ad: 1 for offset 0 and for the antipodal
// column of an even ring, else 2 (delta and -delta)
__device__ __host__ inline int mult_at(int ad, int W) {
  return (ad == 0 || (2 * ad == W)) ? 1 : 2;
}

__device__ __host__ inline int run_len(int m, int W) {
  if (m < 0) return 0;
  if (m >= half_ring(W)) return W;  // full ring
  return 2 * m + 1;
}

constexpr int kRS = 4;  // per-row totals before the ring counts

// run extent: offsets dlo..dhi (full ring of even width: -W/2 .. W/2 - 1)
__device__ __host__ inline void run_extent(int m, int W, int* dlo, int* dhi) {
  const int len = run_len(m, W);
  *dlo = (len == W) ? -(W / 2) : -m;
  *dhi = *dlo + len - 1;
}
__device__ __host__ inline int floordiv(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }
__device__ __host__ inline int ceildiv(int a, int b) { return -floordiv(-a, b); }
// table row lengths of a run (elements, multiples of 8)
__device__ __host__ inline int ftab_len(int m, int W) { return (run_len(m, W) + 16 + 7) & ~7; }
// half-width of a run in decimated (output) columns: max(EH, -EL) with
// EH = floor(dhi / s), EL = ceil((dlo - s + 1) / s)
__device__ __host__ inline int run_halfwidth(int m, int W, int s) {
  int dlo, dhi;
  run_extent(m, W, &dlo, &dhi);
  const int EH = floordiv(dhi, s), EL = ceildiv(dlo - s + 1, s);
  return EH > -EL ? EH : -EL;
}

struct Workspace {
  int32_t* mtab;      // [Hout][Hin]
  int32_t* ringcnt;   // [Hout][Hin][R]
  double* hq;         // [Hout][Hin][R]
  int32_t* rowsum;    // [Hout][4 + R]: len, runs, hval rows, ftab elements, ring counts
  int32_t* off;       // [Hout][Hin]: entry offset of the run inside its row
  int32_t* runidx;    // [Hout][Hin]
  int32_t* csroff;    // [Hout][Hin][R]
  int32_t* hofftab;   // [Hout][Hin]
  int32_t* ftofftab;  // [Hout][Hin]: forward table offset of the run
  double* norm;       // [Hout][R]
  int32_t* tcount;    // [Hin + 1]
  int32_t* gcnt;      // [ngroups][2]: entries, blocks of each input-row group
  int32_t* gboff;     // [ngroups]: first block of each group
  double* lg;         // [2 Hin + Hout]: Legendre-Gauss colatitudes and input weights
};

__host__ __device__ inline int num_groups(const PsiGeom& g) { return (g.Hin + kGrpRows - 1) / kGrpRows; }

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

size_t carve_workspace(const PsiGeom& g, char* base, Workspace* ws) {
  size_t HH = (size_t)g.Hout * g.Hin, o = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + o : nullptr;
    o += align256(bytes);
    return p;
  };
  Workspace w;
  w.mtab = (int32_t*)take(HH * 4);
  w.ringcnt = (int32_t*)take(HH * g.R * 4);
  w.hq = (double*)take(HH * g.R * 8);
  w.rowsum = (int32_t*)take((size_t)g.Hout * (kRS + g.R) * 4);
  w.ftofftab = (int32_t*)take(HH * 4);
  w.off = (int32_t*)take(HH * 4);
  w.runidx = (int32_t*)take(HH * 4);
  w.csroff = (int32_t*)take(HH * g.R * 4);
  w.hofftab = (int32_t*)take(HH * 4);
  w.norm = (double*)take((size_t)g.Hout * g.R * 8);
  w.tcount = (int32_t*)take((size_t)(g.Hin + 1) * 4);
  w.gcnt = (int32_t*)take((size_t)num_groups(g) * 2 * 4);
  w.gboff = (int32_t*)take((size_t)num_groups(g) * 4);
  w.lg = (double*)take((size_t)(2 * g.Hin + g.Hout) * 8);
  if (ws) *ws = w;
  return o;
}

// ------------------------------------------------------------- kernels --

// Legendre-Gauss tables of the grids that use them; one thread per row.
__global__ void lg_kernel(PsiGeom g, Workspace ws) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  double x, w;
  if (t < g.Hin) {
    if (g.pin != 2) return;
    gauss_node(g.Hin, t, &x, &w);
    ws.lg[t] = acos(x);
    ws.lg[g.Hin + t] = w;
  } else if (t < g.Hin + g.Hout) {
    if (g.pout != 2) return;
    gauss_node(g.Hout, t - g.Hin, &x, &w);
    ws.lg[2 * g.Hin + (t - g.Hin)] = acos(x);
  }
}

// One block per output row; threads stride over input rows.
__global__ void count_kernel(PsiGeom g, Workspace ws) {
  int ho = blockIdx.x;
  double th_o = th_out(g, ho);
  for (int hi = threadIdx.x; hi < g.Hin; hi += blockDim.x) {
    size_t t = (size_t)ho * g.Hin + hi;
    double th_i = th_in(g, hi);
    double q = q_in(g, hi);
    int cnt[kMaxRad] = {0};
    double hqs[kMaxRad] = {0};
    int m = -1;
    if (fabs(__dsub_rn(th_i, th_o)) <= g.cutoff + 1e-9) {
      int hr = half_ring(g.Win);
      for (int ad = 0; ad <= hr; ++ad) {
        double h[kMaxRad], d, beta;
        bool st[kMaxRad];
        if (!support_at(g, th_o, th_i, q, ad, h, st, &d, &beta)) break;
        m = ad;
        int mu = mult_at(ad, g.Win);
        for (int r = 0; r < g.R; ++r)
          if (st[r]) {
            cnt[r] += mu;
            double hq = __dmul_rn(h[r], q);
            hqs[r] = __dadd_rn(hqs[r], hq);
            if (mu == 2) hqs[r] = __dadd_rn(hqs[r], hq);
          }
      }
    }
    ws.mtab[t] = m;
    for (int r = 0; r < g.R; ++r) {
      ws.ringcnt[t * g.R + r] = cnt[r];
      ws.hq[t * g.R + r] = hqs[r];
    }
  }
}

// One thread per output row: per-row totals (sequential over hi).
__global__ void rowsum_kernel(PsiGeom g, Workspace ws) {
  int ho = blockIdx.x * blockDim.x + threadIdx.x;
  if (ho >= g.Hout) return;
  int len = 0, runs = 0, hrows = 0, ft = 0, rc[kMaxRad] = {0};
  for (int hi = 0; hi < g.Hin; ++hi) {
    size_t t = (size_t)ho * g.Hin + hi;
    int m = ws.mtab[t];
    if (m < 0) continue;
    len += run_len(m, g.Win);
    runs += 1;
    hrows += m + 1;  // pair steps delta = 0 .. m (m = W/2 includes the antipodal step)
    ft += g.K * ftab_len(m, g.Win);
    for (int r = 0; r < g.R; ++r) rc[r] += ws.ringcnt[t * g.R + r];
  }
  int32_t* o = ws.rowsum + (size_t)ho * (kRS + g.R);
  o[0] = len;
  o[1] = runs;
  o[2] = hrows;
  o[3] = ft;
  for (int r = 0; r < g.R; ++r) o[kRS + r] = rc[r];
}

struct PsiOut {
  int32_t *row_ptr, *idx, *csr_row_ptr, *csr_col, *run_ptr, *trun_ptr, *truns, *row_order;
  float *val, *csr_val, *hval;
  disco_run* runs;
  int32_t* ftab_off;
  uint16_t* ftab;
  int32_t* grp_ptr;
  disco_grp_ent* grp;
  uint16_t* gtab;
  uint16_t* ftab_h;  // the same tables rounded to fp16
  uint16_t* gtab_h;
  // element counts the plan sized the arrays for (extent checks of the
  // bounds-checked build)
  long long nnz, nnz_csr, nruns, nhval, nftab, ngrp_ent, ngtab;
};

__device__ __forceinline__ int ring_of(int kind, int k) { return kind == 1 ? k / 3 : k; }

// Single thread: prefix sums over output rows (and over (k, ho) for CSR).
__global__ void scan_kernel(PsiGeom g, Workspace ws, PsiOut p) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  int32_t e = 0, r = 0;
  p.row_ptr[0] = 0;
  p.run_ptr[0] = 0;
  for (int ho = 0; ho < g.Hout; ++ho) {
    const int32_t* o = ws.rowsum + (size_t)ho * (kRS + g.R);
    e += o[0];
    r += o[1];
    p.row_ptr[ho + 1] = e;
    p.run_ptr[ho + 1] = r;
  }
  int32_t c = 0;
  p.csr_row_ptr[0] = 0;
  for (int k = 0; k < g.K; ++k)
    for (int ho = 0; ho < g.Hout; ++ho) {
      c += ws.rowsum[(size_t)ho * (kRS + g.R) + kRS + ring_of(g.kind, k)];
      p.csr_row_ptr[k * g.Hout + ho + 1] = c;
    }
}

// One thread per output row: offsets of each run inside the global arrays,
// and the per-ring normalisers (summed over input rows in ascending order).
__global__ void offsets_kernel(PsiGeom g, Workspace ws, PsiOut p) {
  int ho = blockIdx.x * blockDim.x + threadIdx.x;
  if (ho >= g.Hout) return;
  int32_t off = 0, run = p.run_ptr[ho];
  // pair-weight rows: runs are numbered globally in (ho, hi) order, so the
  // hval offset of a run is the running total over all earlier runs.
  int32_t hoff = 0, foff = 0;
  for (int h2 = 0; h2 < ho; ++h2) {
    hoff += ws.rowsum[(size_t)h2 * (kRS + g.R) + 2];
    foff += ws.rowsum[(size_t)h2 * (kRS + g.R) + 3];
  }
  int32_t rc[kMaxRad] = {0};
  double nrm[kMaxRad] = {0};
  for (int hi = 0; hi < g.Hin; ++hi) {
    size_t t = (size_t)ho * g.Hin + hi;
    int m = ws.mtab[t];
    ws.off[t] = off;
    ws.runidx[t] = m >= 0 ? run : -1;
    ws.hofftab[t] = hoff;
    ws.ftofftab[t] = foff;
    for (int r = 0; r < g.R; ++r) ws.csroff[t * g.R + r] = rc[r];
    if (m < 0) continue;
    off += run_len(m, g.Win);
    run += 1;
    hoff += m + 1;
    foff += g.K * ftab_len(m, g.Win);
    for (int r = 0; r < g.R; ++r) {
      rc[r] += ws.ringcnt[t * g.R + r];
      nrm[r] = __dadd_rn(nrm[r], ws.hq[t * g.R + r]);
    }
  }
  for (int r = 0; r < g.R; ++r) ws.norm[(size_t)ho * g.R + r] = nrm[r];
}

// One block per output row; threads stride over input rows; each thread
// writes one whole run in neighbour order.
__global__ void fill_kernel(PsiGeom g, Workspace ws, PsiOut p) {
  int ho = blockIdx.x;
  double th_o = th_out(g, ho);
  double nrm[kMaxRad];
  for (int r = 0; r < g.R; ++r) nrm[r] = ws.norm[(size_t)ho * g.R + r];
  for (int hi = threadIdx.x; hi < g.Hin; hi += blockDim.x) {
    size_t t = (size_t)ho * g.Hin + hi;
    int m = ws.mtab[t];
    if (m < 0) continue;
    double th_i = th_in(g, hi);
    double q = q_in(g, hi);
    int W = g.Win, hr = half_ring(W);
    int len = run_len(m, W);
    bool full = (len == W);
    int dlo = full ? -hr : -m;
    int npair = full ? ((W % 2 == 0) ? hr - 1 : hr) : m;
    int anti = (full && W % 2 == 0) ? 1 : 0;
    int32_t e0 = p.row_ptr[ho] + ws.off[t];
    int32_t hoff = ws.hofftab[t];
    disco_run run;
    run.ho = ho;
    run.hi = hi;
    run.D = npair + anti;
    run.hoff = hoff;
    run.e0 = e0;
    run.len = len;
    run.npair = npair;
    run.anti = anti;
    if (DISCO_IN_BOUNDS(ws.runidx[t] >= 0 && ws.runidx[t] < p.nruns)) p.runs[ws.runidx[t]] = run;
    if (!DISCO_IN_BOUNDS(e0 >= 0 && (long long)e0 + len <= p.nnz)) continue;
    int32_t rpos[kMaxRad];
    for (int r = 0; r < g.R; ++r) rpos[r] = ws.csroff[t * g.R + r];
    for (int j = 0; j < len; ++j) {
      int delta = dlo + j;
      int wi = delta < 0 ? delta + W : delta;
      int64_t e = (int64_t)e0 + j;
      double h[kMaxRad], d, beta;
      bool st[kMaxRad];
      support_at(g, th_o, th_i, q, delta < 0 ? -delta : delta, h, st, &d, &beta);
      // bearing needs the signed offset
      geometry(th_o, th_i, delta, W, &d, &beta);
      p.idx[2 * e] = hi;
      p.idx[2 * e + 1] = wi;
      float vals[16];
      for (int k = 0; k < g.K; ++k) {
        int r = ring_of(g.kind, k), a = g.kind == 1 ? k % 3 : 0;
        double v = 0.0;
        if (st[r] && nrm[r] > 0.0) {
          double ang = 1.0;
          if (a != 0) ang = (d < kCoincident) ? 0.0 : (a == 1 ? cos(beta) : sin(beta));
          v = __ddiv_rn(__dmul_rn(__dmul_rn(h[r], ang), q), nrm[r]);
        }
        vals[k] = __double2float_rn(v);
        p.val[e * g.Kp + k] = vals[k];
        if (st[r]) {
          int32_t pos = p.csr_row_ptr[k * g.Hout + ho] + rpos[r];
          if (DISCO_IN_BOUNDS(pos >= 0 && pos < p.nnz_csr)) {
            p.csr_col[pos] = hi * W + wi;
            p.csr_val[pos] = vals[k];
          }
        }
      }
      for (int k = g.K; k < g.Kp; ++k) p.val[e * g.Kp + k] = 0.f;
      for (int r = 0; r < g.R; ++r)
        if (st[r]) rpos[r] += 1;
      // pair weights: delta = 0 .. npair, then the antipodal column
      int hrow = -1;
      float scale = 1.f;
      if (delta >= 0 && delta <= npair) {
        hrow = hoff + delta;
        if (delta == 0) scale = 0.5f;
      } else if (anti && delta == -hr) {
        hrow = hoff + npair + 1;
        scale = 0.5f;
      }
      if (hrow >= 0 && DISCO_IN_BOUNDS(hrow < p.nhval)) {
        for (int k = 0; k < g.K; ++k) p.hval[(int64_t)hrow * g.Kp + k] = vals[k] * scale;
        for (int k = g.K; k < g.Kp; ++k) p.hval[(int64_t)hrow * g.Kp + k] = 0.f;
      }
    }
  }
}

// bf16 tables of each run (forward and polyphase transpose), from val
__global__ void table_kernel(PsiGeom g, Workspace ws, PsiOut p) {
  const int ho = blockIdx.x;
  for (int hi = blockIdx.y; hi < g.Hin; hi += gridDim.y) {
    const size_t t = (size_t)ho * g.Hin + hi;
    const int m = ws.mtab[t];
    if (m < 0) continue;
    const int r = ws.runidx[t];
    const int e0 = p.row_ptr[ho] + ws.off[t];
    int dlo, dhi;
    run_extent(m, g.Win, &dlo, &dhi);
    const int tlf = ftab_len(m, g.Win);
    const int foff = ws.ftofftab[t];
    // (the whole block reads the same run and skips it alike)
    if (!DISCO_IN_BOUNDS(r >= 0 && r < p.nruns && foff >= 0 && (long long)foff + g.K * tlf <= p.nftab &&
                         e0 >= 0 && (long long)e0 + (dhi - dlo + 1) <= p.nnz))
      continue;
    if (threadIdx.x == 0) p.ftab_off[r] = foff;
    for (int i = threadIdx.x; i < g.K * tlf; i += blockDim.x) {
      const int k = i / tlf, x = i - k * tlf;
      const int d = dlo + x - 8;
      const float v = (d >= dlo && d <= dhi) ? p.val[(size_t)(e0 + d - dlo) * g.Kp + k] : 0.f;
      p.ftab[foff + i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
      p.ftab_h[foff + i] = __half_as_ushort(__float2half_rn(v));
    }
  }
}

__global__ void table_tail_kernel(PsiGeom g, Workspace ws, PsiOut p, int32_t nruns) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  int32_t f = 0;
  for (int ho = 0; ho < g.Hout; ++ho) f += ws.rowsum[(size_t)ho * (kRS + g.R) + 3];
  p.ftab_off[nruns] = f;
}

// ---- transpose tables by input-row group (see disco_psi.grp_ptr) --------

// Walks the output rows that input-row group z reads, calling
// f(ho, MW, KB, nch, r0, r1) with r0 .. r1 the group's rows (0 .. 7) that have
// support at ho.
template <typename F>
__device__ void for_group_rows(const PsiGeom& g, const Workspace& ws, int z, F f) {
  const int s = g.Win / g.Wout, TQ = grp_tq(s);
  const int h0 = z * kGrpRows, h1 = min(g.Hin, h0 + kGrpRows);
  for (int ho = 0; ho < g.Hout; ++ho) {
    int E = -1, r0 = kGrpRows, r1 = -1;
    for (int hi = h0; hi < h1; ++hi) {
      const int m = ws.mtab[(size_t)ho * g.Hin + hi];
      if (m >= 0) {
        E = max(E, run_halfwidth(m, g.Win, s));
        r0 = min(r0, hi - h0);
        r1 = hi - h0;
      }
    }
    if (E < 0) continue;
    const int MW = (E + 7) & ~7;
    const int KB = (TQ + 2 * MW + 15) / 16;
    f(ho, MW, KB, (KB + 3) / 4, r0, r1);
  }
}

// One thread per group: entries and table blocks.
__global__ void gcount_kernel(PsiGeom g, Workspace ws) {
  const int z = blockIdx.x * blockDim.x + threadIdx.x;
  if (z >= num_groups(g)) return;
  int ent = 0, blk = 0;
  for_group_rows(g, ws, z, [&](int, int, int, int nch, int, int) {
    ++ent;
    blk += g.K * nch;
  });
  ws.gcnt[2 * z] = ent;
  ws.gcnt[2 * z + 1] = blk;
}

__global__ void gscan_kernel(PsiGeom g, Workspace ws, PsiOut p) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  int32_t e = 0, b = 0;
  const int nz = num_groups(g);
  for (int z = 0; z < nz; ++z) {
    p.grp_ptr[z] = e;
    ws.gboff[z] = b;
    e += ws.gcnt[2 * z];
    b += ws.gcnt[2 * z + 1];
  }
  p.grp_ptr[nz] = e;
}

__global__ void gent_kernel(PsiGeom g, Workspace ws, PsiOut p) {
  const int z = blockIdx.x * blockDim.x + threadIdx.x;
  if (z >= num_groups(g)) return;
  const int blk = grp_block(g.Win / g.Wout);
  int e = p.grp_ptr[z], b = ws.gboff[z];
  for_group_rows(g, ws, z, [&](int ho, int MW, int KB, int nch, int r0, int r1) {
    disco_grp_ent en;
    en.ho = ho;
    en.off = b * blk;
    en.MW = (int16_t)MW;
    en.KB = (int16_t)KB;
    en.nch = (int16_t)nch;
    en.r0 = (int8_t)r0;
    en.r1 = (int8_t)r1;
    if (DISCO_IN_BOUNDS(e >= 0 && e < p.ngrp_ent)) p.grp[e] = en;
    ++e;
    b += g.K * nch;
  });
}

// One block per group: every element of the group's table blocks.
__global__ void gfill_kernel(PsiGeom g, Workspace ws, PsiOut p) {
  const int z = blockIdx.x;
  const int s = g.Win / g.Wout, TQ = grp_tq(s), CW = grp_cw(s), blk = grp_block(s);
  for (int j = p.grp_ptr[z]; j < p.grp_ptr[z + 1]; ++j) {
    if (!DISCO_IN_BOUNDS(j >= 0 && j < p.ngrp_ent)) break;
    const disco_grp_ent en = p.grp[j];
    const int n = g.K * en.nch * blk;
    if (!DISCO_IN_BOUNDS(en.off >= 0 && (long long)en.off + n <= p.ngtab && en.ho >= 0 && en.ho < g.Hout)) continue;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const int bi = i / blk, w = i - bi * blk;  // block (k, c), element (r, ph, y)
      const int k = bi / en.nch, c = bi - k * en.nch;
      const int r = w / (s * CW), ph = (w / CW) % s, y = w % CW;
      const int hi = z * kGrpRows + r;
      float v = 0.f;
      if (hi < g.Hin) {
        const size_t t = (size_t)en.ho * g.Hin + hi;
        const int m = ws.mtab[t];
        const int d = s * (en.MW + TQ - 1 - kGrpChunk * c - y) + ph;
        int dlo, dhi;
        run_extent(m, g.Win, &dlo, &dhi);
        if (m >= 0 && d >= dlo && d <= dhi) {
          const int e0 = p.row_ptr[en.ho] + ws.off[t];
          if (DISCO_IN_BOUNDS(e0 + d - dlo >= 0 && e0 + d - dlo < p.nnz)) v = p.val[(size_t)(e0 + d - dlo) * g.Kp + k];
        }
      }
      p.gtab[(size_t)en.off + i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
      p.gtab_h[(size_t)en.off + i] = __half_as_ushort(__float2half_rn(v));
    }
  }
}

// transposed run list: count per input row, scan, fill (ho ascending)
__global__ void tcount_kernel(PsiGeom g, Workspace ws) {
  int hi = blockIdx.x * blockDim.x + threadIdx.x;
  if (hi >= g.Hin) return;
  int c = 0;
  for (int ho = 0; ho < g.Hout; ++ho) c += ws.mtab[(size_t)ho * g.Hin + hi] >= 0;
  ws.tcount[hi] = c;
}

__global__ void tscan_kernel(PsiGeom g, Workspace ws, PsiOut p) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  int32_t c = 0;
  p.trun_ptr[0] = 0;
  for (int hi = 0; hi < g.Hin; ++hi) {
    c += ws.tcount[hi];
    p.trun_ptr[hi + 1] = c;
  }
}

__global__ void tfill_kernel(PsiGeom g, Workspace ws, PsiOut p) {
  int hi = blockIdx.x * blockDim.x + threadIdx.x;
  if (hi >= g.Hin) return;
  int32_t pos = p.trun_ptr[hi];
  for (int ho = 0; ho < g.Hout; ++ho) {
    int32_t r = ws.runidx[(size_t)ho * g.Hin + hi];
    if (r >= 0) {
      if (DISCO_IN_BOUNDS(pos >= 0 && pos < p.nruns)) p.truns[pos] = r;
      ++pos;
    }
  }
}

// launch order of output rows: descending union length, ties by row index
__global__ void order_kernel(PsiGeom g, Workspace ws, PsiOut p) {
  int ho = blockIdx.x * blockDim.x + threadIdx.x;
  if (ho >= g.Hout) return;
  int my = ws.rowsum[(size_t)ho * (kRS + g.R)];
  int rank = 0;
  for (int h2 = 0; h2 < g.Hout; ++h2) {
    int o = ws.rowsum[(size_t)h2 * (kRS + g.R)];
    rank += (o > my) || (o == my && h2 < ho);
  }
  if (DISCO_IN_BOUNDS(rank >= 0 && rank < g.Hout)) p.row_order[rank] = ho;
}

// The page's uniform K-packed form of the union layout; one block per output row.
__global__ void export_kpacked_kernel(const int32_t* row_ptr, const int32_t* idx, const float* val, int Kp,
                                      int nbr_pad, int64_t* pidx, float* pval, int64_t* pcount) {
  const int ho = blockIdx.x;
  const int e0 = row_ptr[ho];
  int n = row_ptr[ho + 1] - e0;
  if (!DISCO_IN_BOUNDS(n >= 0 && n <= nbr_pad)) n = 0;
  if (threadIdx.x == 0) pcount[ho] = n;
  const int64_t base = (int64_t)ho * nbr_pad;
  for (int j = threadIdx.x; j < nbr_pad; j += blockDim.x) {
    const bool in = j < n;
    pidx[(base + j) * 2] = in ? idx[(size_t)(e0 + j) * 2] : 0;
    pidx[(base + j) * 2 + 1] = in ? idx[(size_t)(e0 + j) * 2 + 1] : 0;
  }
  for (int64_t t = threadIdx.x; t < (int64_t)nbr_pad * Kp; t += blockDim.x) {
    const int j = (int)(t / Kp), k = (int)(t - (int64_t)j * Kp);
    pval[base * Kp + t] = j < n ? val[(size_t)(e0 + j) * Kp + k] : 0.f;
  }
}

int make_geom(const disco_grid* gi, const disco_grid* go, const disco_basis* b, PsiGeom* g) {
  if (!gi || !go || !b) return fail(DISCO_ERR_INVALID_ARG, "null grid or basis");
  if (gi->nlat < 2 || go->nlat < 2 || gi->nlon < 1 || go->nlon < 1)
    return fail(DISCO_ERR_INVALID_ARG, "grid too small (nlat >= 2, nlon >= 1)");
  if (gi->poles < 0 || gi->poles > 2 || go->poles < 0 || go->poles > 2)
    return fail(DISCO_ERR_INVALID_ARG, "grid poles must be 0 (midpoint), 1 (poles) or 2 (Legendre-Gauss)");
  if ((gi->poles == 1 && gi->nlat < 3) || (go->poles == 1 && go->nlat < 3))
    return fail(DISCO_ERR_INVALID_ARG, "pole grid needs nlat >= 3");
  if (gi->nlon % go->nlon != 0)
    return fail(DISCO_ERR_UNSUPPORTED, "W_in (%d) must be a multiple of W_out (%d)", gi->nlon, go->nlon);
  if (b->kind != 0 && b->kind != 1) return fail(DISCO_ERR_INVALID_ARG, "basis kind must be 0 or 1");
  if (b->n_radial < 1 || b->n_radial > kMaxRad)
    return fail(DISCO_ERR_UNSUPPORTED, "n_radial must be in [1, %d]", kMaxRad);
  if (!(b->cutoff > 0.0) || !(b->cutoff < kPi))
    return fail(DISCO_ERR_INVALID_ARG, "cutoff must be in (0, pi)");
  int K = b->kind == 1 ? 3 * b->n_radial : b->n_radial;
  if (K > 16) return fail(DISCO_ERR_UNSUPPORTED, "K = %d > 16", K);
  if ((int64_t)gi->nlat * gi->nlon >= (int64_t)1 << 30)
    return fail(DISCO_ERR_UNSUPPORTED, "input grid too large for int32 indices");
  g->Hin = gi->nlat;
  g->Win = gi->nlon;
  g->pin = gi->poles;
  g->Hout = go->nlat;
  g->Wout = go->nlon;
  g->pout = go->poles;
  g->kind = b->kind;
  g->R = b->n_radial;
  g->K = K;
  g->Kp = (K + 7) / 8 * 8;
  g->cutoff = b->cutoff;
  g->width = b->cutoff / (double)b->n_radial;
  g->lg = nullptr;
  return DISCO_OK;
}

size_t carve_psi(const disco_psi* psi, char* base, PsiOut* out) {
  int Hin = psi->grid_in.nlat, Hout = psi->grid_out.nlat;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + o : nullptr;
    o += align256(bytes);
    return p;
  };
  PsiOut p;
  p.row_ptr = (int32_t*)take((size_t)(Hout + 1) * 4);
  p.idx = (int32_t*)take((size_t)psi->nnz * 8);
  p.val = (float*)take((size_t)psi->nnz * psi->K_pad * 4);
  p.csr_row_ptr = (int32_t*)take(((size_t)psi->K * Hout + 1) * 4);
  p.csr_col = (int32_t*)take((size_t)psi->nnz_csr * 4);
  p.csr_val = (float*)take((size_t)psi->nnz_csr * 4);
  p.run_ptr = (int32_t*)take((size_t)(Hout + 1) * 4);
  p.runs = (disco_run*)take((size_t)psi->nruns * sizeof(disco_run));
  p.trun_ptr = (int32_t*)take((size_t)(Hin + 1) * 4);
  p.truns = (int32_t*)take((size_t)psi->nruns * 4);
  p.hval = (float*)take((size_t)psi->nhval * psi->K_pad * 4);
  p.row_order = (int32_t*)take((size_t)Hout * 4);
  p.ftab_off = (int32_t*)take((size_t)(psi->nruns + 1) * 4);
  p.ftab = (uint16_t*)take((size_t)psi->nftab * 2);
  p.grp_ptr = (int32_t*)take((size_t)(psi->ngrp + 1) * 4);
  p.grp = (disco_grp_ent*)take((size_t)psi->ngrp_ent * sizeof(disco_grp_ent));
  p.gtab = (uint16_t*)take((size_t)psi->ngtab * 2);
  p.ftab_h = (uint16_t*)take((size_t)psi->nftab * 2);
  p.gtab_h = (uint16_t*)take((size_t)psi->ngtab * 2);
  p.nnz = psi->nnz;
  p.nnz_csr = psi->nnz_csr;
  p.nruns = psi->nruns;
  p.nhval = psi->nhval;
  p.nftab = psi->nftab;
  p.ngrp_ent = psi->ngrp_ent;
  p.ngtab = psi->ngtab;
  if (out) *out = p;
  return o;
}

}  // namespace
// This unit's word of failed range checks (always 0 outside the bounds-checked build).
DISCO_BOUNDS_READER(psi_bounds)

}  // namespace disco

using namespace disco;

extern "C" int disco_psi_workspace_bytes(const disco_grid* grid_in, const disco_grid* grid_out,
                                         const disco_basis* basis, size_t* bytes) {
  PsiGeom g;
  int st = make_geom(grid_in, grid_out, basis, &g);
  if (st) return st;
  if (!bytes) return fail(DISCO_ERR_INVALID_ARG, "bytes is null");
  *bytes = carve_workspace(g, nullptr, nullptr);
  return DISCO_OK;
}

extern "C" int disco_psi_plan(const disco_grid* grid_in, const disco_grid* grid_out,
                              const disco_basis* basis, void* workspace, size_t workspace_bytes,
                              void* stream, disco_psi* psi) {
  disco::NvtxScope nvtx_scope("disco_psi_plan");
  PsiGeom g;
  int st = make_geom(grid_in, grid_out, basis, &g);
  if (st) return st;
  if (!psi) return fail(DISCO_ERR_INVALID_ARG, "psi is null");
  if ((st = check_device())) return st;
  size_t need = carve_workspace(g, nullptr, nullptr);
  if (!workspace || workspace_bytes < need)
    return fail(DISCO_ERR_WORKSPACE, "psi workspace needs %zu bytes", need);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(DISCO_ERR_ALIGNMENT, "psi workspace must be 256-byte aligned");
  if ((st = check_dev_ptr(workspace, "psi workspace"))) return st;
  Workspace ws;
  carve_workspace(g, (char*)workspace, &ws);
  g.lg = ws.lg;
  cudaStream_t s = (cudaStream_t)stream;
  if (g.pin == 2 || g.pout == 2) {
    lg_kernel<<<(g.Hin + g.Hout + 127) / 128, 128, 0, s>>>(g, ws);
    if ((st = check_launch("psi Legendre-Gauss nodes"))) return st;
  }
  count_kernel<<<g.Hout, 128, 0, s>>>(g, ws);
  if ((st = check_launch("psi count"))) return st;
  rowsum_kernel<<<(g.Hout + 127) / 128, 128, 0, s>>>(g, ws);
  if ((st = check_launch("psi rowsum"))) return st;
  std::vector<int32_t> rs((size_t)g.Hout * (kRS + g.R));
  cudaError_t ce = cudaMemcpyAsync(rs.data(), ws.rowsum, rs.size() * 4, cudaMemcpyDeviceToHost, s);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(s);
  if (ce != cudaSuccess) return fail(DISCO_ERR_CUDA, "psi plan copy: %s", cudaGetErrorString(ce));
  int64_t nnz = 0, nruns = 0, nhval = 0, nnz_csr = 0, nftab = 0;
  int32_t max_row = 0;
  for (int ho = 0; ho < g.Hout; ++ho) {
    const int32_t* o = &rs[(size_t)ho * (kRS + g.R)];
    nnz += o[0];
    nruns += o[1];
    nhval += o[2];
    nftab += o[3];
    if (o[0] > max_row) max_row = o[0];
    for (int k = 0; k < g.K; ++k) nnz_csr += o[kRS + (g.kind == 1 ? k / 3 : k)];
  }
  // transpose tables by input-row group (s <= 2 only)
  const int sdec = g.Win / g.Wout;
  const int nz = sdec <= 2 ? num_groups(g) : 0;
  int64_t ngrp_ent = 0, ngtab = 0;
  int32_t grp_max = 0;
  if (nz > 0) {
    gcount_kernel<<<(nz + 127) / 128, 128, 0, s>>>(g, ws);
    if ((st = check_launch("psi group count"))) return st;
    std::vector<int32_t> gc((size_t)nz * 2);
    ce = cudaMemcpyAsync(gc.data(), ws.gcnt, gc.size() * 4, cudaMemcpyDeviceToHost, s);
    if (ce == cudaSuccess) ce = cudaStreamSynchronize(s);
    if (ce != cudaSuccess) return fail(DISCO_ERR_CUDA, "psi plan copy: %s", cudaGetErrorString(ce));
    for (int z = 0; z < nz; ++z) {
      ngrp_ent += gc[2 * z];
      ngtab += (int64_t)gc[2 * z + 1] * grp_block(sdec);
      if (gc[2 * z] > grp_max) grp_max = gc[2 * z];
    }
  }
  if (nnz >= ((int64_t)1 << 31) / 16 || nnz_csr >= ((int64_t)1 << 31) || nftab >= ((int64_t)1 << 31) ||
      ngtab >= ((int64_t)1 << 31))
    return fail(DISCO_ERR_UNSUPPORTED, "psi too large for int32 offsets");
  memset(psi, 0, sizeof(*psi));
  psi->grid_in = *grid_in;
  psi->grid_out = *grid_out;
  psi->basis = *basis;
  psi->K = g.K;
  psi->K_pad = g.Kp;
  psi->s = g.Win / g.Wout;
  psi->max_row = max_row;
  psi->nnz = nnz;
  psi->nnz_csr = nnz_csr;
  psi->nruns = nruns;
  psi->nhval = nhval;
  psi->nftab = nftab;
  psi->ngrp = nz;
  psi->grp_max = grp_max;
  psi->ngrp_ent = ngrp_ent;
  psi->ngtab = ngtab;
  psi->bytes = carve_psi(psi, nullptr, nullptr);
  return DISCO_OK;
}

extern "C" int disco_build_psi_kpacked(disco_psi* psi, void* buffer, size_t bytes, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  disco::NvtxScope nvtx_scope("disco_build_psi_kpacked");
  if (!psi) return fail(DISCO_ERR_INVALID_ARG, "psi is null");
  PsiGeom g;
  int st = make_geom(&psi->grid_in, &psi->grid_out, &psi->basis, &g);
  if (st) return st;
  if ((st = check_device())) return st;
  if (psi->K != g.K || psi->K_pad != g.Kp || psi->bytes != carve_psi(psi, nullptr, nullptr))
    return fail(DISCO_ERR_INVALID_ARG, "psi sizes do not match its grids (call disco_psi_plan)");
  if (!buffer || bytes < psi->bytes)
    return fail(DISCO_ERR_INVALID_ARG, "psi buffer needs %zu bytes", psi->bytes);
  if (reinterpret_cast<uintptr_t>(buffer) & 255u)
    return fail(DISCO_ERR_ALIGNMENT, "psi buffer must be 256-byte aligned");
  size_t need = carve_workspace(g, nullptr, nullptr);
  if (!workspace || workspace_bytes < need)
    return fail(DISCO_ERR_WORKSPACE, "psi workspace needs %zu bytes", need);
  if ((st = check_dev_ptr(buffer, "psi buffer")) || (st = check_dev_ptr(workspace, "psi workspace"))) return st;
  Workspace ws;
  carve_workspace(g, (char*)workspace, &ws);
  g.lg = ws.lg;  // Legendre-Gauss tables left in the workspace by disco_psi_plan
  PsiOut p;
  carve_psi(psi, (char*)buffer, &p);
  cudaStream_t s = (cudaStream_t)stream;
  int tb = 128;
  scan_kernel<<<1, 1, 0, s>>>(g, ws, p);
  if ((st = check_launch("psi scan"))) return st;
  offsets_kernel<<<(g.Hout + tb - 1) / tb, tb, 0, s>>>(g, ws, p);
  if ((st = check_launch("psi offsets"))) return st;
  fill_kernel<<<g.Hout, 64, 0, s>>>(g, ws, p);
  if ((st = check_launch("psi fill"))) return st;
  table_kernel<<<dim3(g.Hout, 32), 128, 0, s>>>(g, ws, p);
  if ((st = check_launch("psi tables"))) return st;
  table_tail_kernel<<<1, 1, 0, s>>>(g, ws, p, (int32_t)psi->nruns);
  if ((st = check_launch("psi table tail"))) return st;
  tcount_kernel<<<(g.Hin + tb - 1) / tb, tb, 0, s>>>(g, ws);
  if ((st = check_launch("psi tcount"))) return st;
  tscan_kernel<<<1, 1, 0, s>>>(g, ws, p);
  if ((st = check_launch("psi tscan"))) return st;
  tfill_kernel<<<(g.Hin + tb - 1) / tb, tb, 0, s>>>(g, ws, p);
  if ((st = check_launch("psi tfill"))) return st;
  order_kernel<<<(g.Hout + tb - 1) / tb, tb, 0, s>>>(g, ws, p);
  if ((st = check_launch("psi order"))) return st;
  if (psi->ngrp > 0) {
    // the group counts were left in the workspace by disco_psi_plan
    gscan_kernel<<<1, 1, 0, s>>>(g, ws, p);
    if ((st = check_launch("psi group scan"))) return st;
    gent_kernel<<<(psi->ngrp + 127) / 128, 128, 0, s>>>(g, ws, p);
    if ((st = check_launch("psi group entries"))) return st;
    gfill_kernel<<<psi->ngrp, 256, 0, s>>>(g, ws, p);
    if ((st = check_launch("psi group tables"))) return st;
  }
  psi->row_ptr = p.row_ptr;
  psi->idx = p.idx;
  psi->val = p.val;
  psi->csr_row_ptr = p.csr_row_ptr;
  psi->csr_col = p.csr_col;
  psi->csr_val = p.csr_val;
  psi->run_ptr = p.run_ptr;
  psi->runs = p.runs;
  psi->trun_ptr = p.trun_ptr;
  psi->truns = p.truns;
  psi->hval = p.hval;
  psi->row_order = p.row_order;
  psi->ftab_off = p.ftab_off;
  psi->ftab = p.ftab;
  psi->grp_ptr = p.grp_ptr;
  psi->grp = p.grp;
  psi->gtab = p.gtab;
  psi->ftab_h = p.ftab_h;
  psi->gtab_h = p.gtab_h;
  return DISCO_OK;
}

extern "C" int disco_psi_export_kpacked(const disco_psi* psi, int64_t* pack_idx, float* pack_val,
                                        int64_t* pack_count, int32_t nbr_pad, void* stream) {
  disco::NvtxScope nvtx_scope("disco_psi_export_kpacked");
  int st = check_psi(psi);
  if (st) return st;
  if ((st = check_device())) return st;
  if (!pack_idx || !pack_val || !pack_count) return fail(DISCO_ERR_INVALID_ARG, "null output pointer");
  if ((reinterpret_cast<uintptr_t>(pack_idx) & 7u) || (reinterpret_cast<uintptr_t>(pack_count) & 7u) ||
      (reinterpret_cast<uintptr_t>(pack_val) & 3u))
    return fail(DISCO_ERR_ALIGNMENT, "outputs must be aligned to their element size");
  if (nbr_pad < 1 || nbr_pad < psi->max_row)
    return fail(DISCO_ERR_INVALID_ARG, "nbr_pad (%d) must be >= max_row (%d)", nbr_pad, psi->max_row);
  if ((st = check_dev_ptr(pack_idx, "pack_idx")) || (st = check_dev_ptr(pack_val, "pack_val")) ||
      (st = check_dev_ptr(pack_count, "pack_count")))
    return st;
  export_kpacked_kernel<<<psi->grid_out.nlat, 256, 0, (cudaStream_t)stream>>>(
      psi->row_ptr, psi->idx, psi->val, psi->K_pad, nbr_pad, pack_idx, pack_val, pack_count);
  return check_launch("psi kpacked export");
}
