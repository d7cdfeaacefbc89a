/*
 * disco_oracle.c -- plain, slow, fp64 CPU oracle for the DISCO
 * (discrete-continuous) convolution on the sphere.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file.  It is used by the tests, by the smoke check and by the
 * CPU-baseline leg of the benchmark, and by nothing else.  It shares no code,
 * header, table or constant with the CUDA path.
 *
 * What it computes (DISCO Kernel Development Guide, torch-harmonics,
 * §Architecture snapshot: the sparse contraction of the input grid into
 * X[B,C,K,H,W] and its transpose back to the input grid; §kpacked layout for
 * the neighbour-list form).  The page names the operations but does not give the
 * basis, quadrature or normalisation; the definitions below are the plainest
 * readings of the workload text and every one of them is listed with its
 * reason in the design notes:
 *
 *   grids      midpoint:  theta_i = (i + 1/2) pi / H
 *              poles:     theta_i = i pi / (H - 1)   (theta_{H-1} = pi exactly)
 *              Legendre-Gauss: theta_i = arccos x_i, x_0 > x_1 > ... the H
 *                         roots of the Legendre polynomial P_H (north to
 *                         south), found by Newton's method on the three-term
 *                         recurrence
 *              longitude: phi_j   = 2 pi j / W
 *   distance   haversine great-circle distance between the output point
 *              (theta_o, phi = 0) and the input point (theta_i, dphi),
 *              dphi = 2 pi delta / W_in for the signed column offset delta
 *   hats       R radial hats of width D = cutoff / R centred at r D:
 *              h_r(d) = max(0, 1 - |d - r D| / D)
 *   bearing    beta = atan2(sin dphi sin th_i,
 *                           sin th_o cos th_i - cos th_o sin th_i cos dphi),
 *              0 = north (towards smaller colatitude), pi/2 = east
 *   basis      isotropic:   k = r,          A = 1
 *              anisotropic: k = 3 r + a,    A_0 = 1, A_1 = cos beta,
 *                                           A_2 = sin beta (0 when d < 1e-12)
 *              indicator:   K = 1, psi = 1 on d < cutoff (no quadrature, no
 *                           normalisation; closed-form test basis only)
 *   quadrature q_i = sin theta_i, exactly 0 on the pole rows of a pole grid;
 *              Legendre-Gauss: the Gauss-Legendre weight
 *              w_i = 2 / ((1 - x_i^2) P_H'(x_i)^2), which carries the sin
 *              theta d theta of the area element
 *   support    entry (r, hi, wi) is structural iff h_r(d) > 1e-9 and q_i > 0
 *   normaliser N(r, ho) = sum over the structural entries of ring r of h_r q_i
 *   value      psi[k, ho, hi, wi] = h_r(d) A_a(beta) q_i / N(r, ho)
 *
 *   forward    X[b,c,k,ho,wo] = sum_{(hi,wi) in row (k,ho)}
 *                                 psi[k,ho,hi,wi] x[b,c,hi,(wi + wo s) mod W_in]
 *   transpose  gx = psi^T G: the adjoint of the forward map
 *   einsum     y[b,o,ho,wo] = sum_{c,k} W[o,c,k] X[b,c,k,ho,wo]
 *   input grad dX = sum_o W[o,c,k] dy[b,o,ho,wo];  gx = psi^T dX
 *
 * Alongside every output the oracle returns S = sum of |elementary terms|,
 * the scale of the error bound the tests use.
 *
 * Neighbour order inside a row: hi ascending, then the signed column offset
 * delta = ((wi + floor(W/2)) mod W) - floor(W/2) ascending.  CSR rows are
 * numbered k * H_out + ho, columns are hi * W_in + wi.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no contraction of
 * a*b+c into fma, so x86 and Arm hosts give the same bits).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_PI 3.14159265358979323846
#define OR_TAU_SUPPORT 1e-9
#define OR_D_COINCIDENT 1e-12

enum { OR_ISO = 0, OR_ANISO = 1, OR_INDICATOR = 2 };

typedef struct {
  int32_t nlat, nlon, poles;
} or_grid;

/* ---------------------------------------------------------------- grids -- */

/* Gauss-Legendre node x_i (descending in i) and weight of order n: Newton's
   method from the standard first guess cos(pi (i + 3/4) / (n + 1/2)), with
   P_n and P_n' from the three-term recurrence. */
void oracle_gauss_node(int32_t n, int32_t i, double* x_out, double* w_out) {
  double x = cos(OR_PI * ((double)i + 0.75) / ((double)n + 0.5));
  double dp = 1.0;
  for (int it = 0; it < 100; ++it) {
    double p0 = 1.0, p1 = x;
    for (int32_t j = 1; j < n; ++j) {
      double p2 = ((2.0 * j + 1.0) * x * p1 - (double)j * p0) / ((double)j + 1.0);
      p0 = p1;
      p1 = p2;
    }
    dp = (double)n * (x * p1 - p0) / -((1.0 - x) * (1.0 + x)); /* P_n'(x), p0 = P_{n-1} */
    double dx = p1 / dp;
    x -= dx;
    if (fabs(dx) <= 1e-15) break; /* quadratic convergence: x is now within an ulp or two */
  }
  { /* derivative at the converged node */
    double p0 = 1.0, p1 = x;
    for (int32_t j = 1; j < n; ++j) {
      double p2 = ((2.0 * j + 1.0) * x * p1 - (double)j * p0) / ((double)j + 1.0);
      p0 = p1;
      p1 = p2;
    }
    dp = (double)n * (x * p1 - p0) / -((1.0 - x) * (1.0 + x));
  }
  *x_out = x;
  *w_out = 2.0 / ((1.0 - x) * (1.0 + x) * dp * dp);
}

/* Gauss-Legendre colatitudes and weights of one order, computed once and kept
   (a few orders at a time; the oracle calls these per row in its loops). */
typedef struct { int32_t n; double* th; double* w; } or_gauss;
static or_gauss or_gauss_cache[8];
static const or_gauss* or_gauss_table(int32_t n) {
  const or_gauss* r = NULL;
#pragma omp critical(or_gauss_lock)
  {
    for (int c = 0; c < 8 && !r; ++c)
      if (or_gauss_cache[c].n == n && or_gauss_cache[c].th) r = &or_gauss_cache[c];
    if (!r) {
      int slot = 0;
      while (slot < 8 && or_gauss_cache[slot].th) ++slot;
      if (slot == 8) { /* full: reuse slot 0 */
        free(or_gauss_cache[0].th);
        free(or_gauss_cache[0].w);
        or_gauss_cache[0].th = NULL;
        slot = 0;
      }
      double* th = (double*)malloc(sizeof(double) * (size_t)n);
      double* w = (double*)malloc(sizeof(double) * (size_t)n);
      for (int32_t i = 0; i < n; ++i) {
        double x;
        oracle_gauss_node(n, i, &x, &w[i]);
        th[i] = acos(x);
      }
      or_gauss_cache[slot].n = n;
      or_gauss_cache[slot].w = w;
      or_gauss_cache[slot].th = th;
      r = &or_gauss_cache[slot];
    }
  }
  return r;
}

double oracle_colat(int32_t nlat, int32_t poles, int32_t i) {
  if (poles == 2) return or_gauss_table(nlat)->th[i];
  if (poles) {
    if (i == nlat - 1) return OR_PI;
    return (double)i * OR_PI / (double)(nlat - 1);
  }
  return ((double)i + 0.5) * OR_PI / (double)nlat;
}

double oracle_quad(int32_t nlat, int32_t poles, int32_t i) {
  if (poles == 2) return or_gauss_table(nlat)->w[i];
  if (poles && (i == 0 || i == nlat - 1)) return 0.0;
  return sin(oracle_colat(nlat, poles, i));
}

/* great-circle distance and bearing from (th_o, 0) to (th_i, 2 pi delta / W) */
void oracle_geometry(double th_o, double th_i, int32_t delta, int32_t W,
                     double* d, double* beta) {
  int32_t ad = delta < 0 ? -delta : delta;
  double half = OR_PI * (double)ad / (double)W; /* |dphi| / 2 */
  double s1 = sin(0.5 * (th_i - th_o));
  double s2 = sin(half);
  double hav = s1 * s1 + sin(th_o) * sin(th_i) * (s2 * s2);
  if (hav > 1.0) hav = 1.0;
  *d = 2.0 * asin(sqrt(hav));
  double sdp = sin(2.0 * half);
  double cdp = cos(2.0 * half);
  if (delta < 0) sdp = -sdp;
  *beta = atan2(sdp * sin(th_i),
                sin(th_o) * cos(th_i) - cos(th_o) * sin(th_i) * cdp);
}

double oracle_hat(double d, int32_t r, double width) {
  double v = 1.0 - fabs(d - (double)r * width) / width;
  return v > 0.0 ? v : 0.0;
}

int32_t oracle_basis_K(int32_t kind, int32_t nrad) {
  if (kind == OR_ISO) return nrad;
  if (kind == OR_ANISO) return 3 * nrad;
  if (kind == OR_INDICATOR) return 1;
  return -1;
}

/* ------------------------------------------------------------ psi build -- */

/* One candidate neighbour of an output row, before normalisation. */
typedef struct {
  int32_t hi, wi;
  double h[8];   /* ring values h_r(d), or 1 for the indicator basis */
  int32_t st[8]; /* ring r structural */
  double q;      /* quadrature weight of the input row */
  double beta, d;
} or_cand;

/* Collect the union neighbour list of output row ho in neighbour order.
   Returns the count; fills *out (malloc'ed) when out != NULL. */
static int64_t or_row_candidates(const or_grid* gin, const or_grid* gout,
                                 int32_t kind, int32_t nrad, double cutoff,
                                 int32_t ho, or_cand** out) {
  double th_o = oracle_colat(gout->nlat, gout->poles, ho);
  double width = cutoff / (double)nrad;
  int64_t cap = 64, n = 0;
  or_cand* list = out ? (or_cand*)malloc(sizeof(or_cand) * cap) : NULL;
  int32_t W = gin->nlon;
  int32_t h = W / 2;
  for (int32_t hi = 0; hi < gin->nlat; ++hi) {
    double th_i = oracle_colat(gin->nlat, gin->poles, hi);
    /* d >= |th_i - th_o| on the sphere, so rows further than the cutoff in
       colatitude hold no neighbour (a slack of 1e-9 keeps rounding safe). */
    if (fabs(th_i - th_o) > cutoff + 1e-9) continue;
    double q = oracle_quad(gin->nlat, gin->poles, hi);
    for (int32_t delta = -h; delta < W - h; ++delta) {
      int32_t wi = delta < 0 ? delta + W : delta;
      or_cand c;
      memset(&c, 0, sizeof c);
      c.hi = hi;
      c.wi = wi;
      c.q = q;
      oracle_geometry(th_o, th_i, delta, W, &c.d, &c.beta);
      int any = 0;
      if (kind == OR_INDICATOR) {
        c.h[0] = 1.0;
        c.st[0] = (1.0 - c.d / cutoff) > OR_TAU_SUPPORT;
        any = c.st[0];
      } else {
        for (int32_t r = 0; r < nrad; ++r) {
          c.h[r] = oracle_hat(c.d, r, width);
          c.st[r] = (c.h[r] > OR_TAU_SUPPORT) && (q > 0.0);
          any |= c.st[r];
        }
      }
      if (!any) continue;
      if (list) {
        if (n == cap) {
          cap *= 2;
          list = (or_cand*)realloc(list, sizeof(or_cand) * cap);
        }
        list[n] = c;
      }
      ++n;
    }
  }
  if (out) *out = list;
  return n;
}

/* ring index and angular factor of basis function k at one candidate */
static void or_basis_k(int32_t kind, int32_t k, const or_cand* c, int32_t* ring,
                       double* ang) {
  if (kind == OR_ANISO) {
    int32_t r = k / 3, a = k % 3;
    *ring = r;
    if (a == 0) *ang = 1.0;
    else if (c->d < OR_D_COINCIDENT) *ang = 0.0;
    else *ang = (a == 1) ? cos(c->beta) : sin(c->beta);
  } else {
    *ring = k;
    *ang = 1.0;
  }
}

/* Sizes: union neighbour count and CSR non-zero count over all (k, ho). */
int oracle_psi_count(int32_t in_nlat, int32_t in_nlon, int32_t in_poles,
                     int32_t out_nlat, int32_t out_nlon, int32_t out_poles,
                     int32_t kind, int32_t nrad, double cutoff, int64_t* nnz,
                     int64_t* nnz_csr) {
  or_grid gin = {in_nlat, in_nlon, in_poles}, gout = {out_nlat, out_nlon, out_poles};
  int32_t K = oracle_basis_K(kind, nrad);
  if (K <= 0 || nrad > 8) return -1;
  int64_t tot = 0, tot_csr = 0;
  for (int32_t ho = 0; ho < out_nlat; ++ho) {
    or_cand* list = NULL;
    int64_t n = or_row_candidates(&gin, &gout, kind, nrad, cutoff, ho, &list);
    tot += n;
    for (int32_t k = 0; k < K; ++k) {
      for (int64_t e = 0; e < n; ++e) {
        int32_t ring;
        double ang;
        or_basis_k(kind, k, &list[e], &ring, &ang);
        if (list[e].st[ring]) ++tot_csr;
      }
    }
    free(list);
  }
  *nnz = tot;
  *nnz_csr = tot_csr;
  return 0;
}

/* Fill the union (kpacked) layout and the CSR layout.
   row_ptr[Hout+1], idx[nnz*2] = (hi, wi), val[nnz*K],
   csr_row_ptr[K*Hout+1], csr_col[nnz_csr] = hi*Win+wi, csr_val[nnz_csr]. */
int oracle_psi_fill(int32_t in_nlat, int32_t in_nlon, int32_t in_poles,
                    int32_t out_nlat, int32_t out_nlon, int32_t out_poles,
                    int32_t kind, int32_t nrad, double cutoff, int64_t* row_ptr,
                    int32_t* idx, double* val, int64_t* csr_row_ptr,
                    int32_t* csr_col, double* csr_val) {
  or_grid gin = {in_nlat, in_nlon, in_poles}, gout = {out_nlat, out_nlon, out_poles};
  int32_t K = oracle_basis_K(kind, nrad);
  if (K <= 0 || nrad > 8) return -1;
  int32_t Hout = out_nlat;
  /* pass 1: union rows */
  or_cand** lists = (or_cand**)calloc((size_t)Hout, sizeof(or_cand*));
  int64_t* counts = (int64_t*)calloc((size_t)Hout, sizeof(int64_t));
  for (int32_t ho = 0; ho < Hout; ++ho)
    counts[ho] = or_row_candidates(&gin, &gout, kind, nrad, cutoff, ho, &lists[ho]);
  row_ptr[0] = 0;
  for (int32_t ho = 0; ho < Hout; ++ho) row_ptr[ho + 1] = row_ptr[ho] + counts[ho];

  /* pass 2: normalisers and values, union layout */
  for (int32_t ho = 0; ho < Hout; ++ho) {
    or_cand* list = lists[ho];
    int64_t n = counts[ho];
    double norm[8] = {0};
    if (kind != OR_INDICATOR) {
      for (int32_t r = 0; r < nrad; ++r) {
        double acc = 0.0;
        for (int64_t e = 0; e < n; ++e)
          if (list[e].st[r]) acc += list[e].h[r] * list[e].q;
        norm[r] = acc;
      }
    }
    for (int64_t e = 0; e < n; ++e) {
      int64_t g = row_ptr[ho] + e;
      idx[2 * g + 0] = list[e].hi;
      idx[2 * g + 1] = list[e].wi;
      for (int32_t k = 0; k < K; ++k) {
        int32_t ring;
        double ang, v = 0.0;
        or_basis_k(kind, k, &list[e], &ring, &ang);
        if (list[e].st[ring]) {
          if (kind == OR_INDICATOR) v = 1.0;
          else if (norm[ring] > 0.0) v = list[e].h[ring] * ang * list[e].q / norm[ring];
        }
        val[g * K + k] = v;
      }
    }
  }

  /* pass 3: CSR rows (k, ho), columns in the same neighbour order */
  int64_t pos = 0;
  csr_row_ptr[0] = 0;
  for (int32_t k = 0; k < K; ++k) {
    for (int32_t ho = 0; ho < Hout; ++ho) {
      or_cand* list = lists[ho];
      for (int64_t e = 0; e < counts[ho]; ++e) {
        int32_t ring;
        double ang;
        or_basis_k(kind, k, &list[e], &ring, &ang);
        if (!list[e].st[ring]) continue;
        int64_t g = row_ptr[ho] + e;
        csr_col[pos] = list[e].hi * in_nlon + list[e].wi;
        csr_val[pos] = val[g * K + k];
        ++pos;
      }
      csr_row_ptr[(int64_t)k * Hout + ho + 1] = pos;
    }
  }
  for (int32_t ho = 0; ho < Hout; ++ho) free(lists[ho]);
  free(lists);
  free(counts);
  return 0;
}

/* ------------------------------------------------------- contractions -- */

/* Forward contraction on the CSR layout.  x[BC, Hin, Win] -> X[BC, K, Hout, Wout].
   S = sum |psi| * xabs (xabs = |x| when NULL). */
void oracle_fwd(const int64_t* csr_row_ptr, const int32_t* csr_col,
                const double* csr_val, int32_t K, int32_t Hin, int32_t Win,
                int32_t Hout, int32_t Wout, int64_t BC, const double* x,
                const double* xabs, double* X, double* S) {
  int32_t s = Win / Wout;
  int64_t in_plane = (int64_t)Hin * Win;
  int64_t out_plane = (int64_t)K * Hout * Wout;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bc = 0; bc < BC; ++bc) {
    const double* xp = x + bc * in_plane;
    const double* ap = xabs ? xabs + bc * in_plane : NULL;
    for (int32_t k = 0; k < K; ++k)
      for (int32_t ho = 0; ho < Hout; ++ho) {
        int64_t row = (int64_t)k * Hout + ho;
        for (int32_t wo = 0; wo < Wout; ++wo) {
          double acc = 0.0, sab = 0.0;
          for (int64_t e = csr_row_ptr[row]; e < csr_row_ptr[row + 1]; ++e) {
            int32_t hi = csr_col[e] / Win, wi = csr_col[e] % Win;
            int64_t col = (int64_t)hi * Win + (wi + (int64_t)wo * s) % Win;
            double t = csr_val[e] * xp[col];
            acc += t;
            sab += ap ? fabs(csr_val[e]) * ap[col] : fabs(t);
          }
          int64_t o = bc * out_plane + row * Wout + wo;
          X[o] = acc;
          if (S) S[o] = sab;
        }
      }
  }
}

/* Transpose contraction: gx = psi^T G, written as the plain scatter of every
   term of the forward map onto the input it came from.
   G[BC, K, Hout, Wout] -> gx[BC, Hin, Win];  S = |psi|^T Gabs (|G| when NULL). */
void oracle_bwd(const int64_t* csr_row_ptr, const int32_t* csr_col,
                const double* csr_val, int32_t K, int32_t Hin, int32_t Win,
                int32_t Hout, int32_t Wout, int64_t BC, const double* G,
                const double* Gabs, double* gx, double* S) {
  int32_t s = Win / Wout;
  int64_t in_plane = (int64_t)Hin * Win;
  int64_t out_plane = (int64_t)K * Hout * Wout;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bc = 0; bc < BC; ++bc) {
    double* gp = gx + bc * in_plane;
    double* sp = S ? S + bc * in_plane : NULL;
    for (int64_t i = 0; i < in_plane; ++i) {
      gp[i] = 0.0;
      if (sp) sp[i] = 0.0;
    }
    for (int32_t k = 0; k < K; ++k)
      for (int32_t ho = 0; ho < Hout; ++ho) {
        int64_t row = (int64_t)k * Hout + ho;
        for (int32_t wo = 0; wo < Wout; ++wo) {
          int64_t o = bc * out_plane + row * Wout + wo;
          double g = G[o];
          double ga = Gabs ? Gabs[o] : fabs(g);
          for (int64_t e = csr_row_ptr[row]; e < csr_row_ptr[row + 1]; ++e) {
            int32_t hi = csr_col[e] / Win, wi = csr_col[e] % Win;
            int64_t col = (int64_t)hi * Win + (wi + (int64_t)wo * s) % Win;
            gp[col] += csr_val[e] * g;
            if (sp) sp[col] += fabs(csr_val[e]) * ga;
          }
        }
      }
  }
}

/* Channel/basis einsum y[b,o,p] = sum_{c,k} W[o,c,k] X[b,c,k,p]
   (p = ho*Wout + wo);  Sy = sum |W| * SX. */
void oracle_einsum(const double* W, int32_t Cout, int32_t Cin, int32_t K,
                   int64_t P, int32_t B, const double* X, const double* SX,
                   double* y, double* Sy) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int32_t b = 0; b < B; ++b)
    for (int32_t o = 0; o < Cout; ++o) {
      double* yp = y + ((int64_t)b * Cout + o) * P;
      double* sp = Sy ? Sy + ((int64_t)b * Cout + o) * P : NULL;
      for (int64_t p = 0; p < P; ++p) {
        yp[p] = 0.0;
        if (sp) sp[p] = 0.0;
      }
      for (int32_t c = 0; c < Cin; ++c)
        for (int32_t k = 0; k < K; ++k) {
          double w = W[((int64_t)o * Cin + c) * K + k];
          const double* xp = X + (((int64_t)b * Cin + c) * K + k) * P;
          const double* xs = SX ? SX + (((int64_t)b * Cin + c) * K + k) * P : NULL;
          for (int64_t p = 0; p < P; ++p) {
            yp[p] += w * xp[p];
            if (sp) sp[p] += fabs(w) * xs[p];
          }
        }
    }
}

/* Adjoint einsum dX[b,c,k,p] = sum_o W[o,c,k] dy[b,o,p];  SdX = sum_o |W dy|. */
void oracle_einsum_t(const double* W, int32_t Cout, int32_t Cin, int32_t K,
                     int64_t P, int32_t B, const double* dy, double* dX,
                     double* SdX) {
#pragma omp parallel for collapse(3) schedule(static)
  for (int32_t b = 0; b < B; ++b)
    for (int32_t c = 0; c < Cin; ++c)
      for (int32_t k = 0; k < K; ++k) {
        double* xp = dX + (((int64_t)b * Cin + c) * K + k) * P;
        double* sp = SdX ? SdX + (((int64_t)b * Cin + c) * K + k) * P : NULL;
        for (int64_t p = 0; p < P; ++p) {
          xp[p] = 0.0;
          if (sp) sp[p] = 0.0;
        }
        for (int32_t o = 0; o < Cout; ++o) {
          double w = W[((int64_t)o * Cin + c) * K + k];
          const double* dp = dy + ((int64_t)b * Cout + o) * P;
          for (int64_t p = 0; p < P; ++p) {
            xp[p] += w * dp[p];
            if (sp) sp[p] += fabs(w * dp[p]);
          }
        }
      }
}

/* Weight gradient of the fused forward (the einsum's other adjoint):
   dW[o,c,k] = sum_b sum_p dy[b,o,p] X[b,c,k,p];  SdW = sum |dy| SX.
   X is the forward contraction of x, SX its sum of |terms|. */
void oracle_einsum_w(const double* dy, const double* X, const double* SX, int32_t Cout,
                     int32_t Cin, int32_t K, int64_t P, int32_t B, double* dW, double* SdW) {
#pragma omp parallel for collapse(3) schedule(static)
  for (int32_t o = 0; o < Cout; ++o)
    for (int32_t c = 0; c < Cin; ++c)
      for (int32_t k = 0; k < K; ++k) {
        double acc = 0.0, sacc = 0.0;
        for (int32_t b = 0; b < B; ++b) {
          const double* dp = dy + ((int64_t)b * Cout + o) * P;
          const double* xp = X + (((int64_t)b * Cin + c) * K + k) * P;
          const double* xs = SX ? SX + (((int64_t)b * Cin + c) * K + k) * P : NULL;
          for (int64_t p = 0; p < P; ++p) {
            acc += dp[p] * xp[p];
            sacc += fabs(dp[p]) * (xs ? xs[p] : fabs(xp[p]));
          }
        }
        dW[((int64_t)o * Cin + c) * K + k] = acc;
        if (SdW) SdW[((int64_t)o * Cin + c) * K + k] = sacc;
      }
}

/* ------------------------------------------------------ sampled points -- */
/* The sampled forms read their inputs from fp32 storage (every bf16 or fp32
   input value is exactly representable there) and compute in fp64. */

/* X at points pts[i] = (bc, k, ho, wo). */
void oracle_fwd_points(const int64_t* csr_row_ptr, const int32_t* csr_col,
                       const double* csr_val, int32_t K, int32_t Hin,
                       int32_t Win, int32_t Hout, int32_t Wout,
                       const float* x, int64_t npts, const int64_t* pts,
                       double* out, double* S) {
  int32_t s = Win / Wout;
  int64_t in_plane = (int64_t)Hin * Win;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < npts; ++i) {
    int64_t bc = pts[4 * i], k = pts[4 * i + 1], ho = pts[4 * i + 2], wo = pts[4 * i + 3];
    int64_t row = k * Hout + ho;
    double acc = 0.0, sab = 0.0;
    for (int64_t e = csr_row_ptr[row]; e < csr_row_ptr[row + 1]; ++e) {
      int32_t hi = csr_col[e] / Win, wi = csr_col[e] % Win;
      double t = csr_val[e] * (double)x[bc * in_plane + (int64_t)hi * Win + (wi + wo * s) % Win];
      acc += t;
      sab += fabs(t);
    }
    out[i] = acc;
    S[i] = sab;
  }
}

/* gx at points pts[i] = (bc, hi, wi): every forward term that reads input
   (hi, wi), found by scanning all CSR entries. */
void oracle_bwd_points(const int64_t* csr_row_ptr, const int32_t* csr_col,
                       const double* csr_val, int32_t K, int32_t Hin,
                       int32_t Win, int32_t Hout, int32_t Wout,
                       const float* G, int64_t npts, const int64_t* pts,
                       double* out, double* S) {
  int32_t s = Win / Wout;
  int64_t out_plane = (int64_t)K * Hout * Wout;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < npts; ++i) {
    int64_t bc = pts[3 * i], hi_t = pts[3 * i + 1], wi_t = pts[3 * i + 2];
    double acc = 0.0, sab = 0.0;
    for (int64_t row = 0; row < (int64_t)K * Hout; ++row) {
      for (int64_t e = csr_row_ptr[row]; e < csr_row_ptr[row + 1]; ++e) {
        int32_t hi = csr_col[e] / Win, wi = csr_col[e] % Win;
        if (hi != hi_t) continue;
        int64_t diff = ((wi_t - wi) % Win + Win) % Win; /* = wo * s mod Win */
        if (diff % s) continue;
        int64_t wo = diff / s;
        double t = csr_val[e] * (double)G[bc * out_plane + row * Wout + wo];
        acc += t;
        sab += fabs(t);
      }
    }
    out[i] = acc;
    S[i] = sab;
  }
}

/* Fused forward y at points pts[i] = (b, o, ho, wo):
   y = sum_{c,k} W[o,c,k] sum_e psi x;  S = sum |W psi x|. */
void oracle_fused_points(const int64_t* csr_row_ptr, const int32_t* csr_col,
                         const double* csr_val, int32_t K, int32_t Hin,
                         int32_t Win, int32_t Hout, int32_t Wout, int32_t Cin,
                         int32_t Cout, const float* x, const float* W,
                         int64_t npts, const int64_t* pts, double* out,
                         double* S) {
  int32_t s = Win / Wout;
  int64_t in_plane = (int64_t)Hin * Win;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < npts; ++i) {
    int64_t b = pts[4 * i], o = pts[4 * i + 1], ho = pts[4 * i + 2], wo = pts[4 * i + 3];
    double acc = 0.0, sab = 0.0;
    for (int32_t c = 0; c < Cin; ++c) {
      const float* xp = x + ((int64_t)b * Cin + c) * in_plane;
      for (int32_t k = 0; k < K; ++k) {
        int64_t row = (int64_t)k * Hout + ho;
        double w = (double)W[(o * Cin + c) * K + k];
        double xk = 0.0, xs = 0.0;
        for (int64_t e = csr_row_ptr[row]; e < csr_row_ptr[row + 1]; ++e) {
          int32_t hi = csr_col[e] / Win, wi = csr_col[e] % Win;
          double t = csr_val[e] * (double)xp[(int64_t)hi * Win + (wi + wo * s) % Win];
          xk += t;
          xs += fabs(t);
        }
        acc += w * xk;
        sab += fabs(w) * xs;
      }
    }
    out[i] = acc;
    S[i] = sab;
  }
}

/* Fused input gradient gx at points pts[i] = (b, c, hi, wi):
   gx = sum over forward terms reading (hi, wi) of psi * dX, with
   dX[b,c,k,ho,wo] = sum_o W[o,c,k] dy[b,o,ho,wo];  S = sum |psi W dy|. */
void oracle_fused_bwd_points(const int64_t* csr_row_ptr, const int32_t* csr_col,
                             const double* csr_val, int32_t K, int32_t Hin,
                             int32_t Win, int32_t Hout, int32_t Wout,
                             int32_t Cin, int32_t Cout, const float* dy,
                             const float* W, int64_t npts, const int64_t* pts,
                             double* out, double* S) {
  int32_t s = Win / Wout;
  int64_t plane = (int64_t)Hout * Wout;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < npts; ++i) {
    int64_t b = pts[4 * i], c = pts[4 * i + 1], hi_t = pts[4 * i + 2], wi_t = pts[4 * i + 3];
    double acc = 0.0, sab = 0.0;
    for (int64_t row = 0; row < (int64_t)K * Hout; ++row) {
      int64_t k = row / Hout, ho = row % Hout;
      for (int64_t e = csr_row_ptr[row]; e < csr_row_ptr[row + 1]; ++e) {
        int32_t hi = csr_col[e] / Win, wi = csr_col[e] % Win;
        if (hi != hi_t) continue;
        int64_t diff = ((wi_t - wi) % Win + Win) % Win;
        if (diff % s) continue;
        int64_t wo = diff / s;
        double dx = 0.0, ds = 0.0;
        for (int32_t o = 0; o < Cout; ++o) {
          double t = (double)W[(o * Cin + c) * K + k] *
                     (double)dy[((int64_t)b * Cout + o) * plane + ho * Wout + wo];
          dx += t;
          ds += fabs(t);
        }
        acc += csr_val[e] * dx;
        sab += fabs(csr_val[e]) * ds;
      }
    }
    out[i] = acc;
    S[i] = sab;
  }
}

/* Dense brute force on tiny grids: the basis evaluated at the true output
   longitude phi_wo (no shift), each (k, ho, wo) row normalised on its own.
   M[(k*Hout + ho)*Wout + wo][hi*Win + wi].  Returns 0 on success. */
int oracle_dense_matrix(int32_t in_nlat, int32_t in_nlon, int32_t in_poles,
                        int32_t out_nlat, int32_t out_nlon, int32_t out_poles,
                        int32_t kind, int32_t nrad, double cutoff, double* M) {
  int32_t K = oracle_basis_K(kind, nrad);
  if (K <= 0 || nrad > 8) return -1;
  int64_t ncol = (int64_t)in_nlat * in_nlon;
  double width = cutoff / (double)nrad;
  for (int32_t ho = 0; ho < out_nlat; ++ho)
    for (int32_t wo = 0; wo < out_nlon; ++wo) {
      double th_o = oracle_colat(out_nlat, out_poles, ho);
      double phi_o = 2.0 * OR_PI * (double)wo / (double)out_nlon;
      double norm[8] = {0};
      for (int pass = 0; pass < 2; ++pass)
        for (int32_t hi = 0; hi < in_nlat; ++hi)
          for (int32_t wi = 0; wi < in_nlon; ++wi) {
            double th_i = oracle_colat(in_nlat, in_poles, hi);
            double q = oracle_quad(in_nlat, in_poles, hi);
            double phi_i = 2.0 * OR_PI * (double)wi / (double)in_nlon;
            double dphi = phi_i - phi_o;
            double s1 = sin(0.5 * (th_i - th_o)), s2 = sin(0.5 * dphi);
            double hav = s1 * s1 + sin(th_o) * sin(th_i) * (s2 * s2);
            if (hav > 1.0) hav = 1.0;
            double d = 2.0 * asin(sqrt(hav));
            double beta = atan2(sin(dphi) * sin(th_i),
                                sin(th_o) * cos(th_i) - cos(th_o) * sin(th_i) * cos(dphi));
            for (int32_t k = 0; k < K; ++k) {
              int64_t m = (((int64_t)k * out_nlat + ho) * out_nlon + wo) * ncol +
                          (int64_t)hi * in_nlon + wi;
              double v = 0.0;
              if (kind == OR_INDICATOR) {
                v = ((1.0 - d / cutoff) > OR_TAU_SUPPORT) ? 1.0 : 0.0;
                if (pass == 1) M[m] = v;
                continue;
              }
              int32_t r = (kind == OR_ANISO) ? k / 3 : k;
              int32_t a = (kind == OR_ANISO) ? k % 3 : 0;
              double h = oracle_hat(d, r, width);
              if (!(h > OR_TAU_SUPPORT && q > 0.0)) {
                if (pass == 1) M[m] = 0.0;
                continue;
              }
              if (pass == 0) {
                if (a == 0) norm[r] += h * q;
                continue;
              }
              double ang = 1.0;
              if (a != 0) ang = (d < OR_D_COINCIDENT) ? 0.0 : (a == 1 ? cos(beta) : sin(beta));
              v = norm[r] > 0.0 ? h * ang * q / norm[r] : 0.0;
              M[m] = v;
            }
          }
    }
  return 0;
}
