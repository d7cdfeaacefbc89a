/*
 * disco.h -- C ABI of the GB300 (sm_103a) DISCO convolution library.
 *
 * DISCO = discrete-continuous convolution on the sphere.  The operations
 * follow the DISCO Kernel Development Guide (torch-harmonics).  Its
 * §Architecture snapshot names three kernels, all provided here:
 *   forward   the sparse contraction of the input grid into X[B,C,K,H,W]
 *   backward  its transpose, from X-shaped gradients back to the input grid
 *   fused     the contraction followed by the channel/basis einsum
 *             (y[b,o,ho,wo] = sum_{c,k} W[o,c,k] X[b,c,k,ho,wo])
 * Its §kpacked layout describes the neighbour-list form of psi, with the
 * values of all K basis functions side by side, built once at init.
 *
 * Conventions (all entry points):
 *  - Every tensor argument is a DEVICE pointer to a dense, C-contiguous array
 *    in the layout stated, 16-byte aligned, owned by the caller.  The library
 *    never allocates, frees or keeps a reference to caller memory beyond the
 *    call, and never synchronises the stream except where stated.
 *  - Outputs are fully overwritten (never accumulated into).
 *  - All validation happens on the host before any launch; a failed check
 *    returns a negative disco_status and launches nothing.  disco_last_error()
 *    then returns a message for the calling thread.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and is asynchronous unless stated.
 *  - Accumulation is fp32; the output dtype equals the input dtype.
 *  - The device must have compute capability 10.3 (sm_103a);
 *    DISCO_ERR_UNSUPPORTED_DEVICE otherwise.
 */
#ifndef DISCO_GB300_H
#define DISCO_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DISCO_API __attribute__((visibility("default")))
#else
#define DISCO_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DISCO_OK = 0,
  DISCO_ERR_INVALID_ARG = -1,        /* null pointer, bad size, inconsistent psi */
  DISCO_ERR_UNSUPPORTED = -2,        /* valid but not supported (W_in % W_out, K, dtype, s) */
  DISCO_ERR_ALIGNMENT = -3,          /* a pointer is not 16-byte aligned */
  DISCO_ERR_UNSUPPORTED_DEVICE = -4, /* current device is not compute capability 10.3 */
  DISCO_ERR_LAUNCH = -5,             /* a kernel launch was rejected by the runtime */
  DISCO_ERR_CUDA = -6,               /* another CUDA runtime call failed */
  DISCO_ERR_WORKSPACE = -7,          /* workspace missing or too small */
  DISCO_ERR_DEVICE_BOUNDS = -8       /* bounds-checked build: a kernel's range check failed */
} disco_status;

/* Element type of the activations (x, X, G, gx, y, dy) and of W.  The
   guide's §Profiling / Serial Benchmarks section names fp32, bf16 and fp16
   as the precisions to cover; fp16 runs the same kernels as bf16 with fp16
   operands (and fp16 copies of the Toeplitz tables), fp32 accumulation. */
typedef enum { DISCO_F32 = 0, DISCO_BF16 = 1, DISCO_F16 = 2 } disco_dtype;

/* Latitude rows of a grid.  poles = 0 (equiangular, midpoints): colatitude
   (i + 1/2) pi / nlat; poles = 1 (equiangular, both poles on the grid):
   colatitude i pi / (nlat - 1); poles = 2 (Legendre-Gauss, the grid the
   DISCO Kernel Development Guide's benchmark shapes name "legendre-gauss"):
   colatitude arccos x_i with x_0 > x_1 > ... the roots of the Legendre
   polynomial P_nlat, and the Gauss-Legendre weight of row i as the input
   quadrature weight (sin(colatitude) on the equiangular grids).
   Longitude 2 pi j / nlon on every grid. */
typedef struct {
  int32_t nlat, nlon, poles;
} disco_grid;

/* Filter basis on geodesic distance d.  n_radial hats of width
   cutoff / n_radial centred at r * width (hat_r(d) = max(0, 1 - |d - r w| / w)).
   kind 0 (isotropic): K = n_radial, basis k = hat_k.
   kind 1 (anisotropic): K = 3 n_radial, basis k = 3 r + a is hat_r times
   {1, cos(beta), sin(beta)}[a], beta the bearing from the output point to the
   input point (0 = north, pi/2 = east).
   Values are hat * angular factor * sin(colatitude_in) / N(r, ho) with N the
   sum of hat_r * sin(colatitude_in) over ring r's support (support: hat > 1e-9
   and sin(colatitude_in) > 0; pole rows of a pole grid carry weight 0). */
typedef struct {
  int32_t kind;
  int32_t n_radial;
  double cutoff; /* radians */
} disco_basis;

/* One (ho, hi) segment of psi: the input row hi seen from output row ho is one
   contiguous wrapped window of columns, symmetric about offset 0.  Offsets
   delta in [0, D] address the mirrored pairs (delta, -delta); the weights of
   the self-mirrored offsets (0 and, on a full ring of even width, W_in/2) are
   stored halved so every step is a pair. */
typedef struct {
  int32_t ho, hi;
  int32_t D;     /* pair steps are delta = 0 .. D */
  int32_t hoff;  /* row of this run's first pair weight in psi.hval */
  int32_t e0;    /* first entry of the run in the union (kpacked) arrays */
  int32_t len;   /* entries of the run in the union arrays (2m+1, or W_in) */
  int32_t npair; /* mirrored pairs delta = 1 .. npair */
  int32_t anti;  /* 1 if the run holds the unpaired antipodal column */
} disco_run;

/* One (input-row group, output row) entry of the transpose tables; see
   disco_psi.grp_ptr. */
typedef struct {
  int32_t ho;   /* output row */
  int32_t off;  /* element offset of the entry's blocks in psi.gtab (multiple of 8) */
  int16_t MW;   /* window half-width in output columns, a multiple of 8 */
  int16_t KB;   /* 16-column steps of one tile block: ceil((TQ + 2 MW) / 16) */
  int16_t nch;  /* 64-column chunks: ceil(KB / 4) */
  int8_t r0;    /* first and last input row of the group (0 .. 7) with psi */
  int8_t r1;    /*   support at this output row: the rows the entry's tiles cover */
} disco_grp_ent;

/* psi: sizes set by disco_psi_plan, device pointers (into the caller's psi
   buffer) set by disco_build_psi_kpacked.  Read-only after the build.
   Index structures are int32; values fp32. */
typedef struct {
  disco_grid grid_in, grid_out;
  disco_basis basis;
  int32_t K;        /* basis functions */
  int32_t K_pad;    /* K rounded up to a multiple of 8 (page: K_PAD = ceil(K/8)*8) */
  int32_t s;        /* W_in / W_out */
  int32_t max_row;  /* largest union row (neighbours of one output row) */
  int64_t nnz;      /* union neighbours summed over output rows */
  int64_t nnz_csr;  /* CSR non-zeros summed over (k, ho) rows */
  int64_t nruns;    /* (ho, hi) segments */
  int64_t nhval;    /* rows of hval */
  int64_t nftab;    /* elements of ftab */
  int32_t ngrp;     /* input-row groups with transpose tables (0 if s > 2) */
  int32_t grp_max;  /* most entries of one group */
  int64_t ngrp_ent; /* entries summed over groups */
  int64_t ngtab;    /* elements of gtab */
  size_t bytes;     /* device bytes disco_build_psi_kpacked needs */
  /* Union ("kpacked") layout, shared across k (§kpacked layout):
     neighbours of output row ho (for output longitude 0) are entries
     row_ptr[ho] .. row_ptr[ho+1]-1, ordered by hi ascending then by the
     signed column offset ((wi + floor(W/2)) mod W) - floor(W/2) ascending. */
  int32_t* row_ptr;     /* [Hout + 1] */
  int32_t* idx;         /* [nnz][2] = (hi, wi) */
  float* val;           /* [nnz][K_pad], zero for k >= K and non-structural k */
  /* CSR layout (§Architecture snapshot): row k * Hout + ho, column hi * W_in + wi,
     same neighbour order, only entries whose ring is structural. */
  int32_t* csr_row_ptr; /* [K * Hout + 1] */
  int32_t* csr_col;     /* [nnz_csr] */
  float* csr_val;       /* [nnz_csr] */
  /* Kernel-side forms derived from the above. */
  int32_t* run_ptr;     /* [Hout + 1]: runs of output row ho */
  disco_run* runs;      /* [nruns], ordered by (ho, hi) */
  int32_t* trun_ptr;    /* [Hin + 1]: runs that read input row hi */
  int32_t* truns;       /* [nruns]: run indices ordered by (hi, ho) */
  float* hval;          /* [nhval][K_pad]: pair weights, see disco_run */
  int32_t* row_order;   /* [Hout]: output rows by descending work (launch order) */
  /* bf16 tables of each run for the tensor-core tiles (values rounded from val).
     Forward table of run r: K rows of TLf = roundup8(len + 16) elements at
     ftab + ftab_off[r]; row k holds psi_k(delta) at index 8 + delta - dlo for
     the run's offsets dlo..dhi and zeros elsewhere. */
  int32_t* ftab_off;    /* [nruns + 1], multiples of 8 */
  uint16_t* ftab;       /* [nftab] */
  /* Transpose tables by input-row group, for s <= 2 (the tensor-core
     transpose tiles): group z holds input rows 8z .. 8z+7; with TQ = 32 / s,
     grp_ptr[z] .. grp_ptr[z+1]-1 are its entries, one per output row ho that
     one of its rows reads, ho ascending, with
       MW  = max over the group's runs (ho, hi) of max(EH, -EL) rounded up to 8,
             EH = floor(dhi/s), EL = ceil((dlo - s + 1)/s),
       KB  = ceil((TQ + 2 MW) / 16), nch = ceil(KB / 4).
     Block (k, c), c < nch, of an entry is 8*s*CW bf16 values at
     gtab + off + (k*nch + c) * 8*s*CW, CW = roundup8(63 + TQ); element
     [r][p][y] is psi_k of run (ho, 8z + r) at offset s*e + p,
     e = MW + TQ - 1 - 64c - y, when that run exists and holds that offset,
     else 0. */
  int32_t* grp_ptr;     /* [ngrp + 1] */
  disco_grp_ent* grp;   /* [ngrp_ent] */
  uint16_t* gtab;       /* [ngtab] */
  /* ftab and gtab again with the values rounded to fp16 instead of bf16
     (same offsets), for fp16 inputs: one tensor-core MMA takes A and B of
     the same type. */
  uint16_t* ftab_h;     /* [nftab] */
  uint16_t* gtab_h;     /* [ngtab] */
} disco_psi;

/* Library version (major * 10000 + minor * 100 + patch). */
DISCO_API int32_t disco_version(void);

/* Message for the last non-OK status returned on this thread ("" if none). */
DISCO_API const char* disco_last_error(void);

/* Host only, no device work.  Bytes of device workspace that disco_psi_plan
   and disco_build_psi_kpacked need for these grids and basis. */
DISCO_API int disco_psi_workspace_bytes(const disco_grid* grid_in, const disco_grid* grid_out,
                              const disco_basis* basis, size_t* bytes);

/* Init time; BLOCKS the host (one device-to-host copy of per-row counts).
   Runs the support-counting kernels (fp64 geometry) on `stream` into
   `workspace` and fills the sizes of *psi (pointers are cleared).  The
   workspace contents are consumed by disco_build_psi_kpacked and must be left
   untouched in between.  Requires W_in % W_out == 0, 1 <= K <= 16, nlat >= 2
   (>= 3 on a pole grid), nlon >= 1. */
DISCO_API int disco_psi_plan(const disco_grid* grid_in, const disco_grid* grid_out,
                   const disco_basis* basis, void* workspace, size_t workspace_bytes,
                   void* stream, disco_psi* psi);

/* Init time, asynchronous.  Builds psi (§kpacked layout, CSR layout and the
   kernel-side forms) into `buffer` (device, >= psi->bytes bytes, 256-byte
   aligned) and sets the pointers of *psi into it.  Values are computed in fp64
   on the device and stored as fp32. */
DISCO_API int disco_build_psi_kpacked(disco_psi* psi, void* buffer, size_t bytes, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Init time, asynchronous.  Writes a built psi in the page's uniform
   K-packed form (§kpacked layout), for interoperability with code that reads
   that form:
     pack_idx   [H_out][nbr_pad][2]      int64 (hi, wi), shared across k
     pack_val   [H_out][nbr_pad][K_pad]  fp32, zero for k >= K
     pack_count [H_out]                  int64, neighbours of row ho
   Row ho holds the union entries of output row ho in the union layout's
   order (hi ascending, then signed offset); entries at and past
   pack_count[ho] are (0, 0) with zero values.  nbr_pad >= psi->max_row
   (DISCO_ERR_INVALID_ARG otherwise); all three are caller-owned device
   buffers, fully overwritten. */
DISCO_API int disco_psi_export_kpacked(const disco_psi* psi, int64_t* pack_idx, float* pack_val,
                                       int64_t* pack_count, int32_t nbr_pad, void* stream);

/* Forward S2 contraction (§Architecture snapshot, forward kernel; §Backward
   direction: gather, each output pixel reads a bounded neighbourhood):
     X[b,c,k,ho,wo] = sum_{(hi,wi) in row (k,ho)} psi[k,ho,hi,wi]
                        * x[b,c,hi,(wi + wo*s) mod W_in]
   x: [B, C, H_in, W_in], X: [B, C, K, H_out, W_out], both `dtype`.
   Supports s in {1, 2}.  bf16 or fp16 with W_in % 8 == 0, W_in >= 64 and
   K <= 9 runs on the tensor cores (banded Toeplitz tiles of the run windows,
   fp32 accumulation in tensor memory); fp32, and other bf16 / fp16 shapes,
   run the CUDA-core gather. */
DISCO_API int disco_fwd(const disco_psi* psi, const void* x, void* X, int32_t B, int32_t C,
              disco_dtype dtype, void* stream);

/* Transpose contraction (§Architecture snapshot, backward kernel; §Backward
   direction: gather direction, each input pixel accumulates from its
   neighbourhood, no atomics):  gx = psi^T G, i.e.
     gx[b,c,hi,wi] = sum_{k,ho,wo} sum_{wi0: (wi0 + wo*s) mod W_in = wi}
                       psi[k,ho,hi,wi0] * G[b,c,k,ho,wo]
   G: [B, C, K, H_out, W_out], gx: [B, C, H_in, W_in], both `dtype`.
   Each output element has one owner (latitude-row ownership, no atomics).
   bf16 or fp16 with W_in and W_out multiples of 8, W_out >= 64 and K <= 16
   runs on the tensor cores (polyphase Toeplitz tiles, 8 input rows per tile
   sharing each G window, psi from the tables by input-row group); other
   cases run the CUDA-core gather. */
DISCO_API int disco_bwd(const disco_psi* psi, const void* G, void* gx, int32_t B, int32_t C,
              disco_dtype dtype, void* stream);

/* Device workspace bytes of disco_fused_conv for these B, Cin, Cout: the
   intermediate X[B, Cin, K, H_out, W_out] (dtype) when the tensor-core
   contraction takes the shape (bf16 or fp16, W_in % 8 == 0, W_in >= 64,
   s in {1, 2}, K <= 9), else 0 (no workspace needed). */
DISCO_API size_t disco_fused_conv_workspace_bytes(const disco_psi* psi, int32_t B, int32_t Cin, int32_t Cout,
                                                  disco_dtype dtype);

/* Fused convolution (§Architecture snapshot: the fused kernel, the
   contraction followed by the einsum):
     y[b,o,ho,wo] = sum_{c,k} W[o,c,k] X[b,c,k,ho,wo]
   with X the forward contraction, in one call:
     - where the tensor-core contraction takes the shape, X is produced by it
       into `workspace` (disco_fused_conv_workspace_bytes bytes) and the
       einsum runs as a tcgen05 GEMM (M = 128 pixels, N = Cout, K = Cin*K);
     - otherwise (bf16 only) X is built in shared memory by the CUDA-core
       gather, 16 input channels at a time, and contracted on the tcgen05
       tensor cores without leaving the chip (workspace unused; needs
       Cin % 16 == 0).
   Accumulation is fp32 (TMEM); X is rounded to the dtype before the einsum.
   x: [B, Cin, H_in, W_in], W: [Cout, Cin, K], y: [B, Cout, H_out, W_out],
   all bf16 or all fp16 (dtype).  The einsum GEMM takes any Cout (tiles of
   up to 256 outputs); the CUDA-core gather path needs Cout <= 256.  fp16
   needs the tensor-core path: the forward shape above and the GEMM shape
   (H_out*W_out, Cin*K and Cout multiples of 8, Cin*K >= 64, Cout >= 16);
   else DISCO_ERR_UNSUPPORTED before any launch. */
DISCO_API int disco_fused_conv(const disco_psi* psi, const void* x, const void* W, void* y,
                     int32_t B, int32_t Cin, int32_t Cout, disco_dtype dtype,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Device workspace bytes of disco_fused_conv_bwd_input (the intermediate dX,
   B * Cin * K * H_out * W_out elements of the dtype). */
DISCO_API size_t disco_fused_conv_bwd_input_workspace_bytes(const disco_psi* psi, int32_t B,
                                                  int32_t Cin, disco_dtype dtype);

/* Input gradient of the fused convolution (§Architecture snapshot: the
   fused kernel and its backward are paired through an autograd function;
   §Backward direction for the transpose).  The guide gives no formula; the
   plain reading is the gradient of y = einsum(W, psi x) with respect to x,
   the upstream gradient routed through W^T first, then the transpose:
     dX[b,c,k,ho,wo] = sum_o W[o,c,k] dy[b,o,ho,wo]   (tcgen05 tensor cores)
     gx = psi^T dX                                    (the transpose contraction)
   dy: [B, Cout, H_out, W_out], W: [Cout, Cin, K], gx: [B, Cin, H_in, W_in],
   all bf16 or all fp16 (dtype).  dX is kept in `workspace` (>=
   disco_fused_conv_bwd_input_workspace_bytes) in the dtype: as
   [K*H_out][B*Cin][W_out] when both steps run on the tensor cores (dX GEMM:
   H_out*W_out and Cout multiples of 8, Cout >= 64, Cin*K a multiple of 64;
   transpose: the disco_bwd tensor-core shape), whose 128-channel windows the
   transpose streams faster than those of [B][Cin*K][H_out*W_out], the
   layout of the other cases (bf16 only: a CUDA-core dX GEMM, then
   disco_bwd).  fp16 needs the tensor-core shapes, else DISCO_ERR_UNSUPPORTED
   before any launch. */
DISCO_API int disco_fused_conv_bwd_input(const disco_psi* psi, const void* dy, const void* W,
                               void* gx, int32_t B, int32_t Cin, int32_t Cout,
                               disco_dtype dtype, void* workspace, size_t workspace_bytes,
                               void* stream);

/* Size of the fixed device scratch of disco_fused_conv_bwd_input_noalloc. */
#define DISCO_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20) /* 64 MiB */

/* Allocation-free form of disco_fused_conv_bwd_input (the pages have no
   counterpart; it exists for callers that cannot allocate device memory
   themselves, e.g. a runtime whose allocator owns all device memory from
   start-up, or a hot loop that must not risk the implicit device
   synchronisation of cudaMalloc).  Same arguments, result and accuracy as
   disco_fused_conv_bwd_input, without the workspace: the dX intermediate
   lives in a fixed 64 MiB (DISCO_NOALLOC_SCRATCH_BYTES) device array that
   every GPU loading this library holds until the process exits.  Problems
   whose dX (B * Cin * K * H_out * W_out * 2 bytes) exceeds it are rejected
   with DISCO_ERR_WORKSPACE before any launch.  The call allocates and frees
   nothing.  The first call on a device looks up the array's device address
   (cudaGetSymbolAddress, with that device current) and caches it; make that
   first call before any stream capture.  All calls share the one array and
   it keeps the last call's contents (dX is fully rewritten each call), so
   calls that overlap on the GPU, e.g. on two streams, race and must be
   serialised by the caller. */
DISCO_API int disco_fused_conv_bwd_input_noalloc(const disco_psi* psi, const void* dy,
                                                 const void* W, void* gx, int32_t B,
                                                 int32_t Cin, int32_t Cout, disco_dtype dtype,
                                                 void* stream);

/* Device workspace bytes of disco_fused_conv_bwd_weight: X (dtype) plus the
   fp32 partial sums of the split reduction; 0 when the call does not take the
   shape (see below). */
DISCO_API size_t disco_fused_conv_bwd_weight_workspace_bytes(const disco_psi* psi, int32_t B,
                                                            int32_t Cin, int32_t Cout, disco_dtype dtype);

/* Weight gradient of the fused convolution (§Architecture snapshot: the
   fused variants are paired with their backward through autograd functions;
   the page gives no formula, the plain reading is the gradient of
   y = einsum(W, X) with respect to W):
     dW[o,c,k] = sum_b sum_{ho,wo} dy[b,o,ho,wo] X[b,c,k,ho,wo],
   X the forward contraction of x (recomputed, not stored by the forward).
   x: [B, Cin, H_in, W_in], dy: [B, Cout, H_out, W_out], dW: [Cout, Cin, K],
   all bf16 or all fp16 (dW rounded from an fp32 sum).  X is built by the tensor-core
   contraction into `workspace` (>= disco_fused_conv_bwd_weight_workspace_bytes,
   256-byte aligned), then a tcgen05 GEMM over the pixels (reduction split
   across CTAs into fp32 partials, summed in a fixed order: deterministic).
   Takes bf16 or fp16 with the tensor-core forward shape (W_in % 8 == 0, W_in >= 64,
   s in {1, 2}, K <= 9), H_out*W_out, Cin*K and Cout multiples of 8,
   Cin*K >= 64 and Cout >= 16; else DISCO_ERR_UNSUPPORTED.  Asynchronous on
   `stream`. */
DISCO_API int disco_fused_conv_bwd_weight(const disco_psi* psi, const void* x, const void* dy, void* dW,
                                          int32_t B, int32_t Cin, int32_t Cout, disco_dtype dtype,
                                          void* workspace, size_t workspace_bytes, void* stream);

/* Host-buffer forms of disco_fwd / disco_bwd for data that lives in host
   memory: `in_host` and `out_host` are HOST pointers (page-locked memory
   lets the copies overlap the kernels; pageable memory works, with the
   copies staged by the runtime).  The B*C planes go in blocks of 128: each
   block's host-to-device copy, contraction (on `stream`) and device-to-host
   copy are ordered by events, and consecutive blocks overlap (block i+1 is
   copied in and block i-1 copied out while block i computes).  The copies
   run on two streams the library creates once per device and shares between
   calls, so calls on different caller streams also overlap one another.
   Staging (two slots of one block's input and output) is the caller's
   device workspace of disco_host_workspace_bytes bytes, 256-byte aligned.
   Asynchronous: `stream` waits for the last copy-out, so synchronising
   `stream` makes out_host readable.  Same results as the device forms, bit
   for bit; the same shape and dtype rules.  forward != 0: sizes for
   disco_fwd_host, else disco_bwd_host (0 for invalid arguments). */
DISCO_API size_t disco_host_workspace_bytes(const disco_psi* psi, int32_t B, int32_t C, int32_t forward,
                                            disco_dtype dtype);
DISCO_API int disco_fwd_host(const disco_psi* psi, const void* x_host, void* X_host, int32_t B, int32_t C,
                             disco_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);
DISCO_API int disco_bwd_host(const disco_psi* psi, const void* G_host, void* gx_host, int32_t B, int32_t C,
                             disco_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/* Diagnostics; BLOCKS the host (synchronises the current device).  Reads
   the device status word into *flags (0 = no fault; bit 0 = an mbarrier wait
   of the fused forward timed out, bit 1 = one of the dX GEMM timed out,
   bit 2 = one of the tensor-core forward contraction timed out,
   bit 3 = one of the tensor-core transpose contraction timed out or met an
   input-row group reading more output rows than it can hold, bit 4 = the
   wait of disco_check_wait_timeout ran out, bit 5 = in the bounds-checked
   build, a gather index or a TMA or bulk-copy coordinate fell outside the
   tensor it addresses; a kernel that times out stops issuing work, frees its
   tensor memory and returns, leaving its outputs incomplete).  clear != 0
   resets the word.  Returns DISCO_ERR_DEVICE_BOUNDS (with *flags filled in)
   when bit 5 is set, else DISCO_OK or a CUDA error. */
DISCO_API int disco_device_status(int32_t* flags, int32_t clear);

/* Build options of the loaded library: DISCO_BUILD_DEBUG_BOUNDS when it is the
   bounds-checked build (compiled with -DDISCO_DEBUG_BOUNDS).  In that build
   every kernel checks each gather index and each TMA or bulk-copy coordinate
   against the extents of the tensor it addresses before the access; a failed
   check skips the access (a skipped copy still completes its transaction
   bytes, so no wait runs out), sets bit 5 of the device status word and
   never traps.  It stands in for a memory checker on small cases; its
   kernels are slower and it is not the product build. */
#define DISCO_BUILD_DEBUG_BOUNDS 1
DISCO_API int32_t disco_build_flags(void);

/* Diagnostic of the failure path, asynchronous: launches one small kernel
   whose thread waits on an mbarrier phase that nothing completes, with the
   bounded wait the tensor-core kernels use (`limit` polls, 1 <= limit <=
   2^24).  When the wait runs out the kernel sets bit 4 of the device status
   word and returns: nothing faults, traps or hangs, and the context stays
   usable.  Lets a test check that a timed-out wait reaches
   disco_device_status. */
DISCO_API int disco_check_wait_timeout(uint32_t limit, void* stream);

/* Diagnostic of the tile schedulers, synchronous.  The persistent
   tensor-core kernels draw their tiles from one of 1024 words of a
   library-owned device table (word = launch number mod 1024) holding the
   tag of the launch using it, the number of its CTAs drawing, and its next
   tile.  A CTA joins the word (its own tag: one more drawer; another tag
   with no drawer: the word becomes its launch's, counter 0; another launch
   still drawing: a bounded wait, after which the CTA takes no tile and sets
   bit 2 (forward) or bit 3 (transpose) of the status word), draws with an
   atomic add and leaves on every exit path, so no launch, failed or not,
   leaves a word that blocks a later one.  This call first runs one thread
   through that protocol on a private word (take-over, draws in order, a
   sibling joining, a launch waiting while another draws, take-over once
   the drawers left) and returns DISCO_ERR_CUDA naming the first step that
   went wrong; it then leaves another launch's tag with its counter
   part-way and no drawer in the words the next launch will use.  That
   launch must compute every tile with a clear status word. */
DISCO_API int disco_check_sched_takeover(void);

#ifdef __cplusplus
}
#endif

#endif /* DISCO_GB300_H */
