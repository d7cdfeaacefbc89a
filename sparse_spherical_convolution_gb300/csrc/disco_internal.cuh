// disco_internal.cuh -- helpers shared by the library's translation units
// (error reporting, device checks, bf16 conversion).  Not part of the ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "disco.h"

namespace disco {

// An NVTX range around one C-ABI call, so that a profiler timeline that
// records NVTX shows each call by name (header-only NVTX: no library to link;
// without a profiler attached the push and pop return at once).
struct NvtxScope {
  explicit NvtxScope(const char* name) { nvtxRangePushA(name); }
  ~NvtxScope() { nvtxRangePop(); }
  NvtxScope(const NvtxScope&) = delete;
  NvtxScope& operator=(const NvtxScope&) = delete;
};

// Records `msg` (printf-style) as this thread's last error and returns `st`.
int fail(int st, const char* fmt, ...);

// 0 if the current device is compute capability 10.3, else a failure status.
int check_device();

// Launch-error check right after a launch.
int check_launch(const char* what);

// Process-unique, nonzero id of a kernel launch (selects the launch's
// scheduler slot, disco_sched.cuh); thread-safe.
unsigned long long next_launch_id();
// The id the next launch will get (without taking it).
unsigned long long peek_launch_id();

// DISCO_OK if `p` is device (or managed) memory of the current device, else
// DISCO_ERR_INVALID_ARG naming `name`: a host pointer or a pointer of another
// device is refused on the host instead of faulting in a kernel.
int check_dev_ptr(const void* p, const char* name);

// The calling thread's current CUDA context (driver handle), or null.  Caches
// of device addresses and library streams are keyed on it as well as on the
// device index, so a context that was reset and re-created is seen as new.
void* current_context();

// Scheduler words of the persistent kernels (disco_sched.cuh): leave another
// launch's tag, counter part-way, in the word that launch `id` will use.
cudaError_t fwd_sched_plant(unsigned long long id);
cudaError_t btc_sched_plant(unsigned long long id);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validates the pieces of psi every hot call relies on.
int check_psi(const disco_psi* psi);

// disco_fwd (fwd) / disco_bwd (!fwd); check_ptrs = false skips the device-
// pointer queries, for buffers the library itself hands in.
int contract(bool fwd, const disco_psi* psi, const void* in, void* out, int32_t B, int32_t C,
             disco_dtype dtype, void* stream, bool check_ptrs);

// Forward contraction on the tensor cores (bf16); DISCO_ERR_UNSUPPORTED,
// without launching, for shapes that path does not take.
// f16: x and X are fp16 (else bf16).
int fwd_tensor_core(const disco_psi* psi, const void* x, void* X, int BC, cudaStream_t st, bool f16 = false);
bool fwd_tc_supported(const disco_psi* psi, int BC);

// ORs the tensor-core unit's status word into *v (device already synchronised).
cudaError_t tc_status(int32_t* v, bool clear);

// Transpose contraction on the tensor cores (bf16); DISCO_ERR_UNSUPPORTED,
// without launching, for shapes that path does not take.
// rows_of_channels: G is [K*H_out][BC][W_out] instead of [BC][K*H_out][W_out].
// f16: G and gx are fp16 (else bf16).
int bwd_tensor_core(const disco_psi* psi, const void* G, void* gx, int BC, cudaStream_t st,
                    bool rows_of_channels = false, bool f16 = false);
bool bwd_tc_supported(const disco_psi* psi, int BC);
cudaError_t btc_status(int32_t* v, bool clear);

// Dense GEMMs of the fused paths on the tensor cores (TMA-fed tcgen05):
//   einsum: y[b][o][p] = sum_j X[b][j][p] W[o][j]   (j = c*K + k)
//   dX:     dX[b][j][p] = sum_o dy[b][o][p] W[o][j]
// DISCO_ERR_UNSUPPORTED, without launching, for shapes they do not take.
int einsum_tensor_core(const void* X, const void* W, void* y, int B, int CK, int Cout, int64_t P,
                       cudaStream_t st, bool f16 = false);
// rows_of_channels = {K, H_out, W_out, C} (or null): write dX as
// [K*H_out][B*C][W_out] instead of [B][C*K][P] (W_out % 8 == 0).
bool dx_tensor_core_supported(int Cout, int CK, int64_t P);
// Shape rule of both GEMMs: P % 8 == 0, P >= 128, Kt % 8 == 0, Kt >= 64, Nt % 8 == 0, Nt >= 16.
bool gemm_tc_supported(int64_t P, int Kt, int Nt);
int dx_tensor_core(const void* dy, const void* W, void* dX, int B, int Cout, int CK, int64_t P,
                   cudaStream_t st, const int* rows_of_channels = nullptr, bool f16 = false);
cudaError_t gemm_status(int32_t* v, bool clear);

// Words of failed range checks, one per unit (disco_bounds.cuh): OR into *v
// and optionally clear; always 0 outside the bounds-checked build.
cudaError_t contract_bounds(int32_t* v, bool clear);
cudaError_t psi_bounds(int32_t* v, bool clear);
cudaError_t tc_bounds(int32_t* v, bool clear);
cudaError_t btc_bounds(int32_t* v, bool clear);
cudaError_t gemm_bounds(int32_t* v, bool clear);
cudaError_t fused_bounds(int32_t* v, bool clear);
// Weight gradient dW[o][j] = sum_b sum_p dy[b][o][p] X[b][j][p] (split reduction
// through fp32 partials of dw_partial_bytes bytes, then rounded to bf16).
bool dw_tensor_core_supported(int B, int Cout, int CK, int64_t P);
size_t dw_partial_bytes(int B, int Cout, int CK, int64_t P);
int dw_tensor_core(const void* dy, const void* X, void* dW, void* partials, int B, int Cout, int CK, int64_t P,
                   cudaStream_t st, bool f16 = false);

// Geometry of the transpose tables by input-row group (disco_psi.grp_ptr):
// 8 input rows per group, 64-column chunks, TQ = 32 / s decimated output
// columns per tile block, table rows of CW = roundup8(63 + TQ) elements.
constexpr int kGrpRows = 8;
constexpr int kGrpChunk = 64;
__host__ __device__ constexpr int grp_tq(int s) { return 32 / s; }
__host__ __device__ constexpr int grp_cw(int s) { return (kGrpChunk - 1 + grp_tq(s) + 7) & ~7; }
__host__ __device__ constexpr int grp_block(int s) { return kGrpRows * s * grp_cw(s); }

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ __half from_f32<__half>(float v) {
  return __float2half_rn(v);
}

}  // namespace disco
