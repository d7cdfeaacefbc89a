// disco_bounds.cuh -- range checks of the bounds-checked build.
//
// Compiled with -DDISCO_DEBUG_BOUNDS (build.py --debug-bounds), the kernels
// check every gather index and every TMA or bulk-copy coordinate against the
// extents of the tensor it addresses before the access.  A failed check sets
// kStatusBounds in its translation unit's bounds word and skips the access;
// a skipped copy still completes its transaction bytes on its mbarrier, so
// no wait is left to run out.  Nothing traps.  disco_device_status gathers
// the words of all units and returns DISCO_ERR_DEVICE_BOUNDS.  In the normal
// build DISCO_IN_BOUNDS(cond) is the constant true, `cond` is not evaluated,
// and every check compiles away.
//
// This build stands in for a memory checker: run on small cases it shows
// that no kernel addresses memory outside its tensors.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace disco {

constexpr int kStatusBounds = 1 << 5;

#ifdef DISCO_DEBUG_BOUNDS
static __device__ int g_bounds_word = 0;  // one per translation unit
__device__ __forceinline__ bool bounds_record(bool ok) {
  if (!ok) atomicOr(&g_bounds_word, kStatusBounds);
  return ok;
}
#define DISCO_IN_BOUNDS(cond) (::disco::bounds_record((cond)))
// host: ORs this unit's bounds word into *v (and clears it)
#define DISCO_BOUNDS_READER(name)                                                                    \
  cudaError_t name(int32_t* v, bool clear) {                                                         \
    int32_t t = 0;                                                                                   \
    cudaError_t e = cudaMemcpyFromSymbol(&t, ::disco::g_bounds_word, sizeof(int32_t));               \
    if (e == cudaSuccess && clear) {                                                                 \
      const int32_t zero = 0;                                                                        \
      e = cudaMemcpyToSymbol(::disco::g_bounds_word, &zero, sizeof(int32_t));                        \
    }                                                                                                \
    *v |= t;                                                                                         \
    return e;                                                                                        \
  }
#else
#define DISCO_IN_BOUNDS(cond) (true)
#define DISCO_BOUNDS_READER(name) \
  cudaError_t name(int32_t*, bool) { return cudaSuccess; }
#endif

// Completes `bytes` of an mbarrier's expected transactions without a copy:
// what a copy skipped by a failed check leaves undone.
__device__ __forceinline__ void mbar_complete_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(bar))),
               "r"(bytes)
               : "memory");
}

}  // namespace disco
