// disco_capi.cu -- error reporting, device and argument checks of the C ABI.

#include <stdarg.h>
#include <atomic>
#include <mutex>
#include <stdio.h>

#include "disco_internal.cuh"

namespace disco {

namespace {
thread_local char g_last_error[512] = "";
}

int fail(int st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

int check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DISCO_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  // cached per device: the attribute queries are cheap but not free
  static thread_local int cached_dev = -1, cached_ok = 0;
  if (dev == cached_dev) {
    return cached_ok ? DISCO_OK
                     : fail(DISCO_ERR_UNSUPPORTED_DEVICE, "device %d is not compute capability 10.3", dev);
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return fail(DISCO_ERR_CUDA, "cudaDeviceGetAttribute failed");
  cached_dev = dev;
  cached_ok = (major == 10 && minor == 3);
  if (!cached_ok)
    return fail(DISCO_ERR_UNSUPPORTED_DEVICE, "device %d is compute capability %d.%d, need 10.3", dev,
                major, minor);
  return DISCO_OK;
}

namespace {
std::atomic<unsigned long long> g_launch_seq{0};
}

unsigned long long next_launch_id() { return g_launch_seq.fetch_add(1, std::memory_order_relaxed) + 1; }

unsigned long long peek_launch_id() { return g_launch_seq.load(std::memory_order_relaxed) + 1; }

int check_dev_ptr(const void* p, const char* name) {
  if (!p) return fail(DISCO_ERR_INVALID_ARG, "%s is null", name);
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();  // the failed query is not a sticky error; clear it
    return fail(DISCO_ERR_INVALID_ARG, "%s: the CUDA runtime does not know this pointer (%s)", name,
                cudaGetErrorString(e));
  }
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
    return fail(DISCO_ERR_INVALID_ARG, "%s is not device memory (host or unregistered pointer)", name);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(DISCO_ERR_CUDA, "cudaGetDevice failed");
  if (at.type == cudaMemoryTypeDevice && at.device != dev)
    return fail(DISCO_ERR_INVALID_ARG, "%s lives on device %d, the current device is %d", name, at.device, dev);
  return DISCO_OK;
}

void* current_context() {
  using GetCtx = int (*)(void**);
  static GetCtx fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<GetCtx>(p);
  });
  void* ctx = nullptr;
  if (!fn || fn(&ctx) != 0) return nullptr;
  return ctx;
}

int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(DISCO_ERR_LAUNCH, "%s: %s", what, cudaGetErrorString(e));
  return DISCO_OK;
}

int check_psi(const disco_psi* psi) {
  if (!psi) return fail(DISCO_ERR_INVALID_ARG, "psi is null");
  if (!psi->row_ptr || !psi->run_ptr || !psi->runs || !psi->trun_ptr || !psi->truns || !psi->hval ||
      !psi->row_order || !psi->val || !psi->idx)
    return fail(DISCO_ERR_INVALID_ARG, "psi is not built (call disco_build_psi_kpacked)");
  if (psi->K < 1 || psi->K > 16 || psi->K_pad != (psi->K + 7) / 8 * 8)
    return fail(DISCO_ERR_INVALID_ARG, "psi K / K_pad inconsistent");
  if (psi->grid_out.nlon < 1 || psi->grid_in.nlon % psi->grid_out.nlon != 0 ||
      psi->s != psi->grid_in.nlon / psi->grid_out.nlon)
    return fail(DISCO_ERR_INVALID_ARG, "psi grids inconsistent with s");
  if (psi->grid_in.nlat < 2 || psi->grid_out.nlat < 2 || psi->grid_out.nlat > 65535 ||
      psi->grid_in.nlat > 65535)
    return fail(DISCO_ERR_UNSUPPORTED, "grid rows out of range [2, 65535]");
  return DISCO_OK;
}

}  // namespace disco

extern "C" int32_t disco_version(void) { return 100; }

extern "C" const char* disco_last_error(void) { return disco::g_last_error; }
