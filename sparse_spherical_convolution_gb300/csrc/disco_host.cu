// disco_host.cu -- host-buffer forms of the contractions, with the
// host<->device copies pipelined against the kernels.
//
// The contractions treat every (batch, channel) plane alike (the same psi
// for all of them), so the B*C planes split into blocks of 128 (one channel
// tile of the tensor-core kernels).  For block i:
//   copy stream A:  host -> device, into input slot i % 2
//   caller stream:  the contraction of the block, into output slot i % 2
//   copy stream B:  device -> host, out of output slot i % 2
// with events ordering each block's three steps and the reuse of a slot two
// blocks later.  So while block i computes, block i+1 arrives and block i-1
// leaves.  The two copy streams belong to the library (created once per
// device, non-blocking) and are shared by all calls, so two calls on two
// caller streams (a forward and a transpose, say) also overlap one's copies
// with the other's kernels.  The slots live in the caller's workspace.

#include <mutex>

#include "disco_internal.cuh"

namespace disco {
namespace {

constexpr int kHostBlock = 128;  // planes per block
constexpr int kMaxDevices = 64;

struct CopyStreams {
  cudaStream_t in = nullptr, out = nullptr;
  void* ctx = nullptr;  // the context the streams belong to
};
std::mutex g_copy_mu;
CopyStreams g_copy[kMaxDevices];

int copy_streams(CopyStreams* cs) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(DISCO_ERR_CUDA, "no current device for the copy streams");
  std::lock_guard<std::mutex> lock(g_copy_mu);
  CopyStreams& c = g_copy[dev];
  void* ctx = current_context();
  if (!ctx) {  // no context current on this thread yet: let the runtime make it current
    (void)cudaStreamQuery(nullptr);
    ctx = current_context();
  }
  // streams of a context that was reset are gone with it: make new ones (the
  // old handles are not destroyed, they no longer name anything)
  if (!c.in || (ctx && ctx != c.ctx)) {
    c.in = c.out = nullptr;
    if (cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking) != cudaSuccess) {
      c.in = c.out = nullptr;
      return fail(DISCO_ERR_CUDA, "copy stream creation failed");
    }
    c.ctx = current_context();
  }
  *cs = c;
  return DISCO_OK;
}

size_t align256h(size_t v) { return (v + 255) & ~(size_t)255; }

int elem_bytes(disco_dtype dt) { return dt == DISCO_F32 ? 4 : 2; }

// plane sizes (elements) of the input and output of one contraction
void planes(const disco_psi* psi, bool fwd, int64_t* in_plane, int64_t* out_plane) {
  const int64_t xin = (int64_t)psi->grid_in.nlat * psi->grid_in.nlon;
  const int64_t xout = (int64_t)psi->K * psi->grid_out.nlat * psi->grid_out.nlon;
  *in_plane = fwd ? xin : xout;
  *out_plane = fwd ? xout : xin;
}

size_t host_ws_bytes(const disco_psi* psi, int32_t B, int32_t C, bool fwd, disco_dtype dt) {
  int64_t ip, op;
  planes(psi, fwd, &ip, &op);
  const int64_t BC = (int64_t)B * C;
  const int64_t blk = BC < kHostBlock ? BC : kHostBlock;
  const size_t esz = (size_t)elem_bytes(dt);
  return 2 * (align256h((size_t)blk * ip * esz) + align256h((size_t)blk * op * esz));
}

int contract_host(bool fwd, const disco_psi* psi, const void* in_host, void* out_host, int32_t B, int32_t C,
                  disco_dtype dtype, void* workspace, size_t workspace_bytes, cudaStream_t st) {
  int rc = check_psi(psi);
  if (rc) return rc;
  if ((rc = check_device())) return rc;
  if (!in_host || !out_host) return fail(DISCO_ERR_INVALID_ARG, "null host pointer");
  if (B < 1 || C < 1) return fail(DISCO_ERR_INVALID_ARG, "B and C must be >= 1");
  if (dtype != DISCO_F32 && dtype != DISCO_BF16 && dtype != DISCO_F16)
    return fail(DISCO_ERR_UNSUPPORTED, "dtype");
  const size_t need = host_ws_bytes(psi, B, C, fwd, dtype);
  if (!workspace || workspace_bytes < need) return fail(DISCO_ERR_WORKSPACE, "workspace needs %zu bytes", need);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(DISCO_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if ((rc = check_dev_ptr(workspace, "workspace"))) return rc;
  CopyStreams cs;
  if ((rc = copy_streams(&cs))) return rc;
  int64_t ip, op;
  planes(psi, fwd, &ip, &op);
  const int64_t BC = (int64_t)B * C;
  const int64_t blk = BC < kHostBlock ? BC : kHostBlock;
  const int64_t nblk = (BC + blk - 1) / blk;
  const size_t esz = (size_t)elem_bytes(dtype);
  const size_t in_slot = align256h((size_t)blk * ip * esz), out_slot = align256h((size_t)blk * op * esz);
  char* ws = (char*)workspace;
  char* in_buf[2] = {ws, ws + in_slot};
  char* out_buf[2] = {ws + 2 * in_slot, ws + 2 * in_slot + out_slot};
  const char* src = (const char*)in_host;
  char* dst = (char*)out_host;

  // events: start (caller stream), and per block copied-in, computed, copied-out
  auto mk = [](cudaEvent_t* e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
  cudaEvent_t start;
  if (!mk(&start)) return fail(DISCO_ERR_CUDA, "event creation failed");
  const int64_t nev = 3 * nblk;
  cudaEvent_t* ev = new cudaEvent_t[nev];
  int64_t made = 0;
  bool ok = true;
  for (; made < nev && ok; ++made) ok = mk(&ev[made]);
  if (!ok) --made;
  auto cleanup = [&]() {  // destruction waits for recorded events to complete
    cudaEventDestroy(start);
    for (int64_t i = 0; i < made; ++i) cudaEventDestroy(ev[i]);
    delete[] ev;
  };
  if (!ok) {
    cleanup();
    return fail(DISCO_ERR_CUDA, "event creation failed");
  }
  cudaEvent_t *ev_in = ev, *ev_k = ev + nblk, *ev_out = ev + 2 * nblk;
  auto cu = [&](cudaError_t e, const char* what) {
    if (e != cudaSuccess && rc == DISCO_OK) rc = fail(DISCO_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return e == cudaSuccess;
  };
  // the copies start after the caller's earlier work on `st`
  if (cu(cudaEventRecord(start, st), "record") && cu(cudaStreamWaitEvent(cs.in, start, 0), "wait") &&
      cu(cudaStreamWaitEvent(cs.out, start, 0), "wait")) {
    for (int64_t i = 0; i < nblk && rc == DISCO_OK; ++i) {
      const int sl = (int)(i & 1);
      const int64_t n = (BC - i * blk) < blk ? (BC - i * blk) : blk;
      if (i >= 2 && !cu(cudaStreamWaitEvent(cs.in, ev_k[i - 2], 0), "wait")) break;  // input slot free
      if (!cu(cudaMemcpyAsync(in_buf[sl], src + (size_t)(i * blk) * ip * esz, (size_t)n * ip * esz,
                              cudaMemcpyHostToDevice, cs.in),
              "host-to-device copy") ||
          !cu(cudaEventRecord(ev_in[i], cs.in), "record") || !cu(cudaStreamWaitEvent(st, ev_in[i], 0), "wait"))
        break;
      if (i >= 2 && !cu(cudaStreamWaitEvent(st, ev_out[i - 2], 0), "wait")) break;  // output slot free
      const int crc = fwd ? disco_fwd(psi, in_buf[sl], out_buf[sl], 1, (int32_t)n, dtype, st)
                          : disco_bwd(psi, in_buf[sl], out_buf[sl], 1, (int32_t)n, dtype, st);
      if (crc) {
        rc = crc;
        break;
      }
      if (!cu(cudaEventRecord(ev_k[i], st), "record") || !cu(cudaStreamWaitEvent(cs.out, ev_k[i], 0), "wait") ||
          !cu(cudaMemcpyAsync(dst + (size_t)(i * blk) * op * esz, out_buf[sl], (size_t)n * op * esz,
                              cudaMemcpyDeviceToHost, cs.out),
              "device-to-host copy") ||
          !cu(cudaEventRecord(ev_out[i], cs.out), "record"))
        break;
    }
    // the caller's stream continues once the last block is back on the host
    // (the copy-out stream runs the blocks in order)
    if (rc == DISCO_OK) cu(cudaStreamWaitEvent(st, ev_out[nblk - 1], 0), "wait");
  }
  cleanup();
  return rc;
}

}  // namespace
}  // namespace disco

using namespace disco;

extern "C" size_t disco_host_workspace_bytes(const disco_psi* psi, int32_t B, int32_t C, int32_t forward,
                                             disco_dtype dtype) {
  if (!psi || B < 1 || C < 1) return 0;
  return host_ws_bytes(psi, B, C, forward != 0, dtype);
}

extern "C" int disco_fwd_host(const disco_psi* psi, const void* x_host, void* X_host, int32_t B, int32_t C,
                              disco_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
  disco::NvtxScope nvtx_scope("disco_fwd_host");
  return contract_host(true, psi, x_host, X_host, B, C, dtype, workspace, workspace_bytes, (cudaStream_t)stream);
}

extern "C" int disco_bwd_host(const disco_psi* psi, const void* G_host, void* gx_host, int32_t B, int32_t C,
                              disco_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
  disco::NvtxScope nvtx_scope("disco_bwd_host");
  return contract_host(false, psi, G_host, gx_host, B, C, dtype, workspace, workspace_bytes, (cudaStream_t)stream);
}
