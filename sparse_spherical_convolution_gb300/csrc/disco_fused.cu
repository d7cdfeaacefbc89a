// disco_fused.cu -- placeholder until the tcgen05 fused kernels land.
#include "disco_internal.cuh"

extern "C" int disco_fused_conv(const disco_psi* psi, const void*, const void*, void*, int32_t,
                                int32_t, int32_t, disco_dtype, void*) {
  if (int st = disco::check_psi(psi)) return st;
  return disco::fail(DISCO_ERR_UNSUPPORTED, "fused convolution not built yet");
}

extern "C" size_t disco_fused_conv_bwd_input_workspace_bytes(const disco_psi*, int32_t, int32_t,
                                                             disco_dtype) {
  return 0;
}

extern "C" int disco_fused_conv_bwd_input(const disco_psi* psi, const void*, const void*, void*,
                                          int32_t, int32_t, int32_t, disco_dtype, void*, size_t,
                                          void*) {
  if (int st = disco::check_psi(psi)) return st;
  return disco::fail(DISCO_ERR_UNSUPPORTED, "fused input gradient not built yet");
}
