// Status helpers and the uniform generator shared by every entry point.
#include "common.cuh"
#include "internal.h"

namespace sv {

__global__ void k_uniforms(uint64_t seed, const int32_t *b, const int32_t *pos,
                           const int32_t *stream_id, int n, float *out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = uniform24(seed, (uint32_t)b[i], (uint32_t)pos[i], (uint32_t)stream_id[i]);
}

}  // namespace sv

using namespace sv;

extern "C" const char *spec_status_string(int status) {
  switch (status) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG";
    case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
    case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
    case SPEC_ERR_TIMEOUT: return "SPEC_ERR_TIMEOUT";
    default: return "SPEC_ERR_UNKNOWN";
  }
}

extern "C" int spec_get_status(const void *workspace, spec_stream_t stream, int *device_status) {
  if (workspace == nullptr || device_status == nullptr || !aligned(workspace, 256))
    return SPEC_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SPEC_ERR_CUDA;
  *device_status = v;
  return SPEC_OK;
}

extern "C" int spec_uniforms(uint64_t seed, const int32_t *b, const int32_t *pos,
                             const int32_t *stream_id, int n, float *out, spec_stream_t stream) {
  if (n < 0) return SPEC_ERR_INVALID_ARG;
  if (n == 0) return SPEC_OK;
  if (!b || !pos || !stream_id || !out) return SPEC_ERR_INVALID_ARG;
  k_uniforms<<<(n + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      seed, b, pos, stream_id, n, out);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

extern "C" int spec_profile_row_pass(void *before, void *after) {
  set_row_pass_events(reinterpret_cast<cudaEvent_t>(before), reinterpret_cast<cudaEvent_t>(after));
  return SPEC_OK;
}
