// Status helpers and the uniform generator shared by every entry point.
#include "common.cuh"
#include "internal.h"

namespace sv {

// A bounded wait on something nothing completes, with the waiting code of
// the verifier kernels: kind 0 waits on a shared-memory mbarrier phase (the
// TMA rings' waits), kind 1 polls a global word (the streaming verifier's
// producers). The wait gives up after limit_ns and records SPEC_ERR_TIMEOUT.
__global__ void k_wait_selftest(WsHeader *hdr, int kind, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x != 0) return;
  bool done;
  if (kind == 0) {
    mbar_init(&bar, 1);   // one arrival completes phase 0; none comes
    abort = 0;
    fence_mbar_init();
    done = mbar_wait_bounded(&bar, 0, &abort, limit_ns);
  } else {
    const volatile int *word = &hdr->pad[0];   // zero, and nothing writes it
    done = poll_bounded([&]() -> int { return *word != 0; }, 0, limit_ns) != 0;
  }
  if (!done) set_status(hdr, SPEC_ERR_TIMEOUT, kind);
}

// Reads the word just past the first 256 bytes of the workspace, which the
// caller allocated but which is not registered as the call's: in the
// checked build the access is refused and reported (SPEC_ERR_BOUNDS).
__global__ void k_check_selftest(WsHeader *hdr) {
  const int *beyond = reinterpret_cast<const int *>(reinterpret_cast<const char *>(hdr) + 256);
  const int v = GLD(beyond);
  if (v == 0x5eed) hdr->pad[1] = v;   // keeps the load
}

__global__ void k_uniforms(uint64_t seed, const int32_t *b, const int32_t *pos,
                           const int32_t *stream_id, int n, float *out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n)
    GST(out + i, uniform24(seed, (uint32_t)GLD(b + i), (uint32_t)GLD(pos + i),
                           (uint32_t)GLD(stream_id + i)));
}

#ifdef SPEC_CHECKED
static thread_local CheckTable t_check;
CheckTable &host_check_table() { return t_check; }
void check_begin(WsHeader *hdr) {
  t_check.n = 0;
  t_check.hdr = hdr;
}
void check_add(const void *p, unsigned long long bytes) {
  if (p == nullptr || bytes == 0 || t_check.n >= CHECK_RANGES) return;
  t_check.lo[t_check.n] = (unsigned long long)p;
  t_check.hi[t_check.n] = (unsigned long long)p + bytes;
  ++t_check.n;
}
int check_read_int(const int32_t *dev, cudaStream_t st, int *out) {
  if (cudaMemcpyAsync(out, dev, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}
#endif

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
    case SPEC_ERR_BOUNDS: return "SPEC_ERR_BOUNDS";
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
#ifdef SPEC_CHECKED
  check_begin(nullptr);   // no workspace: an access outside the buffers is skipped unreported
  check_add(b, n * 4ull);
  check_add(pos, n * 4ull);
  check_add(stream_id, n * 4ull);
  check_add(out, n * 4ull);
#endif
  if (check_upload(reinterpret_cast<cudaStream_t>(stream)) != SPEC_OK) return SPEC_ERR_CUDA;
  k_uniforms<<<(n + 255) / 256, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      seed, b, pos, stream_id, n, out);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

extern "C" int spec_wait_selftest(int kind, unsigned long long limit_ns, void *workspace,
                                  spec_stream_t stream) {
  if (kind != 0 && kind != 1) return SPEC_ERR_INVALID_ARG;
  if (limit_ns == 0 || limit_ns > 10000000000ull) return SPEC_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256)) return SPEC_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  WsHeader *hdr = static_cast<WsHeader *>(workspace);
  if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st) != cudaSuccess) return SPEC_ERR_CUDA;
#ifdef SPEC_CHECKED
  check_begin(hdr);
  check_add(workspace, sizeof(WsHeader));
#endif
  if (check_upload(st) != SPEC_OK) return SPEC_ERR_CUDA;
  k_wait_selftest<<<1, 32, 0, st>>>(hdr, kind, limit_ns);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

extern "C" int spec_check_selftest(void *workspace, size_t ws_bytes, spec_stream_t stream) {
#ifndef SPEC_CHECKED
  (void)workspace;
  (void)ws_bytes;
  (void)stream;
  return SPEC_ERR_UNSUPPORTED;
#else
  if (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < 512) return SPEC_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  WsHeader *hdr = static_cast<WsHeader *>(workspace);
  if (cudaMemsetAsync(hdr, 0, sizeof(WsHeader), st) != cudaSuccess) return SPEC_ERR_CUDA;
  check_begin(hdr);
  check_add(workspace, sizeof(WsHeader));   // the header only
  if (check_upload(st) != SPEC_OK) return SPEC_ERR_CUDA;
  k_check_selftest<<<1, 1, 0, st>>>(hdr);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
#endif
}

extern "C" int spec_profile_row_pass(void *before, void *after) {
  set_row_pass_events(reinterpret_cast<cudaEvent_t>(before), reinterpret_cast<cudaEvent_t>(after));
  return SPEC_OK;
}

extern "C" int spec_profile_pending(void) { return row_pass_events_pending() ? 1 : 0; }
