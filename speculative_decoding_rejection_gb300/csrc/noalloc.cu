// Linear verification for callers that cannot hand the library any scratch.
//
// spec_verify_linear() needs a caller-provided device workspace. Some callers
// cannot obtain one: serving engines that reserve nearly all of HBM for their
// KV cache when they start (a later cudaMalloc fails, or has to evict cache),
// and decode loops that must not call cudaMalloc/cudaFree because those calls
// synchronise the whole device. This entry point takes the same inputs and
// outputs but keeps its scratch in a fixed array compiled into the library.
//
// Properties of that array:
//   - SPEC_NOALLOC_SCRATCH_BYTES (16 MiB) per GPU, reserved on every GPU that
//     loads the library and held until the process exits;
//   - shared by all calls on a device and left holding the last call's
//     contents; the header words that must start at zero (status, work
//     counters) are cleared by a cudaMemsetAsync on the call's stream before
//     its first kernel, and everything else is written before it is read
//     within the call;
//   - calls whose work overlaps on the GPU (different streams, or different
//     host threads, without ordering between them) race on it; order them on
//     one stream or with events.
// The first call on each device looks up the array's device address with
// cudaGetSymbolAddress() (with that device current); make that first call
// before any stream capture. The address belongs to the device's context: a
// call made after cudaDeviceReset (a new context) looks it up again, so make
// the first call after a reset before any stream capture too. Nothing here
// calls cudaMalloc, cudaFree or an allocating library routine.
#include <cuda.h>   // context types only: the driver calls are resolved at run time

#include <mutex>

#include "common.cuh"
#include "internal.h"

static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchAddr {
  void *addr;                  // device address of the array in that context
  unsigned long long ctx_id;   // the context it was looked up in
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Unique id of the current thread's context (ids are never reused within a
// process, so a reset device's new context has a new one). Called with
// g_scratch_mu held.
int current_context_id(unsigned long long *id) {
  if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr) {
    void *f0 = nullptr, *f1 = nullptr;
    cudaDriverEntryPointQueryResult q0, q1;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 12000, cudaEnableDefault, &q0) !=
            cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &q1) !=
            cudaSuccess ||
        q0 != cudaDriverEntryPointSuccess || q1 != cudaDriverEntryPointSuccess)
      return SPEC_ERR_CUDA;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f0);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f1);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return SPEC_ERR_CUDA;
  return g_ctx_get_id(ctx, id) == CUDA_SUCCESS ? SPEC_OK : SPEC_ERR_CUDA;
}

// Device address of g_noalloc_scratch on the current device, looked up once
// per device context.
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SPEC_ERR_UNSUPPORTED;
  // makes the device's primary context current on this thread (and creates
  // it if this thread has not used the device yet)
  if (cudaSetDevice(dev) != cudaSuccess) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long ctx = 0;
  const int rc = current_context_id(&ctx);
  if (rc != SPEC_OK) return rc;
  ScratchAddr &s = g_scratch_addr[dev];
  if (s.addr == nullptr || s.ctx_id != ctx) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return SPEC_ERR_CUDA;
    s.addr = p;
    s.ctx_id = ctx;
  }
  *out = s.addr;
  return SPEC_OK;
}
}  // namespace

extern "C" int spec_verify_linear_noalloc(const void *target, int tdt, const void *draft,
                                          int ddt, int dk, const int32_t *draft_idx,
                                          const int32_t *draft_tokens,
                                          const int32_t *cu_draft, const float *temperature,
                                          int B, int V, int max_k, uint64_t seed, int rule,
                                          int32_t *out_tokens, int32_t *out_accepted,
                                          float *out_pq, int32_t *out_status,
                                          spec_stream_t stream) {
  const size_t need = spec_verify_linear_workspace(B, max_k, V, rule);
  if (need == 0) return SPEC_ERR_INVALID_ARG;
  if (need > (size_t)SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_ERR_UNSUPPORTED;
  if (out_status != nullptr && !sv::aligned(out_status, 4)) return SPEC_ERR_INVALID_ARG;
  void *scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != SPEC_OK) return rc;
  rc = spec_verify_linear(target, tdt, draft, ddt, dk, draft_idx, draft_tokens, cu_draft,
                          temperature, B, V, max_k, seed, rule, out_tokens, out_accepted, out_pq,
                          scratch, (size_t)SPEC_NOALLOC_SCRATCH_BYTES, stream);
  if (rc != SPEC_OK) return rc;
  if (out_status != nullptr &&
      cudaMemcpyAsync(out_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}
