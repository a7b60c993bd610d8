// One expansion level of RheoSampling dynamic-tree construction for a batch
// of trees ("RheoSampling 2026": §2 "Dual-Identity Decoupling", §3
// "Parameter Kendali Rheostat & Optimasi Sparse Top-128", §7 "Rekomendasi").
//
// Every frontier row goes through the top-128 select of topk.cu at the
// tree's temperature (its probabilities are the probe's true sampling law
// q~), and the select's block then expands the row from the 128 survivors
// still in shared memory (topk.cu, rheo_epilogue):
//   - the unscaled ranking law q = softmax(z) over the survivors (§7:
//     construction runs without temperature), and their ranks best first
//     (logit descending, ties to the lower id);
//   - the probe, drawn from q~ by inverse CDF in ascending id at
//     u(seed, f, level, 3);
//   - the children in slot order: the m best tokens other than the probe,
//     the probe, then the next best up to K (§3, the rheostat m). The probe's
//     proxy probability is q(x_{m+1}) + eps (m = 0: q(x_1) + eps as on the
//     page); a deterministic child's proxy is its own q. A child's path score
//     is the frontier node's score + ln q_proxy.
// Then one CTA per tree sorts its candidates by (score descending, candidate
// index ascending) in shared memory and keeps the first n_keep (the global
// pruning of §2).
//
// The select streams every frontier row once from HBM and dominates the call.
#include "common.cuh"
#include "internal.h"

#include <algorithm>
#include <climits>

namespace sv {
namespace {

constexpr int RH_SELECT_THREADS = 256;

struct RheoArgs {
  const int32_t *cu;
  const float *fscore;
  const float *temp;
  int B, F, K, n_keep, cap;
  const float *score;
  int32_t *keep;
  WsHeader *hdr;
};

__global__ void k_rheo_validate(RheoArgs a) {
  if (threadIdx.x == 0) {
    a.hdr->status = 0;
    a.hdr->detail = -1;
  }
  __syncthreads();
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
    const int n = GLD(a.cu + (b + 1)) - GLD(a.cu + (b));
    const float T = GLD(a.temp + (b));
    if (n < 0 || !(T >= 0.f) || !isfinite(T)) set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);
    else if ((long long)n * a.K > a.cap) set_status(a.hdr, SPEC_ERR_UNSUPPORTED, b);
  }
  if (threadIdx.x == 0 && (GLD(a.cu + (0)) != 0 || GLD(a.cu + (a.B)) != a.F))
    set_status(a.hdr, SPEC_ERR_INVALID_ARG, a.B);
  for (int f = threadIdx.x; f < a.F; f += blockDim.x) {
    const float s = GLD(a.fscore + (f));
    if (isnan(s) || s == INFINITY) set_status(a.hdr, SPEC_ERR_INVALID_ARG, f);
  }
}

// Order-preserving map of a float to uint32 (ascending).
__device__ __forceinline__ uint32_t ordered_bits(float s) {
  const uint32_t u = __float_as_uint(s + 0.f);   // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(RH_SELECT_THREADS) k_rheo_select(RheoArgs a, int P_max) {
  extern __shared__ unsigned long long sk[];
  const int b = blockIdx.x;
  int32_t *out = a.keep + (size_t)b * a.n_keep;
  const int lo = GLD(a.cu + (b)), hi = GLD(a.cu + (b + 1));
  const bool ok = a.hdr->status == 0 && lo >= 0 && hi <= a.F && lo <= hi &&
                  (long long)(hi - lo) * a.K <= P_max;
  if (!ok) {
    for (int i = threadIdx.x; i < a.n_keep; i += blockDim.x) GST(out + i, -1);
    return;
  }
  const int n = (hi - lo) * a.K;
  const long long base = (long long)lo * a.K;
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = threadIdx.x; i < P; i += blockDim.x)
    sk[i] = i < n ? ((unsigned long long)(~ordered_bits(GLD(a.score + (base + i)))) << 32) | (uint32_t)i
                  : ~0ull;
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += blockDim.x) {
        const int ij = i ^ j;
        if (ij > i) {
          const bool up = (i & k) == 0;
          const unsigned long long x = sk[i], y = sk[ij];
          if ((x > y) == up) {
            sk[i] = y;
            sk[ij] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < a.n_keep; i += blockDim.x)
    GST(out + i, i < n ? (int32_t)(base + (long long)(uint32_t)(sk[i] & 0xffffffffull)) : -1);
}

// the status header, then the top-128 select's candidate lists
inline size_t rheo_ws_bytes(int F, int V) { return 256 + topk_list_bytes_for(F, V); }

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" size_t spec_rheo_expand_workspace(int F, int V) {
  if (F < 0 || F > (1 << 24) || V <= 0 || V > SPEC_MAX_V) return 0;
  return rheo_ws_bytes(F, V);
}

extern "C" int spec_rheo_expand(const void *draft, int ddt, const int32_t *cu_frontier,
                                const float *frontier_score, const float *temperature, int B,
                                int F, int V, int K, int m, float eps, int n_keep,
                                uint64_t seed, int level, int32_t *child_token,
                                float *child_qproxy, float *child_qtrue, float *child_score,
                                int32_t *keep, void *workspace, size_t ws_bytes,
                                spec_stream_t stream) {
  if (B < 0 || F < 0 || F > (1 << 24) || V <= 0 || V > SPEC_MAX_V) return SPEC_ERR_INVALID_ARG;
  if (ddt != SPEC_F32 && ddt != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (K < 1 || K > SPEC_TOPK || K > V || m < 0 || m >= K || n_keep < 0) return SPEC_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || !isfinite(eps) || level < 0 || level >= (1 << 24)) return SPEC_ERR_INVALID_ARG;
  if (n_keep > SPEC_RHEO_MAX_CANDIDATES) return SPEC_ERR_UNSUPPORTED;
  if (cu_frontier == nullptr || (B > 0 && temperature == nullptr)) return SPEC_ERR_INVALID_ARG;
  if (F > 0 && (draft == nullptr || frontier_score == nullptr || child_token == nullptr ||
                child_score == nullptr))
    return SPEC_ERR_INVALID_ARG;
  if (B > 0 && n_keep > 0 && keep == nullptr) return SPEC_ERR_INVALID_ARG;
  if (!aligned(draft, 16) || !aligned(cu_frontier, 4) || !aligned(frontier_score, 4) ||
      !aligned(temperature, 4) || !aligned(child_token, 4) || !aligned(child_qproxy, 4) ||
      !aligned(child_qtrue, 4) || !aligned(child_score, 4) || !aligned(keep, 4))
    return SPEC_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < rheo_ws_bytes(F, V))
    return SPEC_ERR_WORKSPACE;

  RheoArgs a{};
  a.cu = cu_frontier;
  a.fscore = frontier_score;
  a.temp = temperature;
  a.B = B;
  a.F = F;
  a.K = K;
  a.n_keep = n_keep;
  a.cap = SPEC_RHEO_MAX_CANDIDATES;
  a.score = child_score;
  a.keep = keep;
  a.hdr = static_cast<WsHeader *>(workspace);
  RheoEpi epi{};
  epi.fscore = frontier_score;
  epi.K = K;
  epi.m = m;
  epi.eps = eps;
  epi.seed = seed;
  epi.level = level;
  epi.token = child_token;
  epi.qproxy = child_qproxy;
  epi.qtrue = child_qtrue;
  epi.score = child_score;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
#ifdef SPEC_CHECKED
  check_begin(a.hdr);
  check_add(workspace, rheo_ws_bytes(F, V));
  check_add(draft, (unsigned long long)F * V * (ddt == SPEC_BF16 ? 2 : 4));
  check_add(cu_frontier, (B + 1) * 4ull);
  check_add(frontier_score, F * 4ull);
  check_add(temperature, B * 4ull);
  check_add(child_token, (unsigned long long)F * K * 4);
  check_add(child_qproxy, (unsigned long long)F * K * 4);
  check_add(child_qtrue, (unsigned long long)F * K * 4);
  check_add(child_score, (unsigned long long)F * K * 4);
  check_add(keep, (unsigned long long)B * n_keep * 4);
#endif
  if (check_upload(st) != SPEC_OK) return SPEC_ERR_CUDA;
  k_rheo_validate<<<1, 256, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (F > 0) {
    // the top-128 select with its expansion epilogue streams every frontier
    // row and dominates the call: profiling events, if registered, bracket
    // its launch that reads the rows
    cudaEvent_t before, after;
    take_row_pass_events(&before, &after);
    void *lists = rheo_ws_bytes(F, V) > 256 ? static_cast<char *>(workspace) + 256 : nullptr;
    const int rc = launch_topk128(draft, ddt, F, V, cu_frontier, temperature, B, nullptr,
                                  nullptr, a.hdr, st, &epi, lists, before, after);
    if (rc != SPEC_OK) return rc;
  }
  if (B > 0 && n_keep > 0) {
    // shared memory for the largest tree the call can hold
    const long long most = std::min<long long>((long long)F * K, SPEC_RHEO_MAX_CANDIDATES);
    int P = 1;
    while (P < most) P <<= 1;
    const size_t smem = sizeof(unsigned long long) * (size_t)P;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(k_rheo_select, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return SPEC_ERR_CUDA;
    k_rheo_select<<<B, RH_SELECT_THREADS, smem, st>>>(a, P);
    if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}
