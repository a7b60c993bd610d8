// One expansion level of RheoSampling dynamic-tree construction for a batch
// of trees ("RheoSampling 2026": §2 "Dual-Identity Decoupling", §3
// "Parameter Kendali Rheostat & Optimasi Sparse Top-128", §7 "Rekomendasi").
//
// Every frontier row is cut to its 128 largest draft logits (the top-128
// select of topk.cu, at the tree's temperature: its probabilities are the
// probe's true sampling law q~). Then one warp per frontier row:
//   - gathers the 128 surviving logits, forms the unscaled ranking law
//     q = softmax(z) over them (§7: construction runs without temperature)
//     and ranks them best first (logit descending, ties to the lower id);
//   - draws the probe from q~ by inverse CDF in ascending id at
//     u(seed, f, level, 3);
//   - writes the children in slot order: the m best tokens other than the
//     probe, the probe, then the next best up to K (§3, the rheostat m). The
//     probe's proxy probability is q(x_{m+1}) + eps (m = 0: q(x_1) + eps as
//     on the page); a deterministic child's proxy is its own q. A child's
//     path score is the frontier node's score + ln q_proxy.
// Finally one CTA per tree sorts its candidates by (score descending,
// candidate index ascending) in shared memory and keeps the first n_keep
// (the global pruning of §2).
//
// The top-128 select streams every frontier row once from HBM and dominates
// the call; the rest reads 128 logits and 1 KB of top-128 output per row.
#include "common.cuh"
#include "internal.h"

#include <algorithm>
#include <climits>

namespace sv {
namespace {

constexpr int RH_WARPS = 8;               // frontier rows per CTA, one per warp
constexpr int RH_SELECT_THREADS = 1024;
constexpr uint32_t STREAM_PROBE = 3;

struct RheoArgs {
  const char *draft;
  int dtype;
  long long row_bytes;
  const int32_t *cu;
  const float *fscore;
  const float *temp;
  int B, F, V, K, m, n_keep, cap;
  float eps;
  uint64_t seed;
  int level;
  const int32_t *tk_idx;
  const float *tk_prob;
  int32_t *token;
  float *qproxy, *qtrue, *score;
  int32_t *keep;
  WsHeader *hdr;
};

// Register-array element t (t in 0..3) without local-memory indexing.
template <class T>
__device__ __forceinline__ T pick4(const T (&v)[4], int t) {
  return t == 0 ? v[0] : t == 1 ? v[1] : t == 2 ? v[2] : v[3];
}

__global__ void k_rheo_validate(RheoArgs a) {
  if (threadIdx.x == 0) {
    a.hdr->status = 0;
    a.hdr->detail = -1;
  }
  __syncthreads();
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
    const int n = a.cu[b + 1] - a.cu[b];
    const float T = a.temp[b];
    if (n < 0 || !(T >= 0.f) || !isfinite(T)) set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);
    else if ((long long)n * a.K > a.cap) set_status(a.hdr, SPEC_ERR_UNSUPPORTED, b);
  }
  if (threadIdx.x == 0 && (a.cu[0] != 0 || a.cu[a.B] != a.F))
    set_status(a.hdr, SPEC_ERR_INVALID_ARG, a.B);
  for (int f = threadIdx.x; f < a.F; f += blockDim.x) {
    const float s = a.fscore[f];
    if (isnan(s) || s == INFINITY) set_status(a.hdr, SPEC_ERR_INVALID_ARG, f);
  }
}

__global__ void __launch_bounds__(32 * RH_WARPS) k_rheo_children(RheoArgs a) {
  if (a.hdr->status != 0) return;
  const int lane = threadIdx.x & 31;
  const int f = blockIdx.x * RH_WARPS + (threadIdx.x >> 5);
  if (f >= a.F) return;
  const unsigned FULL = 0xffffffffu;

  // slots 4*lane .. 4*lane+3 of the top-128 output, ascending id, -1 padded
  const int4 id4 = reinterpret_cast<const int4 *>(a.tk_idx + (size_t)f * SPEC_TOPK)[lane];
  const float4 p4 = reinterpret_cast<const float4 *>(a.tk_prob + (size_t)f * SPEC_TOPK)[lane];
  // ids outside [0, V) (padding when V < 128) are empty slots
  const int id[4] = {(unsigned)id4.x < (unsigned)a.V ? id4.x : -1,
                     (unsigned)id4.y < (unsigned)a.V ? id4.y : -1,
                     (unsigned)id4.z < (unsigned)a.V ? id4.z : -1,
                     (unsigned)id4.w < (unsigned)a.V ? id4.w : -1};
  const float qt[4] = {p4.x, p4.y, p4.z, p4.w};
  const char *row = a.draft + (size_t)f * a.row_bytes;
  float z[4];
  int key[4];
  float mz = -INFINITY;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    z[t] = id[t] >= 0 ? load_elem(row, a.dtype, id[t]) : -INFINITY;
    key[t] = id[t] >= 0 ? id[t] : INT_MAX;
    mz = fmaxf(mz, z[t]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mz = fmaxf(mz, __shfl_xor_sync(FULL, mz, o));

  // unscaled ranking law over the survivors
  float e[4], S = 0.f;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    e[t] = z[t] > -INFINITY ? expf(z[t] - mz) : 0.f;
    S += e[t];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(FULL, S, o);
  float q[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) q[t] = e[t] / S;

  // rank best first: logit descending, ties (and -inf) to the lower id,
  // padding slots last
  int rank[4] = {0, 0, 0, 0};
  for (int src = 0; src < 32; ++src) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float zj = __shfl_sync(FULL, z[u], src);
      const int kj = __shfl_sync(FULL, key[u], src);
#pragma unroll
      for (int t = 0; t < 4; ++t) rank[t] += (zj > z[t] || (zj == z[t] && kj < key[t])) ? 1 : 0;
    }
  }

  // probe: inverse CDF over q~ in ascending id (inclusive prefix sums)
  float c[4];
  c[0] = qt[0];
  c[1] = c[0] + qt[1];
  c[2] = c[1] + qt[2];
  c[3] = c[2] + qt[3];
  float incl = c[3];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += y;
  }
  float excl = __shfl_up_sync(FULL, incl, 1);
  if (lane == 0) excl = 0.f;
#pragma unroll
  for (int t = 0; t < 4; ++t) c[t] += excl;
  const float Z = __shfl_sync(FULL, c[3], 31);
  const float tu = uniform24(a.seed, (uint32_t)f, (uint32_t)a.level, STREAM_PROBE) * Z;
  const int first_hit = tu < c[0] ? 0 : tu < c[1] ? 1 : tu < c[2] ? 2 : tu < c[3] ? 3 : 4;
  const unsigned hit_lanes = __ballot_sync(FULL, first_hit < 4);
  int ps;                                   // the probe's slot
  if (hit_lanes) {
    const int L = __ffs(hit_lanes) - 1;
    ps = 4 * L + __shfl_sync(FULL, first_hit, L);
  } else {                                  // rounding: the last slot with weight
    const int last = qt[3] > 0.f ? 3 : qt[2] > 0.f ? 2 : qt[1] > 0.f ? 1 : qt[0] > 0.f ? 0 : -1;
    const unsigned pos_lanes = __ballot_sync(FULL, last >= 0);
    const int H = pos_lanes ? 31 - __clz(pos_lanes) : 0;
    ps = 4 * H + max(__shfl_sync(FULL, last, H), 0);
  }
  const int probe_id = __shfl_sync(FULL, pick4(id, ps & 3), ps >> 2);
  const int probe_rank = __shfl_sync(FULL, pick4(rank, ps & 3), ps >> 2);
  const float probe_qt = __shfl_sync(FULL, pick4(qt, ps & 3), ps >> 2);

  // q(x_{m+1}): the survivor of rank m (valid ranks are unique)
  int found = -1;
#pragma unroll
  for (int t = 0; t < 4; ++t)
    if (id[t] >= 0 && rank[t] == a.m) found = t;
  const unsigned fl = __ballot_sync(FULL, found >= 0);
  float q_m = 0.f;
  if (fl) {
    const int L = __ffs(fl) - 1;
    q_m = __shfl_sync(FULL, found >= 0 ? pick4(q, found) : 0.f, L);
  }

  const size_t out0 = (size_t)f * a.K;
  const float fs = a.fscore[f];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    if (id[t] < 0 || id[t] == probe_id) continue;
    const int r = rank[t] - (probe_rank < rank[t] ? 1 : 0);
    if (r >= a.K - 1) continue;
    const int slot = r < a.m ? r : r + 1;
    a.token[out0 + slot] = id[t];
    if (a.qproxy) a.qproxy[out0 + slot] = q[t];
    if (a.qtrue) a.qtrue[out0 + slot] = qt[t];
    a.score[out0 + slot] = fs + logf(q[t]);
  }
  if (lane == 0) {
    const float pr = q_m + a.eps;
    a.token[out0 + a.m] = probe_id;
    if (a.qproxy) a.qproxy[out0 + a.m] = pr;
    if (a.qtrue) a.qtrue[out0 + a.m] = probe_qt;
    a.score[out0 + a.m] = fs + logf(pr);
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
  const int lo = a.cu[b], hi = a.cu[b + 1];
  const bool ok = a.hdr->status == 0 && lo >= 0 && hi <= a.F && lo <= hi &&
                  (long long)(hi - lo) * a.K <= P_max;
  if (!ok) {
    for (int i = threadIdx.x; i < a.n_keep; i += blockDim.x) out[i] = -1;
    return;
  }
  const int n = (hi - lo) * a.K;
  const long long base = (long long)lo * a.K;
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = threadIdx.x; i < P; i += blockDim.x)
    sk[i] = i < n ? ((unsigned long long)(~ordered_bits(a.score[base + i])) << 32) | (uint32_t)i
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
    out[i] = i < n ? (int32_t)(base + (long long)(uint32_t)(sk[i] & 0xffffffffull)) : -1;
}

inline size_t rheo_ws_bytes(int F) {
  return 256 + align256(sizeof(int32_t) * (size_t)F * SPEC_TOPK) +
         align256(sizeof(float) * (size_t)F * SPEC_TOPK);
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" size_t spec_rheo_expand_workspace(int F, int V) {
  if (F < 0 || F > (1 << 24) || V <= 0 || V > SPEC_MAX_V) return 0;
  return rheo_ws_bytes(F);
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
  if (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < rheo_ws_bytes(F))
    return SPEC_ERR_WORKSPACE;

  char *ws = static_cast<char *>(workspace);
  RheoArgs a{};
  a.draft = static_cast<const char *>(draft);
  a.dtype = ddt;
  a.row_bytes = (long long)V * (ddt == SPEC_BF16 ? 2 : 4);
  a.cu = cu_frontier;
  a.fscore = frontier_score;
  a.temp = temperature;
  a.B = B;
  a.F = F;
  a.V = V;
  a.K = K;
  a.m = m;
  a.n_keep = n_keep;
  a.cap = SPEC_RHEO_MAX_CANDIDATES;
  a.eps = eps;
  a.seed = seed;
  a.level = level;
  a.hdr = reinterpret_cast<WsHeader *>(ws);
  int32_t *tk_idx = reinterpret_cast<int32_t *>(ws + 256);
  float *tk_prob = reinterpret_cast<float *>(
      ws + 256 + align256(sizeof(int32_t) * (size_t)F * SPEC_TOPK));
  a.tk_idx = tk_idx;
  a.tk_prob = tk_prob;
  a.token = child_token;
  a.qproxy = child_qproxy;
  a.qtrue = child_qtrue;
  a.score = child_score;
  a.keep = keep;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  k_rheo_validate<<<1, 256, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (F > 0) {
    // the top-128 select streams every frontier row and dominates the call:
    // profiling events, if registered, bracket it
    cudaEvent_t before, after;
    take_row_pass_events(&before, &after);
    if (before && cudaEventRecord(before, st) != cudaSuccess) return SPEC_ERR_CUDA;
    const int rc = launch_topk128(draft, ddt, F, V, cu_frontier, temperature, B, tk_idx,
                                  tk_prob, a.hdr, st);
    if (rc != SPEC_OK) return rc;
    if (after && cudaEventRecord(after, st) != cudaSuccess) return SPEC_ERR_CUDA;
    k_rheo_children<<<(F + RH_WARPS - 1) / RH_WARPS, 32 * RH_WARPS, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
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
