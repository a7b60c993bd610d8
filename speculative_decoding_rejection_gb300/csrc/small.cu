// Fused verification of small batches: the whole linear verify in one
// kernel, one block per request, for calls whose rows are few and short
// (decode steps of a few requests over small vocabularies, where the
// multi-kernel schedule's launches and grid-wide passes cost more than the
// rows themselves). Each warp reduces whole rows, so all of a request's rows
// are read at once.
//
// Same rule and outputs as the multi-kernel path ("Acceptance Is Not
// Speed", §6; "RheoSampling 2026", §4; nalar.dev "Semantik penerimaan"):
// the block reduces each of its request's rows to (max, normaliser,
// argmax), decides the drafts in order with the same decision code
// (position_rejects_z), writes the accepted prefix, then draws the final
// token by inverse CDF in ascending id: from norm(max(0, p - q)) after a
// rejection (from p itself when that has no mass), from p_{K+1} after full
// acceptance, or the target's argmax for a greedy request.
#include "common.cuh"
#include "internal.h"
#include "linear.cuh"

namespace sv {

namespace {

constexpr int SMALL_THREADS = 512;
constexpr int SMALL_WARPS = SMALL_THREADS / 32;
constexpr int SMALL_TILE = SMALL_THREADS * SAMPLE_EPT;

struct SmallSmem {
  RowStat ts[SPEC_MAX_K + 1];   // target rows 1..K+1
  RowStat ds[SPEC_MAX_K];       // dense draft rows 1..K (sampling, draft logits)
  float zt[SPEC_MAX_K], zq[SPEC_MAX_K];   // z_t(d_i) and q(d_i) (or z_d(d_i)) per position
  int dtok[SPEC_MAX_K];
  float scratch[33];
  float red[SMALL_WARPS];
  int bad, n, xmin, xlast;
  float Z;
};

// Running (max, sum of 2^((z - m) c), lowest index of the max) of
// SAMPLE_EPT consecutive logits; c == 0 keeps the max and argmax only.
__device__ __forceinline__ void small_stat_update(const float *z, int x0, float c, float &m,
                                                  float &S, int &idx) {
  float vm = z[0];
  int j = 0;
#pragma unroll
  for (int k = 1; k < SAMPLE_EPT; ++k)
    if (z[k] > vm) { vm = z[k]; j = k; }
  if (vm > m) {
    if (c != 0.f) S *= ex2((m - vm) * c);
    m = vm;
    idx = x0 + j;
  }
  if (c != 0.f) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k) t += ex2((z[k] - m) * c);
    S += t;
  }
}

// The row's statistics over one warp (lanes merged by butterflies).
__device__ RowStat warp_row_stat_direct(const char *row, int dt, int V, float c, int lane) {
  const bool vec = ((uintptr_t)row & 15) == 0;
  float m = NO_MAX, S = 0.f;
  int idx = 0x7fffffff;
  float z[SAMPLE_EPT];
  for (int x0 = lane * SAMPLE_EPT; x0 < V; x0 += 32 * SAMPLE_EPT) {
    load_ept(row, dt, vec, x0, V, -INFINITY, z);
    small_stat_update(z, x0, c, m, S, idx);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float S2 = __shfl_xor_sync(0xffffffffu, S, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    merge_stat(m, S, idx, m2, S2, i2, c);
  }
  return RowStat{m, S, idx};
}

// Weights of SAMPLE_EPT elements from x0: the residual max(0, p - q) when
// `drow` is set, else p.
template <int DK>
__device__ __forceinline__ void small_weights(const LinearArgs &a, const char *trow, bool tvec,
                                              const char *drow, bool dvec, float c,
                                              const RowStat &t, const RowStat &d, int x0,
                                              float *w) {
  float z[SAMPLE_EPT];
  load_ept(trow, a.tdt, tvec, x0, a.V, -INFINITY, z);
  const float invSt = 1.f / t.S;
#pragma unroll
  for (int k = 0; k < SAMPLE_EPT; ++k) w[k] = ex2((z[k] - t.m) * c) * invSt;
  if (drow == nullptr) return;
  float y[SAMPLE_EPT];
  if (DK == SPEC_DRAFT_PROBS) {
    load_ept(drow, a.ddt, dvec, x0, a.V, 0.f, y);
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k) w[k] = fmaxf(0.f, w[k] - y[k]);
  } else {
    load_ept(drow, a.ddt, dvec, x0, a.V, -INFINITY, y);
    const float invSd = d.S > 0.f ? 1.f / d.S : 0.f;
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k) w[k] = fmaxf(0.f, w[k] - ex2((y[k] - d.m) * c) * invSd);
  }
}

// Inverse-CDF draw at u over the row's weights in ascending id: the smallest
// x with u * Z < C_x, else the last positive weight. Sets sh.Z; returns -1
// when the row has no mass.
template <int DK>
__device__ int small_draw(const LinearArgs &a, SmallSmem &sh, const char *trow, const char *drow,
                          float c, const RowStat &t, const RowStat &d, float u) {
  const bool tvec = ((uintptr_t)trow & 15) == 0, dvec = drow && ((uintptr_t)drow & 15) == 0;
  float w[SAMPLE_EPT];
  float s = 0.f;
  for (int x0 = (int)threadIdx.x * SAMPLE_EPT; x0 < a.V; x0 += SMALL_TILE) {
    small_weights<DK>(a, trow, tvec, drow, dvec, c, t, d, x0, w);
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k) s += w[k];
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) sh.red[warp] = s;
  if (threadIdx.x == 0) {
    sh.xmin = 0x7fffffff;
    sh.xlast = -1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float Z = 0.f;
    for (int k = 0; k < SMALL_WARPS; ++k) Z += sh.red[k];
    sh.Z = Z;
  }
  __syncthreads();
  const float Z = sh.Z;
  if (!(Z > 0.f)) return -1;
  const float target = u * Z;
  float carry = 0.f;
  for (int t0 = 0; t0 < a.V; t0 += SMALL_TILE) {
    const int x0 = t0 + (int)threadIdx.x * SAMPLE_EPT;
    small_weights<DK>(a, trow, tvec, drow, dvec, c, t, d, x0, w);
    float ts = 0.f;
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k) ts += w[k];
    float tot;
    const float excl = block_excl_scan(ts, sh.scratch, &tot);
    float pre = 0.f;
    int cand = 0x7fffffff, lastpos = -1;
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k) {
      pre += w[k];
      if (cand == 0x7fffffff && carry + (excl + pre) > target && x0 + k < a.V) cand = x0 + k;
      if (w[k] > 0.f && x0 + k < a.V) lastpos = x0 + k;
    }
    if (cand != 0x7fffffff) atomicMin(&sh.xmin, cand);
    if (lastpos >= 0) atomicMax(&sh.xlast, lastpos);
    __syncthreads();
    if (sh.xmin != 0x7fffffff) break;   // uniform: read after the barrier
    carry += tot;
  }
  const int x = sh.xmin != 0x7fffffff ? sh.xmin : sh.xlast;
  __syncthreads();
  return x;
}

template <int DK>
__global__ void __launch_bounds__(SMALL_THREADS) k_verify_small(const LinearArgs a) {
  __shared__ SmallSmem sh;
  const int b = blockIdx.x;
  const int W = a.max_k + 1;
  int32_t *out = a.out_tokens + (long long)b * W;
  // every block checks every request, so that an invalid input anywhere
  // leaves every request unverified, as the multi-kernel path does
  if (threadIdx.x == 0) sh.bad = 0;
  __syncthreads();
  for (int q = threadIdx.x; q < a.B; q += blockDim.x) {
    ReqInfo rq;
    if (!load_request(a, q, rq)) sh.bad = 1;
  }
  __syncthreads();
  ReqInfo r;
  load_request(a, b, r);
  if (sh.bad) {
    for (int j = threadIdx.x; j < W; j += blockDim.x) GST(out + j, -1);
    if (threadIdx.x == 0) GST(a.out_accepted + (b), -1);
    return;
  }
  const int K = r.K;
  const float c = r.c;
  const bool sample = r.mode == MODE_SAMPLE;
  const bool dense_draft = sample && DK == SPEC_DRAFT_LOGITS;
  {   // a warp per row, every row of the request at once
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R = K + 1 + (dense_draft ? K : 0);
    for (int q = warp; q < R; q += SMALL_WARPS) {
      const bool tr = q <= K;
      const RowStat s =
          tr ? warp_row_stat_direct(a.target + (long long)(r.t0 + q) * a.t_row_bytes, a.tdt,
                                    a.V, c, lane)
             : warp_row_stat_direct(a.draft + (long long)(r.d0 + q - K - 1) * a.d_row_bytes,
                                    a.ddt, a.V, c, lane);
      if (lane == 0) {
        if (tr) sh.ts[q] = s;
        else sh.ds[q - K - 1] = s;
      }
    }
  }
  __syncthreads();
  // each position's token and the two logits (or q(d)) its coin needs, all
  // loaded at once
  for (int i = threadIdx.x; i < K; i += blockDim.x) {
    const int d = GLD(a.tokens + (r.d0 + i));
    const bool dok = (unsigned)d < (unsigned)a.V;
    float zt = 0.f, zq = 0.f;
    if (sample && dok && !row_empty(sh.ts[i].m)) {
      zt = load_elem(a.target + (long long)(r.t0 + i) * a.t_row_bytes, a.tdt, d);
      zq = DK == SPEC_DRAFT_PROBS
               ? draft_prob_at(a, r.d0 + i, d, c, RowStat{NO_MAX, 0.f, 0x7fffffff})
               : load_elem(a.draft + (long long)(r.d0 + i) * a.d_row_bytes, a.ddt, d);
    }
    sh.dtok[i] = d;
    sh.zt[i] = zt;
    sh.zq[i] = zq;
  }
  __syncthreads();
  // the drafts in order (every position's p(d), q(d) is reported)
  if (threadIdx.x == 0) {
    int n = K;
    for (int i = 0; i < K; ++i) {
      const RowStat ds = dense_draft ? sh.ds[i] : RowStat{NO_MAX, 0.f, 0x7fffffff};
      const bool rej = position_rejects_z(a, b, r, i, sample, sh.ts[i], ds, 0, sh.dtok[i],
                                          sh.zt[i], sh.zq[i], DK == SPEC_DRAFT_PROBS);
      if (rej && n == K) n = i;
    }
    sh.n = n;
  }
  __syncthreads();
  const int n = sh.n;
  for (int j = threadIdx.x; j < W; j += blockDim.x) GST(out + j, j < n ? GLD(a.tokens + (r.d0 + j)) : -1);
  __syncthreads();
  int x;
  if (!sample) {
    x = sh.ts[n].idx;
  } else {
    const char *trow = a.target + (long long)(r.t0 + n) * a.t_row_bytes;
    const float u = uniform24(seed_of(a), (uint32_t)b, (uint32_t)(n + 1), n < K ? 1u : 2u);
    x = -1;
    if (n < K) {   // residual of the rejected position
      const RowStat dn = dense_draft ? sh.ds[n] : RowStat{NO_MAX, 0.f, 0x7fffffff};
      x = small_draw<DK>(a, sh, trow, a.draft + (long long)(r.d0 + n) * a.d_row_bytes, c,
                         sh.ts[n], dn, u);
    }
    if (x < 0)   // bonus draw, or a residual without mass: p with the same u
      x = small_draw<DK>(a, sh, trow, nullptr, c, sh.ts[n], RowStat{}, u);
  }
  if (threadIdx.x == 0) {
    if (x < 0 || x == 0x7fffffff) {
      set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);   // a row without mass
      x = -1;
    }
    GST(out + n, x);
    GST(a.out_accepted + (b), n);
  }
}

}  // namespace

int launch_verify_small(const LinearArgs &a, cudaStream_t stream) {
  if (check_upload(stream) != SPEC_OK) return SPEC_ERR_CUDA;
  cudaEvent_t before, after;
  take_row_pass_events(&before, &after);
  if (before && cudaEventRecord(before, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  if (a.dk == SPEC_DRAFT_PROBS)
    k_verify_small<SPEC_DRAFT_PROBS><<<a.B, SMALL_THREADS, 0, stream>>>(a);
  else
    k_verify_small<SPEC_DRAFT_LOGITS><<<a.B, SMALL_THREADS, 0, stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (after && cudaEventRecord(after, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

}  // namespace sv
