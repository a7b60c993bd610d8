// Arguments of a linear verification call and the per-request decision
// logic shared by the accept scan, the position-lazy rounds and the
// streaming verifier.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace sv {

constexpr int ACCEPT_WARPS = 8;

struct StreamEntry;

struct LinearArgs {
  const char *target;
  const char *draft;
  int tdt, ddt, dk, rule;
  const int32_t *draft_idx;   // sparse ids (caller's, or the top-128 scratch)
  const float *sparse_prob;   // sparse probabilities (caller's or scratch)
  const int32_t *tokens;
  const int32_t *cu;
  const float *temp;
  int B, V, max_k;
  uint64_t seed;
  const uint64_t *seed_dev;   // optional: the seed read on the device at run time
  int32_t *out_tokens;
  int32_t *out_accepted;
  float *out_pq;
  WsHeader *hdr;
  WsHeader *err;              // where the decision code reports invalid inputs
  ReqInfo *req;
  Job *jobs_a;                // residual draws over dense draft rows
  Job *jobs_b;                // bonus draws and sparse residual draws
  float *tsum;                // [B][ntiles][RS_CONS_WARPS] residual tile sums of jobs_a
  int ntiles;
  long long rows_max;
  RowTask *list;
  Part *part;
  long long t_row_bytes, d_row_bytes;
  int nch_t, nch_d, nch_max;   // chunks of the mode's chunk size
  int chunk_bytes;
  int rt_max;                 // slot offset of draft rows
  int sparse;                 // the draft law is sparse (given or top-128)
  int stream_draft;           // the row pass reads dense draft logits
  // relaxed rule and target ranks
  float alpha, min_prob;
  int max_rank;
  int want_rank;              // the row pass counts ranks
  float *rank_thr;            // [rt_max] draft token's target logit per slot
  int32_t *out_rank;
  // position-lazy schedule: one row pass + decide per position (round)
  int lazy, round;
  // per-position KL(p || q): target and draft rows streamed as pairs
  int want_kl;
  float *kl_part;             // A partials of the pair rows' target slots
  float *out_kl;
  // streaming verifier: per-position progress and residual entries
  StreamEntry *ent_d;         // [cap_d] residual entries allocated while the kernel runs
  int *ready_d;               // [2 cap_d] 1 once ent_d[e] is written; then, per
                              // request, the completed items of its residual entry
  int *pos_done;              // [B * (max_k + 1)] completed work items of a position's rows
  int *pos_join;              // [B * (max_k + 1)] events of a position: its rows are
                              // complete, the previous position was accepted
  int *rej_at;                // [B] position of the first rejection (INT_MAX: none yet)
  float *zd_at;               // [R_d] z_d(d_i), gathered by the setup
  int cap_d;                  // B
  int stride;                 // tickets per position of a request
  int n_res_items;            // residual work items per final draw
};

// Validates request b and fills its record (first rows, drafts, mode and
// c = log2(e)/T). Returns false, with the status word set, on an invalid
// request: a bad offset, a draft count outside [0, max_k], a negative or
// non-finite temperature, or a sampling request without a draft tensor.
// The call's seed: from device memory when the caller gave a pointer (so a
// captured CUDA graph draws new uniforms after the caller writes a new seed).
__device__ __forceinline__ uint64_t seed_of(const LinearArgs &a) {
  return a.seed_dev != nullptr ? GLDG(a.seed_dev) : a.seed;
}

__device__ __forceinline__ bool load_request(const LinearArgs &a, int b, ReqInfo &r) {
  const int cb = GLD(a.cu + b), cb1 = GLD(a.cu + b + 1);
  const int K = cb1 - cb;
  const float T = GLD(a.temp + b);
  const long long dmax = a.rows_max - a.rt_max;
  r.t0 = cb + b;
  r.d0 = cb;
  r.K = K;
  r.n = 0;
  r.pad[0] = r.pad[1] = 0;
  const bool greedy = a.rule == SPEC_RULE_GREEDY || T < SPEC_GREEDY_T;
  bool ok = (b > 0 || cb == 0) && K >= 0 && K <= a.max_k && cb >= 0 &&
            (long long)cb1 <= dmax && T >= 0.f && isfinite(T);
  if (ok && !greedy && a.draft == nullptr) ok = false;
  if (!ok) {
    set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);
    r.mode = MODE_SKIP;
    r.c = 0.f;
    return false;
  }
  r.mode = greedy ? MODE_GREEDY : MODE_SAMPLE;
  r.c = greedy ? 0.f : (float)(1.4426950408889634 / (double)T);
  return true;
}

// ------------------------------------------------------------ accept scan
// Part slots of position i's rows of request b: eager, one per listed row;
// lazy, entries b and B + b of the current round.
__device__ __forceinline__ int tslot(const LinearArgs &a, const ReqInfo &r, int b, int i) {
  return a.lazy ? b : r.t0 + i;
}
__device__ __forceinline__ int dslot(const LinearArgs &a, const ReqInfo &r, int b, int i) {
  return a.lazy ? a.B + b : a.rt_max + r.d0 + i;
}

// Rank count of a target row: the sum of the chunk partials' counts.
__device__ __forceinline__ int warp_row_count(const LinearArgs &a, int slot, int lane) {
  const Part *p = a.part + (long long)slot * a.nch_max * RS_CONS_WARPS;
  const int n = a.nch_t * RS_CONS_WARPS;
  int c = 0;
  for (int i = lane; i < n; i += 32) c += ldcg_part(p + i).cnt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  return c;
}
__device__ __forceinline__ RowStat target_stat(const LinearArgs &a, int slot, float c, int lane) {
  return warp_row_stat(a.part + (long long)slot * a.nch_max * RS_CONS_WARPS,
                       a.nch_t * RS_CONS_WARPS, c, lane);
}
__device__ __forceinline__ RowStat draft_stat(const LinearArgs &a, int slot, float c, int lane) {
  return warp_row_stat(a.part + (long long)slot * a.nch_max * RS_CONS_WARPS,
                       a.nch_d * RS_CONS_WARPS, c, lane);
}

// KL(p || q) of a pair row: the target partials merged with their A sums
// (warp-wide, fixed order), then KL = (A/S - (m_t - m_d))/T - ln S + ln S_d.
__device__ __forceinline__ float warp_pair_kl(const LinearArgs &a, int tslot_, const RowStat &ds,
                                              float c, int lane) {
  const long long base = (long long)tslot_ * a.nch_max * RS_CONS_WARPS;
  const int n = a.nch_t * RS_CONS_WARPS;
  float m = NO_MAX, S = 0.f, A = 0.f;
  int idx = 0x7fffffff;
  for (int i = lane; i < n; i += 32) {
    const Part q = ldcg_part(a.part + base + i);
    merge_stat_a(m, S, idx, A, q.m, q.S, q.idx, GLDCG(a.kl_part + base + i), c);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float S2 = __shfl_xor_sync(0xffffffffu, S, o);
    const float A2 = __shfl_xor_sync(0xffffffffu, A, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    merge_stat_a(m, S, idx, A, m2, S2, i2, A2, c);
  }
  const float inv_t = c * 0.6931471805599453f;   // 1/T = ln 2 * log2(e)/T
  return inv_t * (A / S - (m - ds.m)) + logf(ds.S / S);
}

// q(d) for draft row `row` given its statistics ds (dense logits), the
// probability itself, or a search of the sparse ids (any order).
static __device__ float draft_prob_at(const LinearArgs &a, int row, int d, float c, RowStat ds) {
  if (a.sparse) {
    const int32_t *ids = a.draft_idx + (long long)row * SPEC_TOPK;
    const float *pr = a.sparse_prob + (long long)row * SPEC_TOPK;
    for (int k = 0; k < SPEC_TOPK; ++k)
      if (GLD(ids + k) == d) return GLD(pr + k);
    return 0.f;
  }
  const char *drow = a.draft + (long long)row * a.d_row_bytes;
  if (a.dk == SPEC_DRAFT_PROBS) return load_elem(drow, a.ddt, d);
  if (row_empty(ds.m)) return 0.f;
  return ex2((load_elem(drow, a.ddt, d) - ds.m) * c) / ds.S;
}

// q(d) of sparse draft row `row` (up to SPEC_TOPK (id, prob) pairs, any
// order, -1 for an empty slot): the warp searches the ids together; 0 when d
// is not listed. Every lane returns the value.
__device__ __forceinline__ float warp_sparse_q(const LinearArgs &a, int row, int d, int lane) {
  const long long base = (long long)row * SPEC_TOPK;
  for (int k0 = 0; k0 < SPEC_TOPK; k0 += 32) {
    const unsigned m = __ballot_sync(0xffffffffu, GLD(a.draft_idx + base + k0 + lane) == d);
    if (m) return GLD(a.sparse_prob + base + k0 + __ffs(m) - 1);
  }
  return 0.f;
}

// Decision on draft position i (0-based) of request b from the statistics of
// its target row (ts) and dense draft row (ds), its target rank, its token d
// and, for a valid d, the target logit zt = z_t(d) and either the draft
// logit (q_is_prob false: q(d) = softmax of the dense draft row at d) or
// q(d) itself: greedy prefix match, the lossless coin, or the CACTUS guard
// and coin. Writes p(d), q(d) and the rank. Returns true when the draft is
// rejected.
static __device__ bool position_rejects_z(const LinearArgs &a, int b, const ReqInfo &r, int i,
                                          bool sample, const RowStat &ts, const RowStat &ds,
                                          int rank, int d, float zt, float zq, bool q_is_prob) {
  const float c = r.c;
  const bool dok = (unsigned)d < (unsigned)a.V;
  if (!dok) set_status(a.err, SPEC_ERR_INVALID_ARG, b);
  if (row_empty(ts.m)) set_status(a.err, SPEC_ERR_INVALID_ARG, b);
  float pd, qd;
  bool rej;
  if (!sample) {
    rej = !(dok && d == ts.idx);
    pd = rej ? 0.f : 1.f;
    qd = -1.f;
  } else if (dok && !row_empty(ts.m)) {
    pd = ex2((zt - ts.m) * c) / ts.S;
    qd = q_is_prob ? zq : row_empty(ds.m) ? 0.f : ex2((zq - ds.m) * c) / ds.S;
    if (a.rule == SPEC_RULE_CACTUS) {
      const float g = fminf(pd + sqrtf(2.f * a.alpha * pd * (1.f - pd)), 1.f);
      const float acc = qd <= g ? 1.f : g / qd;
      const bool guard = (a.max_rank > 0 && rank > a.max_rank) || pd < a.min_prob;
      rej = guard || !(uniform24(seed_of(a), (uint32_t)b, (uint32_t)(i + 1), 0) < acc);
    } else {
      const float acc = qd <= pd ? 1.f : pd / qd;
      rej = !(uniform24(seed_of(a), (uint32_t)b, (uint32_t)(i + 1), 0) < acc);
    }
  } else {
    pd = 0.f;
    qd = 0.f;
    rej = true;
  }
  if (a.out_pq) {
    GST(a.out_pq + 2LL * (r.d0 + i), pd);
    GST(a.out_pq + 2LL * (r.d0 + i) + 1, qd);
  }
  if (a.out_rank) GST(a.out_rank + r.d0 + i, rank);
  return rej;
}

// position_rejects_z with its inputs loaded here: the token, z_t(d), and q(d)
// (given by the caller for sparse laws, else from the draft row).
static __device__ bool position_rejects(const LinearArgs &a, int b, const ReqInfo &r, int i,
                                        bool sample, const RowStat &ts, const RowStat &ds,
                                        int rank, float q_given = -1.f) {
  const int d = GLD(a.tokens + r.d0 + i);
  const bool dok = (unsigned)d < (unsigned)a.V;
  float zt = 0.f, zq = 0.f;
  bool q_is_prob = true;
  if (sample && dok && !row_empty(ts.m)) {
    zt = load_elem(a.target + (long long)(r.t0 + i) * a.t_row_bytes, a.tdt, d);
    if (q_given >= 0.f) {
      zq = q_given;
    } else if (a.sparse || a.dk == SPEC_DRAFT_PROBS) {
      zq = draft_prob_at(a, r.d0 + i, d, r.c, ds);
    } else {
      zq = load_elem(a.draft + (long long)(r.d0 + i) * a.d_row_bytes, a.ddt, d);
      q_is_prob = false;
    }
  }
  return position_rejects_z(a, b, r, i, sample, ts, ds, rank, d, zt, zq, q_is_prob);
}

// n drafts accepted: write them and queue the final token (greedy: the
// argmax of p_{n+1}; sampling: a residual job when n < K, else a bonus job).
// tf / df are the statistics of target row n+1 and dense draft row n+1.
static __device__ void finish_request(const LinearArgs &a, int b, const ReqInfo &r, int n, bool sample,
                               const RowStat &tf, const RowStat &df, int lane) {
  const int W = a.max_k + 1;
  int32_t *out = a.out_tokens + (long long)b * W;
  for (int j = lane; j < W; j += 32) GST(out + j, j < n ? GLD(a.tokens + r.d0 + j) : -1);
  __syncwarp();
  if (lane == 0) {
    GST(a.out_accepted + b, n);
    if (!sample) {
      GST(out + n, tf.idx);
    } else {
      const Job j{b, n, n < r.K ? 1 : 2, 0, tf.m, tf.S, df.m, df.S};
      if (j.kind == 1 && !a.sparse) GST(a.jobs_a + atomicAdd(&a.hdr->n_jobs_a, 1), j);
      else GST(a.jobs_b + atomicAdd(&a.hdr->n_jobs_b, 1), j);
    }
  }
}

// The streaming verifier (one persistent kernel for the position-lazy
// schedule) and the inputs it covers.
bool stream_supported(const LinearArgs &a);
int launch_verify_stream(const LinearArgs &a, cudaStream_t stream);

// The cluster-resident verifier (the position-lazy schedule with each
// position's rows held in the shared memory of a CTA cluster, so every row
// is read from HBM once) and the inputs it covers: the strict rule on dense
// bf16 logits, V % 8 == 0, V in [16384, 204800], no rank or KL outputs.
bool resident_supported(const LinearArgs &a);
int launch_verify_resident(const LinearArgs &a, cudaStream_t stream);

// Small calls whose rows are too long for the fused kernel (at most 128
// requests, dense bf16 logits, V % 8 == 0, at most 8 drafts, a request's
// 2K+1 row slices within 100 KB per CTA; off when `limit_bytes`, the fused
// limit, is 0): one launch, one cluster per request, the rows through a few
// shared-memory buffers per CTA, two exchanges per request.
bool cluster_small_supported(const LinearArgs &a, const spec_linear_ext *ext,
                             size_t limit_bytes);
int launch_verify_cluster_small(const LinearArgs &a, cudaStream_t stream);

// The fused small-batch verifier (one kernel, one block per request) and the
// calls it takes.
bool small_supported(const LinearArgs &a, const spec_linear_ext *ext);
int launch_verify_small(const LinearArgs &a, cudaStream_t stream);

// Rows and laws of a final draw.
struct JobRows {
  const char *trow, *drow;
  bool tvec, dvec;
  float c, mt, invSt, md, invSd;
};

__device__ __forceinline__ JobRows job_rows(const LinearArgs &a, const Job &j) {
  const ReqInfo r = GLD(a.req + j.b);
  JobRows q;
  q.trow = a.target + (long long)(r.t0 + j.n) * a.t_row_bytes;
  q.tvec = ((uintptr_t)q.trow & 15) == 0;
  q.drow = nullptr;
  q.dvec = false;
  if (j.kind == 1 && !a.sparse) {
    q.drow = a.draft + (long long)(r.d0 + j.n) * a.d_row_bytes;
    q.dvec = ((uintptr_t)q.drow & 15) == 0;
  }
  q.c = r.c;
  q.mt = j.mt;
  q.invSt = 1.f / j.St;
  q.md = j.md;
  q.invSd = j.Sd > 0.f ? 1.f / j.Sd : 0.f;
  return q;
}

}  // namespace sv
