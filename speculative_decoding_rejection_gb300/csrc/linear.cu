// Linear verification: setup, row pass, accept scan, final-token sampler.
//
// Per request b with drafts d_1..d_K:
//   accept scan   a_i = 1 if q_i(d_i) <= p_i(d_i) else p_i(d_i)/q_i(d_i);
//                 accept iff u(seed, b, i, 0) < a_i; stop at the first
//                 rejection ("Acceptance Is Not Speed", §6; "RheoSampling
//                 2026", §4 step 1; nalar.dev "Penolakan memendekkan
//                 pekerjaan speculative": drafts after it are discarded).
//                 Greedy: accept while d_i == argmax p_i (nalar.dev
//                 "Semantik penerimaan").
//   final token   n < K: draw from max(0, p_{n+1} - q_{n+1}) / Z at
//                 u(seed, b, n+1, 1) ("RheoSampling 2026", §4 step 3; p
//                 itself when Z == 0); n == K: bonus draw from p_{K+1} at
//                 u(seed, b, K+1, 2); greedy: argmax p_{n+1}.
//                 Draw = smallest x (ascending id) with u*Z < C_x.
//   CACTUS rule   a_i = min(1, gamma/q_i(d_i)) with gamma = min(p + sqrt(2
//                 alpha p (1 - p)), 1), p = p_i(d_i), after the low-support
//                 guard (reject outright when rank(d_i) > max_rank or
//                 p < min_prob) ("Acceptance Is Not Speed", §6 rules 1-3 and
//                 §7 item 3); the rank is counted by the row pass. The
//                 replacement after a rejection is the lossless residual
//                 draw (the page's residual for the rule is lost).
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "linear.cuh"

namespace sv {

struct LinearLayout {
  size_t hdr, err, req, jobs_a, jobs_b, tsum, list, part, kl_part, tk_idx, tk_prob, tk_list;
  size_t rank_thr;
  size_t ent_d, ready_d, pos_done, pos_join, rej_at, zd_at, total;
  int nch_max, nch_max_lazy, nch_max_stream;
  long long rows_max;
};

static LinearLayout linear_layout(int B, int max_k, int V, int rule) {
  LinearLayout L;
  L.nch_max = nchunks(V, SPEC_F32, CHUNK_BYTES);
  L.nch_max_lazy = nchunks(V, SPEC_F32, LAZY_CHUNK_BYTES);
  L.rows_max = (long long)B * (2LL * max_k + 1);
  size_t o = 0;
  L.hdr = o;  o += align256(sizeof(WsHeader));
  L.err = o;  o += align256(sizeof(WsHeader));   // errors found by the streaming verifier
  L.req = o;  o += align256(sizeof(ReqInfo) * (size_t)B);
  L.jobs_a = o; o += align256(sizeof(Job) * (size_t)B);
  L.jobs_b = o; o += align256(sizeof(Job) * (size_t)B);
  L.tsum = o;
  o += align256(sizeof(float) * (size_t)B * ((V + SAMPLE_TILE - 1) / SAMPLE_TILE) * RS_CONS_WARPS);
  L.list = o; o += align256(sizeof(RowTask) * (size_t)std::max(L.rows_max, 2LL * B));
  // eager: one slot per listed row; lazy: two per request (its rows of the
  // current round), in finer chunks
  L.nch_max_stream = nchunks(V, SPEC_BF16, STREAM_CHUNK_BYTES);   // bf16 rows only
  L.part = o;
  o += align256(sizeof(Part) * RS_CONS_WARPS *
                std::max({(size_t)L.rows_max * L.nch_max, (size_t)2 * B * L.nch_max_lazy,
                          (size_t)L.rows_max * L.nch_max_stream}));
  const size_t tk = rule == SPEC_RULE_STRICT_TOP128 ? (size_t)B * max_k * SPEC_TOPK : 0;
  L.kl_part = o;
  o += align256(sizeof(float) * RS_CONS_WARPS *
                std::max((size_t)B * (max_k + 1) * L.nch_max, (size_t)B * L.nch_max_lazy));
  L.tk_idx = o;  o += align256(sizeof(int32_t) * tk);
  L.tk_prob = o; o += align256(sizeof(float) * tk);
  L.tk_list = o;   // the top-128 select's candidate lists
  o += rule == SPEC_RULE_STRICT_TOP128 ? topk_list_bytes((long long)B * max_k) : 0;
  L.rank_thr = o; o += align256(sizeof(float) * (size_t)B * (max_k + 1));
  // streaming verifier: residual entries (32 B) and their ready flags,
  // per-position counters, first rejections
  const size_t npos = (size_t)B * (max_k + 1);
  L.ent_d = o; o += align256(32 * (size_t)B);
  L.ready_d = o; o += align256(sizeof(int) * 2 * (size_t)B);   // flags, then counts
  L.pos_done = o; o += align256(sizeof(int) * npos);
  L.pos_join = o; o += align256(sizeof(int) * npos);
  L.rej_at = o; o += align256(sizeof(int) * (size_t)B);
  L.zd_at = o; o += align256(sizeof(float) * (size_t)B * max_k);
  L.total = o;
  return L;
}

// ------------------------------------------------------------------ setup
// One thread per request. The row list is indexed by slot (target row r at
// position r, draft row r at position rt_max + r), so every thread writes its
// own entries without a scan; positions no request owns are marked unused.
// The header was cleared before the launch; an invalid request sets the
// status word, which makes every later kernel of the call skip its work.
// Position-lazy: the list holds, per request b, entry b (target row) and
// entry B + b (draft row) of the first position only.
__global__ void __launch_bounds__(64) k_setup_linear(const LinearArgs a) {
  const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
  const int gsize = gridDim.x * blockDim.x;
  if (gtid == 0) a.hdr->n_list = a.lazy ? 2 * a.B : (int)a.rows_max;
  const long long dmax = a.rows_max - a.rt_max;
  if (!a.lazy) {
    const long long Rd = a.B > 0 ? min(max((long long)GLD(a.cu + (a.B)), 0LL), dmax) : 0;
    const long long Rt = min(Rd + a.B, (long long)a.rt_max);
    for (long long p = Rt + gtid; p < a.rt_max; p += gsize) GST(&a.list[p].slot, -1);
    for (long long p = a.rt_max + Rd + gtid; p < a.rows_max; p += gsize) GST(&a.list[p].slot, -1);
  }
  const int b = gtid;
  if (b >= a.B) return;
  if (a.lazy) {   // idle until the request validates
    GST(&a.list[b].slot, -1);
    GST(&a.list[a.B + b].slot, -1);
  }
  ReqInfo r;
  if (!load_request(a, b, r)) {
    GST(a.req + (b), r);
    return;
  }
  const int K = r.K;
  GST(a.req + (b), r);
  const bool drafts = r.mode == MODE_SAMPLE && a.stream_draft;
  // with KL, a draft row travels with its target row as one pair entry
  const bool pairs = drafts && a.want_kl;
  if (a.lazy) {
    if (pairs && K > 0) {
      GST(a.list + (b), RowTask{b, r.t0, ROW_PAIR, r.c, a.B + b, r.d0});
      GST(&a.list[a.B + b].slot, -1);
    } else {
      GST(a.list + (b), RowTask{b, r.t0, 0, r.c});
      GST(a.list + (a.B + b), RowTask{drafts && K > 0 ? a.B + b : -1, r.d0, 1, r.c});
    }
  } else {
    for (int i = 0; i <= K; ++i)
      GST(a.list + (r.t0 + i), pairs && i < K
                             ? RowTask{r.t0 + i, r.t0 + i, ROW_PAIR, r.c, a.rt_max + r.d0 + i, r.d0 + i}
                             : RowTask{r.t0 + i, r.t0 + i, 0, r.c});
    for (int i = 0; i < K; ++i)
      GST(a.list + (a.rt_max + r.d0 + i), RowTask{drafts && !pairs ? a.rt_max + r.d0 + i : -1, r.d0 + i, 1, r.c});
  }
  if (a.want_rank) {   // threshold of the rank count: the draft token's target logit
    for (int i = 0; i < K; ++i) {
      const int d = GLD(a.tokens + (r.d0 + i));
      GST(a.rank_thr + (r.t0 + i), (unsigned)d < (unsigned)a.V
              ? load_elem(a.target + (long long)(r.t0 + i) * a.t_row_bytes, a.tdt, d)
              : INFINITY);   // reported by the accept scan
    }
    GST(a.rank_thr + (r.t0 + K), INFINITY);
  }
}

// warp_row_stat of up to ACC_ROWS rows at once. Each row keeps that
// function's merge order exactly (lane l merges partials l, l+32, ..., then
// the butterfly), so the statistics are bit for bit the same; only the rows'
// partial loads are issued together, and the warp waits one memory latency
// per group of rows instead of one per row. With `cnt`, the first rows'
// rank counts (the sum of their partials' counts) come from the same loads.
constexpr int ACC_G = 4;               // positions per group
constexpr int ACC_ROWS = 2 * ACC_G;    // their target rows, then their draft rows
__device__ __forceinline__ void warp_row_stats_group(const Part *const (&rows)[ACC_ROWS],
                                                     const int (&nparts)[ACC_ROWS], float c,
                                                     int lane, RowStat (&out)[ACC_ROWS],
                                                     int (&cnt)[ACC_G]) {
  float m[ACC_ROWS], S[ACC_ROWS];
  int idx[ACC_ROWS];
  int nmax = 0;
#pragma unroll
  for (int k = 0; k < ACC_ROWS; ++k) {
    m[k] = NO_MAX;
    S[k] = 0.f;
    idx[k] = 0x7fffffff;
    nmax = max(nmax, nparts[k]);
  }
#pragma unroll
  for (int k = 0; k < ACC_G; ++k) cnt[k] = 0;
  for (int i = lane; i < nmax; i += 32) {
    Part q[ACC_ROWS];
#pragma unroll
    for (int k = 0; k < ACC_ROWS; ++k)
      if (i < nparts[k]) q[k] = ldcg_part(rows[k] + i);
#pragma unroll
    for (int k = 0; k < ACC_ROWS; ++k)
      if (i < nparts[k]) {
        merge_stat(m[k], S[k], idx[k], q[k].m, q[k].S, q[k].idx, c);
        if (k < ACC_G) cnt[k] += q[k].cnt;
      }
  }
#pragma unroll
  for (int k = 0; k < ACC_ROWS; ++k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m[k], o);
      const float S2 = __shfl_xor_sync(0xffffffffu, S[k], o);
      const int i2 = __shfl_xor_sync(0xffffffffu, idx[k], o);
      merge_stat(m[k], S[k], idx[k], m2, S2, i2, c);
    }
    out[k] = RowStat{m[k], S[k], idx[k]};
  }
#pragma unroll
  for (int k = 0; k < ACC_G; ++k)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt[k] += __shfl_xor_sync(0xffffffffu, cnt[k], o);
}

__device__ __forceinline__ RowStat shfl_stat(const RowStat &s, int src) {
  return RowStat{__shfl_sync(0xffffffffu, s.m, src), __shfl_sync(0xffffffffu, s.S, src),
                 __shfl_sync(0xffffffffu, s.idx, src)};
}

// q(d) of sparse draft row `row` for one lane: the probability listed with
// id d, 0 when d is not listed. 16-byte loads, eight in flight, no early
// exit, where the ids are 16-byte aligned (the top-128 scratch); a caller's
// ids need only 4-byte alignment and are read one by one.
__device__ __forceinline__ float lane_sparse_q(const LinearArgs &a, int row, int d) {
  const int32_t *ids = a.draft_idx + (long long)row * SPEC_TOPK;
  int hit = -1;
  if (((uintptr_t)ids & 15) == 0) {
    const int4 *ids4 = reinterpret_cast<const int4 *>(ids);
#pragma unroll 8
    for (int k = 0; k < SPEC_TOPK / 4; ++k) {
      const int4 v = GLD(ids4 + k);
      if (hit < 0)
        hit = v.x == d ? 4 * k : v.y == d ? 4 * k + 1 : v.z == d ? 4 * k + 2
            : v.w == d ? 4 * k + 3 : -1;
    }
  } else {
    for (int k = 0; k < SPEC_TOPK && hit < 0; ++k)
      if (GLD(ids + k) == d) hit = k;
  }
  return hit >= 0 ? GLD(a.sparse_prob + ((long long)row * SPEC_TOPK + hit)) : 0.f;
}

__global__ void __launch_bounds__(ACCEPT_WARPS * 32) k_accept(const LinearArgs a) {
  const int b = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= a.B) return;
  const int W = a.max_k + 1;
  int32_t *out = a.out_tokens + (long long)b * W;
  // inputs rejected by the setup (or an expired wait): no request is verified
  if (*(volatile int *)&a.hdr->status != SPEC_OK) {
    for (int j = lane; j < W; j += 32) GST(out + j, -1);
    if (lane == 0) GST(a.out_accepted + (b), -1);
    return;
  }
  const ReqInfo r = GLD(a.req + (b));
  const int K = r.K;
  const float c = r.c;
  const bool sample = r.mode == MODE_SAMPLE;
  const bool dense = sample && a.stream_draft;   // dense draft logits, reduced by the row pass
  const long long rstride = (long long)a.nch_max * RS_CONS_WARPS;
  int n = K;
  // lane 0's statistics of target row n+1 and draft row n+1 (the final
  // draw's law), taken when the first rejection is found
  RowStat tf{NO_MAX, 0.f, 0x7fffffff}, df{NO_MAX, 0.f, 0x7fffffff};
  for (int base = 0; base < K; base += 32) {
    const int cnt = min(32, K - base);
    // lane i decides position base + i; its token and, for dense drafts, the
    // two logits at it are loaded first so their latency overlaps the
    // statistics below
    const int i = base + lane;
    int d = -1;
    float zt = 0.f, zq = 0.f;
    if (lane < cnt) {
      d = GLD(a.tokens + (r.d0 + i));
      if (dense && (unsigned)d < (unsigned)a.V) {
        zt = load_elem(a.target + (long long)(r.t0 + i) * a.t_row_bytes, a.tdt, d);
        zq = load_elem(a.draft + (long long)(r.d0 + i) * a.d_row_bytes, a.ddt, d);
      }
    }
    // statistics of this block of positions: lane i keeps position base + i
    // as reduced on lane i (its decision) and as reduced on lane 0 (the
    // final draw's law, as the job records it)
    RowStat ts{NO_MAX, 0.f, 0x7fffffff}, ds{NO_MAX, 0.f, 0x7fffffff};
    RowStat ts0 = ts, ds0 = ds;
    int rank = 0;
    float kl = __int_as_float(0x7fc00000);   // NaN: greedy requests
    for (int g0 = 0; g0 < cnt; g0 += ACC_G) {
      const Part *rows[ACC_ROWS];
      int np[ACC_ROWS];
#pragma unroll
      for (int k = 0; k < ACC_G; ++k) {
        const bool on = g0 + k < cnt;
        rows[k] = a.part + (long long)tslot(a, r, b, base + g0 + k) * rstride;
        np[k] = on ? a.nch_t * RS_CONS_WARPS : 0;
        rows[ACC_G + k] = a.part + (long long)dslot(a, r, b, base + g0 + k) * rstride;
        np[ACC_G + k] = on && dense ? a.nch_d * RS_CONS_WARPS : 0;
      }
      RowStat st[ACC_ROWS];
      int rc[ACC_G];
      warp_row_stats_group(rows, np, c, lane, st, rc);
#pragma unroll
      for (int k = 0; k < ACC_G; ++k) {
        if (g0 + k >= cnt) break;
        const RowStat t0 = shfl_stat(st[k], 0), d0 = shfl_stat(st[ACC_G + k], 0);
        if (lane == g0 + k) {
          ts = st[k];
          ds = st[ACC_G + k];
          ts0 = t0;
          ds0 = d0;
          rank = a.want_rank ? 1 + rc[k] : 0;
        }
        if (dense && a.want_kl) {
          const float kk = warp_pair_kl(a, tslot(a, r, b, base + g0 + k), st[ACC_G + k], c, lane);
          if (lane == g0 + k) kl = kk;
        }
      }
    }
    if (a.out_kl && lane < cnt) GST(a.out_kl + (r.d0 + base + lane), kl);
    // (a sparse law's q(d) is searched by each lane for its own position: the
    // positions' searches run side by side)
    const bool rej =
        lane < cnt && (dense ? position_rejects_z(a, b, r, i, sample, ts, ds, rank, d, zt, zq,
                                                  false)
                             : position_rejects(a, b, r, i, sample, ts, ds, rank,
                                                a.sparse && sample && (unsigned)d < (unsigned)a.V
                                                    ? lane_sparse_q(a, r.d0 + i, d)
                                                    : -1.f));
    const unsigned bal = __ballot_sync(0xffffffffu, rej);
    if (n == K && bal) {
      n = base + __ffs(bal) - 1;
      tf = shfl_stat(ts0, n - base);
      df = shfl_stat(ds0, n - base);
    }
  }
  if (n == K) tf = target_stat(a, tslot(a, r, b, n), c, lane);
  finish_request(a, b, r, n, sample, tf, df, lane);
}

// ------------------------------------------------ position-lazy rounds
// Round `a.round` = j: the row pass has just streamed, for every request
// still active, target row p_{j+1} and (sampling, dense draft) draft row
// q_{j+1}. One warp per request decides draft j+1 (or, at j == K, takes the
// bonus row), then either lists the next position's rows or finishes the
// request. The row list is indexed by request: entry b the target row,
// entry B + b the draft row, slot -1 when idle. Rows after the first
// rejection are never streamed (nalar.dev, "Penolakan memendekkan pekerjaan
// speculative").
__global__ void __launch_bounds__(ACCEPT_WARPS * 32) k_lazy_decide(const LinearArgs a) {
  const int b = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0) a.hdr->work = 0;   // the next round's counter
  if (b >= a.B) return;
  const int W = a.max_k + 1;
  int32_t *out = a.out_tokens + (long long)b * W;
  if (*(volatile int *)&a.hdr->status != SPEC_OK) {
    for (int j = lane; j < W; j += 32) GST(out + j, -1);
    if (lane == 0) {
      GST(a.out_accepted + (b), -1);
      GST(&a.list[b].slot, -1);
      GST(&a.list[a.B + b].slot, -1);
    }
    return;
  }
  if (GLD(&a.list[b].slot) < 0) return;   // finished in an earlier round
  const ReqInfo r = GLD(a.req + (b));
  const int K = r.K, j = a.round;
  const float c = r.c;
  const bool sample = r.mode == MODE_SAMPLE;
  const RowStat ts = target_stat(a, tslot(a, r, b, j), c, lane);
  RowStat ds{NO_MAX, 0.f, 0x7fffffff};
  int n = K;
  if (j < K) {
    const int rank = a.want_rank ? 1 + warp_row_count(a, tslot(a, r, b, j), lane) : 0;
    if (sample && a.stream_draft) ds = draft_stat(a, dslot(a, r, b, j), c, lane);
    if (a.out_kl) {
      const float kl = sample && a.stream_draft ? warp_pair_kl(a, tslot(a, r, b, j), ds, c, lane)
                                                : __int_as_float(0x7fc00000);
      if (lane == 0) GST(a.out_kl + (r.d0 + j), kl);
    }
    // a sparse draft's q(d): the warp searches the row's 128 ids together
    const float qs = sample && a.sparse ? warp_sparse_q(a, r.d0 + j, GLD(a.tokens + (r.d0 + j)), lane)
                                        : -1.f;
    const bool rej = __shfl_sync(
        0xffffffffu, lane == 0 && position_rejects(a, b, r, j, sample, ts, ds, rank, qs), 0);
    if (!rej) {   // accepted: list the next position's rows
      if (lane == 0) {
        const bool drow = sample && a.stream_draft && j + 1 < K;
        if (drow && a.want_kl) {
          GST(a.list + (b), RowTask{b, r.t0 + j + 1, ROW_PAIR, c, a.B + b, r.d0 + j + 1});
          GST(&a.list[a.B + b].slot, -1);
        } else {
          GST(a.list + (b), RowTask{b, r.t0 + j + 1, 0, c});
          GST(a.list + (a.B + b), RowTask{drow ? a.B + b : -1, r.d0 + j + 1, 1, c});
        }
      }
      return;
    }
    n = j;
  }
  finish_request(a, b, r, n, sample, ts, ds, lane);
  // positions after n+1 were never read
  for (int i = n + 1 + lane; i < K; i += 32) {
    if (a.out_pq) {
      GST(a.out_pq + (2LL * (r.d0 + i)), __int_as_float(0x7fc00000));
      GST(a.out_pq + (2LL * (r.d0 + i) + 1), __int_as_float(0x7fc00000));
    }
    if (a.out_rank) GST(a.out_rank + (r.d0 + i), -1);
    if (a.out_kl) GST(a.out_kl + (r.d0 + i), __int_as_float(0x7fc00000));
  }
  if (lane == 0) {
    GST(&a.list[b].slot, -1);
    GST(&a.list[a.B + b].slot, -1);
  }
}

// --------------------------------------------------- final-token sampler
// Tiles of SAMPLE_TILE elements; thread t of a SAMPLE_THREADS block owns
// elements [tile + 16 t, tile + 16 t + 16).
struct SampleSmem {
  float scratch[33];
  float wsum[SAMPLE_THREADS / 32];
  float csum[64];            // per-tile sums inside one chunk (<= 16 tiles)
  float cwarp[64 * (SAMPLE_THREADS / 32)];   // per-warp sums of those tiles
  float corr[MAX_SAMPLE_TILES];  // chunk masses / tile sums of one row
  int s_idx[SPEC_TOPK];
  float s_prob[SPEC_TOPK];
  float pmin[SPEC_TOPK];
  int n_sparse;
  int jstar;
  float carry, target, Z;
  int xmin, xlast;
  int kind;
};

// Weights of this thread's SAMPLE_EPT elements of tile j: the residual
// max(0, p - q) (kind 1) or p (kind 2).
// (tile_weights_z: the same from target logits z already loaded; x0 is the
// thread's first element.)
template <int DK>
__device__ __forceinline__ void tile_weights_z(const LinearArgs &a, const SampleSmem &sh,
                                               const float *z, int x0, const char *drow,
                                               bool dvec, int kind, float c, float mt,
                                               float invSt, float md, float invSd, float *w) {
#pragma unroll
  for (int k = 0; k < SAMPLE_EPT; ++k) w[k] = ex2((z[k] - mt) * c) * invSt;
  if (kind != 1) return;
  if (DK == SPEC_DRAFT_SPARSE128) {
    // sorted ids: walk the ones inside [x0, x0 + EPT)
    int lo = 0, hi = sh.n_sparse;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sh.s_idx[mid] < x0) lo = mid + 1; else hi = mid;
    }
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k) {
      float q = 0.f;
      if (lo < sh.n_sparse && sh.s_idx[lo] == x0 + k) { q = sh.s_prob[lo]; ++lo; }
      w[k] = fmaxf(0.f, w[k] - q);
    }
    return;
  }
  float y[SAMPLE_EPT];
  if (DK == SPEC_DRAFT_PROBS) {
    load_ept(drow, a.ddt, dvec, x0, a.V, 0.f, y);
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k) w[k] = fmaxf(0.f, w[k] - y[k]);
  } else {
    load_ept(drow, a.ddt, dvec, x0, a.V, -INFINITY, y);
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k) w[k] = fmaxf(0.f, w[k] - ex2((y[k] - md) * c) * invSd);
  }
}

template <int DK>
__device__ __forceinline__ void tile_weights(const LinearArgs &a, const SampleSmem &sh,
                                             const char *trow, bool tvec, const char *drow,
                                             bool dvec, int kind, float c, float mt,
                                             float invSt, float md, float invSd, int j,
                                             float *w) {
  const int x0 = j * SAMPLE_TILE + (int)threadIdx.x * SAMPLE_EPT;
  float z[SAMPLE_EPT];
  load_ept(trow, a.tdt, tvec, x0, a.V, -INFINITY, z);
  tile_weights_z<DK>(a, sh, z, x0, drow, dvec, kind, c, mt, invSt, md, invSd, w);
}

// A thread's SAMPLE_EPT target logits of tile j as raw 16-byte vectors
// (bf16: two, f32: four), loaded without being used, so that several tiles'
// loads are in flight at once; `full` is false for a tile the vectors do not
// cover (a ragged end, an unaligned row), whose logits load_ept reads later.
struct RawEpt {
  uint4 v[SAMPLE_EPT / 4];
  bool full;
};
__device__ __forceinline__ void load_raw_ept(const char *row, int dt, bool vec_ok, int x0, int V,
                                             RawEpt &r) {
  r.full = vec_ok && x0 + SAMPLE_EPT <= V;
  if (!r.full) return;
  const int esz = dt == SPEC_BF16 ? 2 : 4;
  const uint4 *p = reinterpret_cast<const uint4 *>(row + (long long)esz * x0);
#pragma unroll
  for (int k = 0; k < SAMPLE_EPT / 4; ++k)
    if (k < SAMPLE_EPT * esz / 16) r.v[k] = GLDG(p + k);
}
// The logits of a RawEpt, as load_ept gives them.
__device__ __forceinline__ void raw_to_z(const RawEpt &r, const char *row, int dt, bool vec_ok,
                                         int x0, int V, float *z) {
  if (!r.full) {
    load_ept(row, dt, vec_ok, x0, V, -INFINITY, z);
    return;
  }
  if (dt == SPEC_BF16) {
#pragma unroll
    for (int q = 0; q < SAMPLE_EPT / 8; ++q) {
      const uint4 w = r.v[q];
      z[8 * q + 0] = bf16lo(w.x); z[8 * q + 1] = bf16hi(w.x);
      z[8 * q + 2] = bf16lo(w.y); z[8 * q + 3] = bf16hi(w.y);
      z[8 * q + 4] = bf16lo(w.z); z[8 * q + 5] = bf16hi(w.z);
      z[8 * q + 6] = bf16lo(w.w); z[8 * q + 7] = bf16hi(w.w);
    }
  } else {
#pragma unroll
    for (int q = 0; q < SAMPLE_EPT / 4; ++q) {
      const uint4 w = r.v[q];
      z[4 * q + 0] = __uint_as_float(w.x); z[4 * q + 1] = __uint_as_float(w.y);
      z[4 * q + 2] = __uint_as_float(w.z); z[4 * q + 3] = __uint_as_float(w.w);
    }
  }
}

// Block sum of one float per thread in a fixed order (warp butterflies,
// then warp 0 over the warp sums); the result is returned to every thread.
__device__ __forceinline__ float block_sum(float v, SampleSmem &sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sh.wsum[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int q = 0; q < SAMPLE_THREADS / 32; ++q) t += sh.wsum[q];
    sh.scratch[32] = t;
  }
  __syncthreads();
  const float t = sh.scratch[32];
  __syncthreads();
  return t;
}

// Residual tile sums of the dense-draft residual draws. Persistent blocks
// take (job, pair of tiles) items from a counter; the loads of both tiles are
// issued before any arithmetic, so every SM keeps many rows' bytes in flight.
constexpr int TILES_PER_ITEM = 2;

template <int DK>
__global__ void __launch_bounds__(SAMPLE_THREADS) k_sample_tiles(const LinearArgs a) {
  __shared__ SampleSmem sh;
  __shared__ int s_item;
  const int na = *(volatile int *)&a.hdr->n_jobs_a;
  const int ipj = (a.ntiles + TILES_PER_ITEM - 1) / TILES_PER_ITEM;
  const long long n_items = (long long)na * ipj;
  while (true) {
    if (threadIdx.x == 0) s_item = (int)atomicAdd(&a.hdr->work2, 1u);
    __syncthreads();
    const long long item = s_item;
    __syncthreads();
    if (item >= n_items) return;
    const int ja = (int)(item / ipj);
    const int j0 = (int)(item % ipj) * TILES_PER_ITEM;
    const Job job = GLD(a.jobs_a + (ja));
    const JobRows q = job_rows(a, job);
    const int xa = j0 * SAMPLE_TILE + (int)threadIdx.x * SAMPLE_EPT;
    const bool fast = DK == SPEC_DRAFT_LOGITS && a.tdt == SPEC_BF16 && a.ddt == SPEC_BF16 &&
                      q.tvec && q.dvec && j0 + TILES_PER_ITEM <= a.ntiles &&
                      (j0 + TILES_PER_ITEM) * SAMPLE_TILE <= a.V;
    if (fast) {
      // both tiles' packed bf16 in registers first, arithmetic after
      uint4 rt[TILES_PER_ITEM][2], rd[TILES_PER_ITEM][2];
#pragma unroll
      for (int u = 0; u < TILES_PER_ITEM; ++u) {
        const uint4 *pt = reinterpret_cast<const uint4 *>(q.trow + 2LL * (xa + u * SAMPLE_TILE));
        const uint4 *pd = reinterpret_cast<const uint4 *>(q.drow + 2LL * (xa + u * SAMPLE_TILE));
        rt[u][0] = GLDG(pt); rt[u][1] = GLDG(pt + 1);
        rd[u][0] = GLDG(pd); rd[u][1] = GLDG(pd + 1);
      }
#pragma unroll
      for (int u = 0; u < TILES_PER_ITEM; ++u) {
        float s = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t wt[4] = {rt[u][h].x, rt[u][h].y, rt[u][h].z, rt[u][h].w};
          const uint32_t wd[4] = {rd[u][h].x, rd[u][h].y, rd[u][h].z, rd[u][h].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float p0 = ex2((bf16lo(wt[k]) - q.mt) * q.c) * q.invSt;
            const float p1 = ex2((bf16hi(wt[k]) - q.mt) * q.c) * q.invSt;
            const float q0 = ex2((bf16lo(wd[k]) - q.md) * q.c) * q.invSd;
            const float q1 = ex2((bf16hi(wd[k]) - q.md) * q.c) * q.invSd;
            s += fmaxf(0.f, p0 - q0) + fmaxf(0.f, p1 - q1);
          }
        }
        const float t = block_sum(s, sh);
        if (threadIdx.x < RS_CONS_WARPS)
          GST(a.tsum + (((long long)ja * a.ntiles + j0 + u) * RS_CONS_WARPS + threadIdx.x), threadIdx.x == 0 ? t : 0.f);
      }
    } else {
      for (int u = 0; u < TILES_PER_ITEM && j0 + u < a.ntiles; ++u) {
        float zt[SAMPLE_EPT], zd[SAMPLE_EPT];
        const int x0 = xa + u * SAMPLE_TILE;
        load_ept(q.trow, a.tdt, q.tvec, x0, a.V, -INFINITY, zt);
        load_ept(q.drow, a.ddt, q.dvec, x0, a.V, DK == SPEC_DRAFT_PROBS ? 0.f : -INFINITY, zd);
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < SAMPLE_EPT; ++k) {
          const float p = ex2((zt[k] - q.mt) * q.c) * q.invSt;
          const float qq = DK == SPEC_DRAFT_PROBS ? zd[k] : ex2((zd[k] - q.md) * q.c) * q.invSd;
          s += fmaxf(0.f, p - qq);
        }
        const float t = block_sum(s, sh);
        if (threadIdx.x < RS_CONS_WARPS)
          GST(a.tsum + (((long long)ja * a.ntiles + j0 + u) * RS_CONS_WARPS + threadIdx.x), threadIdx.x == 0 ? t : 0.f);
      }
    }
  }
}

// Inverse-CDF step inside tile js: the smallest x with carry + C(x) > target,
// else the last positive weight of the tile (rounding). Every thread returns x.
template <int DK>
__device__ int fine_draw(const LinearArgs &a, SampleSmem &sh, const JobRows &q, int kind, int js) {
  if (threadIdx.x == 0) {
    sh.xmin = 0x7fffffff;
    sh.xlast = -1;
  }
  __syncthreads();
  float w[SAMPLE_EPT];
  tile_weights<DK>(a, sh, q.trow, q.tvec, q.drow, q.dvec, kind, q.c, q.mt, q.invSt, q.md,
                   q.invSd, js, w);
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < SAMPLE_EPT; ++k) s += w[k];
  float tot;
  const float excl = block_excl_scan(s, sh.scratch, &tot);
  const int x0 = js * SAMPLE_TILE + (int)threadIdx.x * SAMPLE_EPT;
  float pre = 0.f;
  int cand = 0x7fffffff, lastpos = -1;
#pragma unroll
  for (int k = 0; k < SAMPLE_EPT; ++k) {
    pre += w[k];
    if (cand == 0x7fffffff && sh.carry + (excl + pre) > sh.target) cand = x0 + k;
    if (w[k] > 0.f) lastpos = x0 + k;
  }
  if (cand != 0x7fffffff) atomicMin(&sh.xmin, cand);
  if (lastpos >= 0) atomicMax(&sh.xlast, lastpos);
  __syncthreads();
  const int x = sh.xmin != 0x7fffffff ? sh.xmin : sh.xlast;
  __syncthreads();
  return x;
}

// Bonus draws and sparse residual draws: the chunk holding the target mass
// is found from the row pass's per-chunk statistics of the target row (minus
// the sparse corrections min(p, q) at the listed ids), so only that chunk of
// the row is read again.
template <int DK, bool BATCH>
__device__ int chunk_draw(const LinearArgs &a, SampleSmem &sh, const Job &job, const JobRows &q,
                          int kind, float u) {
  const ReqInfo r = GLD(a.req + (job.b));
  const int esz = dtype_size(a.tdt);
  const int chunk_elems = a.chunk_bytes / esz;
  const int tpc = chunk_elems / SAMPLE_TILE;  // tiles per chunk
  const int nch = a.nch_t;
  const Part *pp = a.part + (long long)tslot(a, r, job.b, job.n) * a.nch_max * RS_CONS_WARPS;
  const bool sparse_res = kind == 1 && DK == SPEC_DRAFT_SPARSE128;
  if (sparse_res && threadIdx.x < sh.n_sparse) {   // min(p, q) at every listed id
    const int id = sh.s_idx[threadIdx.x];
    const float p = ex2((load_elem(q.trow, a.tdt, id) - q.mt) * q.c) * q.invSt;
    sh.pmin[threadIdx.x] = fminf(p, sh.s_prob[threadIdx.x]);
  }
  if (sparse_res) __syncthreads();
  for (int ch = threadIdx.x; ch < nch; ch += blockDim.x) {
    float m = 0.f;
    for (int w = 0; w < RS_CONS_WARPS; ++w) {
      const Part p = GLD(pp + ch * RS_CONS_WARPS + w);
      m += p.S * ex2((p.m - q.mt) * q.c);
    }
    m *= q.invSt;   // chunk mass of p
    if (sparse_res)   // less min(p, q) at the chunk's listed ids, in id order
      for (int k = 0; k < sh.n_sparse; ++k)
        if (sh.s_idx[k] / chunk_elems == ch) m -= sh.pmin[k];
    sh.corr[ch] = m;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float Z = 0.f;
    for (int ch = 0; ch < nch; ++ch) Z += fmaxf(sh.corr[ch], 0.f);
    sh.Z = Z;
    sh.target = u * Z;
    float carry = 0.f;
    int cs = -1;
    for (int ch = 0; ch < nch; ++ch) {
      const float nc = carry + fmaxf(sh.corr[ch], 0.f);
      if (nc > sh.target) { cs = ch; break; }
      carry = nc;
    }
    if (cs < 0)
      for (int ch = nch - 1; ch >= 0 && cs < 0; --ch)
        if (sh.corr[ch] > 0.f) cs = ch;
    sh.jstar = cs;
    sh.carry = carry;
  }
  __syncthreads();
  const int cs = sh.jstar;
  if (cs < 0) return -1;
  // tile sums inside the chunk in one sweep (per-warp sums, one sync), then
  // the tile, then the element
  const int j0 = cs * tpc, j1 = min(a.ntiles, j0 + tpc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float w[SAMPLE_EPT];
  if constexpr (BATCH) {
    // the weights read only the target row here (the bonus law, or a
    // residual against a sparse law held in shared memory): the target loads
    // of SWEEP_BATCH tiles are issued before the first of them is used (more
    // registers per thread, fewer blocks per SM)
    constexpr int SWEEP_BATCH = 4;
    for (int jb = j0; jb < j1; jb += SWEEP_BATCH) {
      RawEpt raw[SWEEP_BATCH];
#pragma unroll
      for (int u = 0; u < SWEEP_BATCH; ++u)
        if (jb + u < j1)
          load_raw_ept(q.trow, a.tdt, q.tvec,
                       (jb + u) * SAMPLE_TILE + (int)threadIdx.x * SAMPLE_EPT, a.V, raw[u]);
#pragma unroll
      for (int u = 0; u < SWEEP_BATCH; ++u) {
        const int j = jb + u;
        if (j >= j1) break;
        const int x0 = j * SAMPLE_TILE + (int)threadIdx.x * SAMPLE_EPT;
        float z[SAMPLE_EPT];
        raw_to_z(raw[u], q.trow, a.tdt, q.tvec, x0, a.V, z);
        // a residual against a sparse law sums p here; the listed ids'
        // min(p, q) come off each tile's sum below
        tile_weights_z<DK>(a, sh, z, x0, q.drow, q.dvec, sparse_res ? 2 : kind, q.c, q.mt,
                           q.invSt, q.md, q.invSd, w);
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < SAMPLE_EPT; ++k) s += w[k];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) sh.cwarp[(j - j0) * (SAMPLE_THREADS / 32) + warp] = s;
      }
    }
  } else {
#pragma unroll 4
    for (int j = j0; j < j1; ++j) {
      tile_weights<DK>(a, sh, q.trow, q.tvec, q.drow, q.dvec, kind, q.c, q.mt, q.invSt, q.md,
                       q.invSd, j, w);
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < SAMPLE_EPT; ++k) s += w[k];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) sh.cwarp[(j - j0) * (SAMPLE_THREADS / 32) + warp] = s;
    }
  }
  __syncthreads();
  if (threadIdx.x < j1 - j0) {
    float t = 0.f;
    for (int q2 = 0; q2 < SAMPLE_THREADS / 32; ++q2)
      t += sh.cwarp[threadIdx.x * (SAMPLE_THREADS / 32) + q2];
    if (BATCH && sparse_res) {   // max(0, p - q) = p - min(p, q) at the listed ids
      const int x_lo = (j0 + (int)threadIdx.x) * SAMPLE_TILE, x_hi = x_lo + SAMPLE_TILE;
      for (int k = 0; k < sh.n_sparse; ++k) {
        const int id = sh.s_idx[k];
        if (id >= x_lo && id < x_hi) t -= sh.pmin[k];
      }
      t = fmaxf(t, 0.f);
    }
    sh.csum[threadIdx.x] = t;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float carry = sh.carry;
    int js = -1;
    for (int j = j0; j < j1; ++j) {
      const float nc = carry + sh.csum[j - j0];
      if (nc > sh.target) { js = j; break; }
      carry = nc;
    }
    if (js < 0)
      for (int j = j1 - 1; j >= j0 && js < 0; --j)
        if (sh.csum[j - j0] > 0.f) js = j;
    sh.jstar = js;
    sh.carry = carry;
  }
  __syncthreads();
  const int js = sh.jstar;
  if (js < 0) return -1;
  return fine_draw<DK>(a, sh, q, kind, js);
}

// JOBS: the queues the launch serves. The first queue holds the dense
// residual draws (tile sums already made; one tile is read), the second the
// bonus draws and the residual draws against sparse laws (a chunk of the
// target row is swept first). SAMPLE_JOBS_ALL serves both in one launch;
// SAMPLE_JOBS_B only the second, with the sweep's loads batched, for calls
// whose draws are all there (sparse laws). Measured: a second launch for the
// dense calls' bonus draws costs more than the batched sweep saves.
constexpr int SAMPLE_JOBS_ALL = 0, SAMPLE_JOBS_B = 2;
template <int DK, int JOBS>
__global__ void __launch_bounds__(SAMPLE_THREADS) k_sample_final(const LinearArgs a) {
  __shared__ SampleSmem sh;
  const int g = blockIdx.x;
  const int na = JOBS == SAMPLE_JOBS_B ? 0 : *(volatile int *)&a.hdr->n_jobs_a;
  const int nb = *(volatile int *)&a.hdr->n_jobs_b;
  if (g >= na + nb) return;
  const bool dense = g < na;
  const Job job = dense ? GLD(a.jobs_a + (g)) : GLD(a.jobs_b + (g - na));
  const JobRows q = job_rows(a, job);
  const float u = uniform24(seed_of(a), (uint32_t)job.b, (uint32_t)(job.n + 1), job.kind == 1 ? 1u : 2u);
  int x = -1;
  bool done = false;
  if (dense) {
    // tile sums (the consumer warps' partials in a fixed order)
    const float *ts4 = a.tsum + (long long)g * a.ntiles * RS_CONS_WARPS;
    for (int j = threadIdx.x; j < a.ntiles; j += blockDim.x) {
      float t = 0.f;
      for (int w = 0; w < RS_CONS_WARPS; ++w) t += GLD(ts4 + j * RS_CONS_WARPS + w);
      sh.corr[j] = t;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      const float *ts = sh.corr;
      float Z = 0.f;
      for (int j = 0; j < a.ntiles; ++j) Z += ts[j];
      sh.Z = Z;
      sh.target = u * Z;
      float carry = 0.f;
      int js = -1;
      for (int j = 0; j < a.ntiles; ++j) {
        const float nc = carry + ts[j];
        if (nc > sh.target) { js = j; break; }
        carry = nc;
      }
      if (js < 0)
        for (int j = a.ntiles - 1; j >= 0 && js < 0; --j)
          if (ts[j] > 0.f) js = j;
      sh.jstar = js;
      sh.carry = carry;
    }
    __syncthreads();
    if (sh.Z > 0.f && sh.jstar >= 0) {
      x = fine_draw<DK>(a, sh, q, 1, sh.jstar);
      done = true;
    }
    // no residual mass (p == q): the same u draws from p
  } else if (DK == SPEC_DRAFT_SPARSE128 && job.kind == 1) {
    const ReqInfo r = GLD(a.req + (job.b));
    const int t = threadIdx.x;
    if (t < SPEC_TOPK) {   // the row's sparse law, sorted by id (bitonic)
      const long long row = (long long)(r.d0 + job.n) * SPEC_TOPK + t;
      const int id = GLD(a.draft_idx + (row));
      const bool ok = id >= 0 && id < a.V;
      sh.s_idx[t] = ok ? id : 0x7fffffff;
      sh.s_prob[t] = ok ? GLD(a.sparse_prob + (row)) : 0.f;
    }
    __syncthreads();
    // the internal top-128 returns its ids ascending (-1 padding last); a
    // caller's sparse law may list them in any order
    for (int size = 2; size <= SPEC_TOPK && a.rule != SPEC_RULE_STRICT_TOP128; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        if (t < SPEC_TOPK) {
          const int p = t ^ stride;
          if (p > t) {
            const bool up = (t & size) == 0;
            const int ka = sh.s_idx[t], kb = sh.s_idx[p];
            if ((ka > kb) == up) {
              sh.s_idx[t] = kb; sh.s_idx[p] = ka;
              const float fa = sh.s_prob[t];
              sh.s_prob[t] = sh.s_prob[p]; sh.s_prob[p] = fa;
            }
          }
        }
        __syncthreads();
      }
    }
    if (t == 0) {
      int cnt = 0;
      while (cnt < SPEC_TOPK && sh.s_idx[cnt] != 0x7fffffff) ++cnt;
      sh.n_sparse = cnt;
    }
    __syncthreads();
    x = chunk_draw<DK, JOBS == SAMPLE_JOBS_B>(a, sh, job, q, 1, u);
    done = sh.Z > 0.f;
  }
  if (!done)   // bonus, or residual without mass
    x = chunk_draw<DK, JOBS == SAMPLE_JOBS_B>(a, sh, job, q, 2, u);
  if (threadIdx.x == 0) {
    if (x < 0) set_status(a.hdr, SPEC_ERR_INVALID_ARG, job.b);   // a row without mass
    GST(a.out_tokens + ((long long)job.b * (a.max_k + 1) + job.n), x);
  }
}

// Calls whose rows total at most this many bytes, with rows of at most
// SMALL_V elements and a request's rows at most SMALL_REQUEST_BYTES, run as
// one fused kernel; 0 turns that off. Longer rows are faster on the
// multi-kernel path (measured: V = 32000 bf16, 16 and 64 requests).
static size_t g_small_limit = (size_t)32 << 20;
constexpr size_t SMALL_REQUEST_BYTES = (size_t)1 << 20;
constexpr int SMALL_V = 8192;

bool small_supported(const LinearArgs &a, const spec_linear_ext *ext) {
  if (ext != nullptr && (ext->flags != 0 || ext->out_kl != nullptr || ext->out_rank != nullptr))
    return false;
  if ((a.rule != SPEC_RULE_STRICT && a.rule != SPEC_RULE_GREEDY) ||
      (a.dk != SPEC_DRAFT_LOGITS && a.dk != SPEC_DRAFT_PROBS))
    return false;
  if (a.V > SMALL_V) return false;
  const size_t drow = (size_t)a.V * (a.ddt == SPEC_BF16 ? 2 : 4);
  const size_t per_req = (size_t)(a.max_k + 1) * (size_t)a.t_row_bytes + (size_t)a.max_k * drow;
  return per_req <= SMALL_REQUEST_BYTES && (size_t)a.B * per_req <= g_small_limit;
}

}  // namespace sv

using namespace sv;


extern "C" size_t spec_set_fused_limit(size_t bytes) {
  const size_t old = g_small_limit;
  g_small_limit = bytes;
  return old;
}

extern "C" size_t spec_verify_linear_workspace(int B, int max_k, int V, int rule) {
  if (B < 0 || max_k < 0 || max_k > SPEC_MAX_K || V <= 0 || V > SPEC_MAX_V) return 0;
  if (rule < SPEC_RULE_STRICT || rule > SPEC_RULE_CACTUS) return 0;
  return linear_layout(B, max_k, V, rule).total;
}

extern "C" int spec_verify_linear(const void *target, int tdt, const void *draft, int ddt,
                                  int dk, const int32_t *draft_idx,
                                  const int32_t *draft_tokens, const int32_t *cu_draft,
                                  const float *temperature, int B, int V, int max_k,
                                  uint64_t seed, int rule, int32_t *out_tokens,
                                  int32_t *out_accepted, float *out_pq, void *workspace,
                                  size_t ws_bytes, spec_stream_t stream) {
  return spec_verify_linear_ext(target, tdt, draft, ddt, dk, draft_idx, draft_tokens, cu_draft,
                                temperature, B, V, max_k, seed, rule, nullptr, out_tokens,
                                out_accepted, out_pq, workspace, ws_bytes, stream);
}

extern "C" int spec_verify_linear_ext(const void *target, int tdt, const void *draft, int ddt,
                                      int dk, const int32_t *draft_idx,
                                      const int32_t *draft_tokens, const int32_t *cu_draft,
                                      const float *temperature, int B, int V, int max_k,
                                      uint64_t seed, int rule, const spec_linear_ext *ext,
                                      int32_t *out_tokens, int32_t *out_accepted,
                                      float *out_pq, void *workspace, size_t ws_bytes,
                                      spec_stream_t stream) {
  if (B < 0 || V <= 0 || V > SPEC_MAX_V || max_k < 0) return SPEC_ERR_INVALID_ARG;
  if (max_k > SPEC_MAX_K) return SPEC_ERR_UNSUPPORTED;
  if ((tdt != SPEC_F32 && tdt != SPEC_BF16) || (ddt != SPEC_F32 && ddt != SPEC_BF16))
    return SPEC_ERR_INVALID_ARG;
  if (dk < SPEC_DRAFT_LOGITS || dk > SPEC_DRAFT_SPARSE128) return SPEC_ERR_INVALID_ARG;
  if (rule < SPEC_RULE_STRICT || rule > SPEC_RULE_CACTUS) return SPEC_ERR_INVALID_ARG;
  if (rule == SPEC_RULE_STRICT_TOP128 && dk != SPEC_DRAFT_LOGITS) return SPEC_ERR_INVALID_ARG;
  if (rule == SPEC_RULE_CACTUS && ext == nullptr) return SPEC_ERR_INVALID_ARG;
  if (ext != nullptr &&
      (!(ext->alpha >= 0.f) || !isfinite(ext->alpha) || ext->max_rank < 0 ||
       !(ext->min_prob >= 0.f) || !isfinite(ext->min_prob) ||
       (ext->flags & ~(SPEC_EXT_LAZY | SPEC_EXT_RESIDENT | SPEC_EXT_EAGER)) != 0 ||
       ((ext->flags & SPEC_EXT_EAGER) && (ext->flags & ~SPEC_EXT_EAGER)) ||
       !aligned(ext->out_kl, 4) ||
       !aligned(ext->out_rank, 4) || !aligned(ext->seed_dev, 8)))
    return SPEC_ERR_INVALID_ARG;
  if (dk == SPEC_DRAFT_SPARSE128 && (ddt != SPEC_F32 || draft_idx == nullptr || draft == nullptr))
    return SPEC_ERR_INVALID_ARG;
  if (B > 0 && (target == nullptr || draft_tokens == nullptr || cu_draft == nullptr ||
                temperature == nullptr || out_tokens == nullptr || out_accepted == nullptr))
    return SPEC_ERR_INVALID_ARG;
  if (!aligned(target, 16) || !aligned(draft, 16) || !aligned(draft_idx, 4) ||
      !aligned(draft_tokens, 4) || !aligned(cu_draft, 4) || !aligned(temperature, 4) ||
      !aligned(out_tokens, 4) || !aligned(out_accepted, 4) || !aligned(out_pq, 4))
    return SPEC_ERR_INVALID_ARG;
  const LinearLayout L = linear_layout(B, max_k, V, rule);
  if (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < L.total)
    return SPEC_ERR_WORKSPACE;

  char *ws = static_cast<char *>(workspace);
  LinearArgs a;
  a.target = static_cast<const char *>(target);
  a.draft = static_cast<const char *>(draft);
  a.tdt = tdt;
  a.ddt = ddt;
  a.dk = dk;
  a.rule = rule;
  a.tokens = draft_tokens;
  a.cu = cu_draft;
  a.temp = temperature;
  a.B = B;
  a.V = V;
  a.max_k = max_k;
  a.seed = seed;
  a.seed_dev = ext ? ext->seed_dev : nullptr;
  a.out_tokens = out_tokens;
  a.out_accepted = out_accepted;
  a.out_pq = out_pq;
  a.hdr = reinterpret_cast<WsHeader *>(ws + L.hdr);
  a.err = a.hdr;
  a.req = reinterpret_cast<ReqInfo *>(ws + L.req);
  a.jobs_a = reinterpret_cast<Job *>(ws + L.jobs_a);
  a.jobs_b = reinterpret_cast<Job *>(ws + L.jobs_b);
  a.tsum = reinterpret_cast<float *>(ws + L.tsum);
  a.ntiles = (V + SAMPLE_TILE - 1) / SAMPLE_TILE;
  a.rows_max = L.rows_max;
  a.list = reinterpret_cast<RowTask *>(ws + L.list);
  a.part = reinterpret_cast<Part *>(ws + L.part);
  a.t_row_bytes = (long long)V * (tdt == SPEC_BF16 ? 2 : 4);
  a.d_row_bytes = dk == SPEC_DRAFT_SPARSE128 ? (long long)SPEC_TOPK * 4
                                             : (long long)V * (ddt == SPEC_BF16 ? 2 : 4);
  const int flags = ext ? ext->flags : 0;
  const bool lazy = (flags & (SPEC_EXT_LAZY | SPEC_EXT_RESIDENT)) != 0;
  const bool want_kl = ext && ext->out_kl != nullptr;
  if (want_kl && (dk != SPEC_DRAFT_LOGITS || rule == SPEC_RULE_STRICT_TOP128 || tdt != ddt ||
                  ((long long)V * (tdt == SPEC_BF16 ? 2 : 4)) % 16 != 0))
    return SPEC_ERR_INVALID_ARG;
  // pairs split each row into chunks of 32768 elements (the slots' chunk
  // capacity); lazy rounds keep their finer chunks
  a.chunk_bytes = lazy ? LAZY_CHUNK_BYTES
                       : want_kl ? 32768 * (tdt == SPEC_BF16 ? 2 : 4) : CHUNK_BYTES;
  a.nch_t = nchunks(V, tdt, a.chunk_bytes);
  a.nch_d = nchunks(V, ddt, a.chunk_bytes);
  a.nch_max = lazy ? L.nch_max_lazy : L.nch_max;
  a.rt_max = B * (max_k + 1);
  a.sparse = dk == SPEC_DRAFT_SPARSE128 || rule == SPEC_RULE_STRICT_TOP128;
  a.stream_draft = dk == SPEC_DRAFT_LOGITS && rule != SPEC_RULE_STRICT_TOP128;
  a.alpha = ext ? ext->alpha : 0.f;
  a.min_prob = ext ? ext->min_prob : 0.f;
  a.max_rank = ext ? ext->max_rank : 0;
  a.out_rank = ext ? ext->out_rank : nullptr;
  a.want_rank = a.out_rank != nullptr || (rule == SPEC_RULE_CACTUS && a.max_rank > 0);
  a.lazy = lazy ? 1 : 0;
  a.want_kl = want_kl ? 1 : 0;
  a.out_kl = want_kl ? ext->out_kl : nullptr;
  a.kl_part = reinterpret_cast<float *>(ws + L.kl_part);
  a.round = 0;
  a.rank_thr = reinterpret_cast<float *>(ws + L.rank_thr);
  if (dk == SPEC_DRAFT_SPARSE128) {
    a.draft_idx = draft_idx;
    a.sparse_prob = static_cast<const float *>(draft);
  } else if (rule == SPEC_RULE_STRICT_TOP128) {
    a.draft_idx = reinterpret_cast<int32_t *>(ws + L.tk_idx);
    a.sparse_prob = reinterpret_cast<float *>(ws + L.tk_prob);
  } else {
    a.draft_idx = nullptr;
    a.sparse_prob = nullptr;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  if (cudaMemsetAsync(a.hdr, 0, sizeof(WsHeader), st) != cudaSuccess) return SPEC_ERR_CUDA;
  if (B == 0) return SPEC_OK;
#ifdef SPEC_CHECKED
  {   // the call's buffers, sized by its row count cu_draft[B]
    int Rd = 0;
    if (check_read_int(cu_draft + B, st, &Rd) != SPEC_OK) return SPEC_ERR_CUDA;
    const long long rd = Rd > 0 ? Rd : 0;
    check_begin(a.hdr);
    check_add(workspace, L.total);
    check_add(target, (rd + B) * a.t_row_bytes);
    check_add(draft, rd * a.d_row_bytes);
    check_add(draft_idx, rd * SPEC_TOPK * 4);
    check_add(draft_tokens, rd * 4);
    check_add(cu_draft, (B + 1) * 4ull);
    check_add(temperature, B * 4ull);
    check_add(out_tokens, (unsigned long long)B * (max_k + 1) * 4);
    check_add(out_accepted, B * 4ull);
    check_add(out_pq, rd * 8);
    check_add(a.out_rank, rd * 4);
    check_add(a.out_kl, rd * 4);
    check_add(a.seed_dev, 8);
  }
#endif
  if (check_upload(st) != SPEC_OK) return SPEC_ERR_CUDA;
  a.ent_d = reinterpret_cast<StreamEntry *>(ws + L.ent_d);
  a.ready_d = reinterpret_cast<int *>(ws + L.ready_d);
  a.pos_done = reinterpret_cast<int *>(ws + L.pos_done);
  a.pos_join = reinterpret_cast<int *>(ws + L.pos_join);
  a.rej_at = reinterpret_cast<int *>(ws + L.rej_at);
  a.zd_at = reinterpret_cast<float *>(ws + L.zd_at);
  a.cap_d = B;
  a.n_res_items = (a.ntiles + RES_TILES_PER_ITEM - 1) / RES_TILES_PER_ITEM;
  if (small_supported(a, ext)) return launch_verify_small(a, st);
  if (cluster_small_supported(a, ext, g_small_limit)) return launch_verify_cluster_small(a, st);
  if ((flags & SPEC_EXT_RESIDENT) && resident_supported(a)) {
    // position-lazy schedule with each position's rows resident on chip
    // (setup, then one persistent cluster kernel that also draws)
    a.lazy = 0;
    return launch_verify_resident(a, st);
  }
  // the streaming schedule: asked for, or a plain call (no per-position
  // outputs, no option) whose inputs it takes
  const bool plain = !(flags & SPEC_EXT_EAGER) && out_pq == nullptr && !want_kl &&
                     a.out_rank == nullptr && (rule == SPEC_RULE_STRICT || rule == SPEC_RULE_GREEDY);
  if ((a.lazy || plain) && stream_supported(a)) {
    // partial slots by absolute row (as the eager schedule), in the
    // streaming verifier's chunks
    a.lazy = 0;
    a.chunk_bytes = STREAM_CHUNK_BYTES;
    a.nch_t = nchunks(V, tdt, a.chunk_bytes);
    a.nch_d = nchunks(V, ddt, a.chunk_bytes);
    a.nch_max = L.nch_max_stream;
    a.stride = a.nch_t + a.nch_d;
    // position-lazy schedule in one persistent kernel; decisions report
    // invalid inputs through a second header, merged at the end
    a.err = reinterpret_cast<WsHeader *>(ws + L.err);
    if (cudaMemsetAsync(a.err, 0, sizeof(WsHeader), st) != cudaSuccess) return SPEC_ERR_CUDA;
    const int rc = launch_verify_stream(a, st);
    if (rc != SPEC_OK) return rc;
    k_sample_final<SPEC_DRAFT_LOGITS, SAMPLE_JOBS_ALL><<<B, SAMPLE_THREADS, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
  }
  k_setup_linear<<<(B + 63) / 64, 64, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (rule == SPEC_RULE_STRICT_TOP128) {
    // the top-128 select reads every draft row and dominates this rule's
    // call: profiling events, if registered, bracket its launch that reads
    // the rows
    cudaEvent_t before, after;
    take_row_pass_events(&before, &after);
    const int rc = launch_topk128(draft, ddt, B * max_k, V, cu_draft, temperature, B,
                                  reinterpret_cast<int32_t *>(ws + L.tk_idx),
                                  reinterpret_cast<float *>(ws + L.tk_prob), a.hdr, st, nullptr,
                                  ws + L.tk_list, before, after);
    if (rc != SPEC_OK) return rc;
  }
  RowPassArgs rp;
  rp.base[0] = a.target;
  rp.base[1] = a.draft;
  rp.row_bytes[0] = a.t_row_bytes;
  rp.row_bytes[1] = (long long)V * (ddt == SPEC_BF16 ? 2 : 4);
  rp.dtype[0] = tdt;
  rp.dtype[1] = ddt;
  rp.nch[0] = a.nch_t;
  rp.nch[1] = a.nch_d;
  rp.nch_max = a.nch_max;
  rp.chunk_bytes = a.chunk_bytes;
  rp.list = a.list;
  rp.hdr = a.hdr;
  rp.part = a.part;
  rp.rank_thr = a.want_rank ? a.rank_thr : nullptr;
  rp.kl_part = a.want_kl ? a.kl_part : nullptr;
  rp.residual = 0;
  rp.jobs = nullptr;
  rp.req = nullptr;
  rp.tsum4 = nullptr;
  rp.ntiles = 0;
  rp.V = V;
  int rc;
  if (a.lazy) {
    // profiling events, if any, bracket all rounds (row passes and decisions)
    cudaEvent_t before, after;
    take_row_pass_events(&before, &after);
    if (before && cudaEventRecord(before, st) != cudaSuccess) return SPEC_ERR_CUDA;
    for (int j = 0; j <= max_k; ++j) {
      rc = launch_row_pass(rp, st);
      if (rc != SPEC_OK) return rc;
      a.round = j;
      k_lazy_decide<<<(B + ACCEPT_WARPS - 1) / ACCEPT_WARPS, ACCEPT_WARPS * 32, 0, st>>>(a);
      if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
    }
    if (after && cudaEventRecord(after, st) != cudaSuccess) return SPEC_ERR_CUDA;
  } else {
    rc = launch_row_pass(rp, st);
    if (rc != SPEC_OK) return rc;
    k_accept<<<(B + ACCEPT_WARPS - 1) / ACCEPT_WARPS, ACCEPT_WARPS * 32, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  }
  const int tiles_grid = 8 * num_sms();
  if (a.sparse) {   // every draw is in the second queue
    k_sample_final<SPEC_DRAFT_SPARSE128, SAMPLE_JOBS_B><<<B, SAMPLE_THREADS, 0, st>>>(a);
  } else if (dk == SPEC_DRAFT_PROBS) {
    k_sample_tiles<SPEC_DRAFT_PROBS><<<tiles_grid, SAMPLE_THREADS, 0, st>>>(a);
    k_sample_final<SPEC_DRAFT_PROBS, SAMPLE_JOBS_ALL><<<B, SAMPLE_THREADS, 0, st>>>(a);
  } else {
    if (tdt == SPEC_BF16 && ddt == SPEC_BF16 && V % 8 == 0) {
      // residual tile pairs through the TMA row pass
      RowPassArgs rr = rp;
      rr.residual = 1;
      rr.jobs = a.jobs_a;
      rr.req = a.req;
      rr.tsum4 = a.tsum;
      rr.ntiles = a.ntiles;
      rr.V = V;
      rc = launch_row_pass(rr, st);
      if (rc != SPEC_OK) return rc;
    } else {
      k_sample_tiles<SPEC_DRAFT_LOGITS><<<tiles_grid, SAMPLE_THREADS, 0, st>>>(a);
    }
    k_sample_final<SPEC_DRAFT_LOGITS, SAMPLE_JOBS_ALL><<<B, SAMPLE_THREADS, 0, st>>>(a);
  }
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}
