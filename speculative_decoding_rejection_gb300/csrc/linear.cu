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
#include "common.cuh"
#include "internal.h"

namespace sv {

constexpr int ACCEPT_WARPS = 8;

struct FinalInfo {   // per request, written by the accept kernel
  int n;             // accepted drafts
  int kind;          // 0: final token already written, 1: residual, 2: bonus
  float mt, St;      // statistics of target row n+1
  float md, Sd;      // statistics of draft row n+1 (dense logits only)
  int pad[2];
};

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
  int32_t *out_tokens;
  int32_t *out_accepted;
  float *out_pq;
  WsHeader *hdr;
  ReqInfo *req;
  FinalInfo *fin;
  RowTask *list;
  Part *part;
  long long t_row_bytes, d_row_bytes;
  int nch_t, nch_d, nch_max;
  int rt_max;                 // slot offset of draft rows
  int sparse;                 // the draft law is sparse (given or top-128)
  int stream_draft;           // the row pass reads dense draft logits
};

struct LinearLayout {
  size_t hdr, req, fin, list, part, tk_idx, tk_prob, total;
  int nch_max;
  long long rows_max;
};

static LinearLayout linear_layout(int B, int max_k, int V, int rule) {
  LinearLayout L;
  L.nch_max = nchunks(V, SPEC_F32);
  L.rows_max = (long long)B * (2LL * max_k + 1);
  size_t o = 0;
  L.hdr = o;  o += align256(sizeof(WsHeader));
  L.req = o;  o += align256(sizeof(ReqInfo) * (size_t)B);
  L.fin = o;  o += align256(sizeof(FinalInfo) * (size_t)B);
  L.list = o; o += align256(sizeof(RowTask) * (size_t)L.rows_max);
  L.part = o; o += align256(sizeof(Part) * (size_t)L.rows_max * L.nch_max * RS_CONS_WARPS);
  const size_t tk = rule == SPEC_RULE_STRICT_TOP128 ? (size_t)B * max_k * SPEC_TOPK : 0;
  L.tk_idx = o;  o += align256(sizeof(int32_t) * tk);
  L.tk_prob = o; o += align256(sizeof(float) * tk);
  L.total = o;
  return L;
}

// ------------------------------------------------------------------ setup
__global__ void __launch_bounds__(1024) k_setup_linear(const LinearArgs a) {
  __shared__ int scratch[33];
  if (threadIdx.x == 0) {
    a.hdr->status = SPEC_OK;
    a.hdr->detail = -1;
    a.hdr->work = 0;
    a.hdr->n_list = 0;
  }
  __syncthreads();
  const int per = (a.B + blockDim.x - 1) / blockDim.x;
  const int b0 = min(a.B, (int)threadIdx.x * per), b1 = min(a.B, b0 + per);
  const bool cu0_ok = a.B == 0 || a.cu[0] == 0;
  int cnt = 0;
  for (int b = b0; b < b1; ++b) {
    ReqInfo r;
    const int K = a.cu[b + 1] - a.cu[b];
    const float T = a.temp[b];
    r.t0 = a.cu[b] + b;
    r.d0 = a.cu[b];
    r.K = K;
    r.n = 0;
    r.pad[0] = r.pad[1] = 0;
    const bool greedy = a.rule == SPEC_RULE_GREEDY || T < SPEC_GREEDY_T;
    bool ok = cu0_ok && K >= 0 && K <= a.max_k && a.cu[b] >= 0 && T >= 0.f && isfinite(T);
    if (ok && !greedy && a.draft == nullptr) ok = false;
    if (!ok) {
      set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);
      r.mode = MODE_SKIP;
      r.c = 0.f;
    } else {
      r.mode = greedy ? MODE_GREEDY : MODE_SAMPLE;
      r.c = greedy ? 0.f : (float)(1.4426950408889634 / (double)T);
      cnt += (K + 1) + ((r.mode == MODE_SAMPLE && a.stream_draft) ? K : 0);
    }
    a.req[b] = r;
  }
  // Row offsets of one request are only in bounds when all of cu_draft is
  // well formed, so any invalid request disables the whole call.
  int local_bad = 0;
  for (int b = b0; b < b1; ++b) local_bad |= a.req[b].mode == MODE_SKIP;
  if (__syncthreads_or(local_bad)) {
    for (int b = b0; b < b1; ++b) a.req[b].mode = MODE_SKIP;
    return;  // n_list stays 0
  }
  int total;
  int off = block_excl_scan_int(cnt, scratch, &total);
  for (int b = b0; b < b1; ++b) {
    const ReqInfo r = a.req[b];
    if (r.mode == MODE_SKIP) continue;
    for (int i = 0; i <= r.K; ++i) a.list[off++] = RowTask{r.t0 + i, r.t0 + i, 0, r.c};
    if (r.mode == MODE_SAMPLE && a.stream_draft)
      for (int i = 0; i < r.K; ++i) a.list[off++] = RowTask{a.rt_max + r.d0 + i, r.d0 + i, 1, r.c};
  }
  if (threadIdx.x == 0) a.hdr->n_list = total;
}

// ------------------------------------------------------------ accept scan
// Row statistics combined by the whole warp: lane l merges partials
// l, l+32, ..., then a butterfly merges the lanes (every lane gets the row's
// statistics; the merge order is fixed, so the result is deterministic).
__device__ __forceinline__ RowStat warp_row_stat(const Part *p, int n, float c, int lane) {
  float m = NO_MAX, S = 0.f;
  int idx = 0x7fffffff;
  for (int i = lane; i < n; i += 32) {
    const Part q = p[i];
    merge_stat(m, S, idx, q.m, q.S, q.idx, c);
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
__device__ __forceinline__ RowStat target_stat(const LinearArgs &a, int row, float c, int lane) {
  return warp_row_stat(a.part + (long long)row * a.nch_max * RS_CONS_WARPS,
                       a.nch_t * RS_CONS_WARPS, c, lane);
}
__device__ __forceinline__ RowStat draft_stat(const LinearArgs &a, int row, float c, int lane) {
  return warp_row_stat(a.part + (long long)(a.rt_max + row) * a.nch_max * RS_CONS_WARPS,
                       a.nch_d * RS_CONS_WARPS, c, lane);
}

// q(d) for draft row `row` given its statistics ds (dense logits), the
// probability itself, or a search of the sparse ids (any order).
__device__ float draft_prob_at(const LinearArgs &a, int row, int d, float c, RowStat ds) {
  if (a.sparse) {
    const int32_t *ids = a.draft_idx + (long long)row * SPEC_TOPK;
    const float *pr = a.sparse_prob + (long long)row * SPEC_TOPK;
    for (int k = 0; k < SPEC_TOPK; ++k)
      if (ids[k] == d) return pr[k];
    return 0.f;
  }
  const char *drow = a.draft + (long long)row * a.d_row_bytes;
  if (a.dk == SPEC_DRAFT_PROBS) return load_elem(drow, a.ddt, d);
  if (row_empty(ds.m)) return 0.f;
  return ex2((load_elem(drow, a.ddt, d) - ds.m) * c) / ds.S;
}

__global__ void __launch_bounds__(ACCEPT_WARPS * 32) k_accept(const LinearArgs a) {
  const int b = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= a.B) return;
  const ReqInfo r = a.req[b];
  const int W = a.max_k + 1;
  int32_t *out = a.out_tokens + (long long)b * W;
  if (r.mode == MODE_SKIP) {
    for (int j = lane; j < W; j += 32) out[j] = -1;
    if (lane == 0) {
      a.out_accepted[b] = -1;
      a.fin[b] = FinalInfo{0, 0, 0.f, 0.f, 0.f, 0.f, {0, 0}};
    }
    return;
  }
  const int K = r.K;
  const float c = r.c;
  const bool sample = r.mode == MODE_SAMPLE;
  int n = K;
  for (int base = 0; base < K; base += 32) {
    const int cnt = min(32, K - base);
    // statistics of this block of positions: lane i keeps position base + i
    RowStat ts{NO_MAX, 0.f, 0x7fffffff}, ds{NO_MAX, 0.f, 0x7fffffff};
    for (int i = 0; i < cnt; ++i) {
      const RowStat t = target_stat(a, r.t0 + base + i, c, lane);
      if (lane == i) ts = t;
      if (sample && a.stream_draft) {
        const RowStat d = draft_stat(a, r.d0 + base + i, c, lane);
        if (lane == i) ds = d;
      }
    }
    const int i = base + lane;
    bool rej = false;
    if (lane < cnt) {
      const int d = a.tokens[r.d0 + i];
      const bool dok = (unsigned)d < (unsigned)a.V;
      if (!dok) set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);
      if (row_empty(ts.m)) set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);
      float pd, qd;
      if (!sample) {
        rej = !(dok && d == ts.idx);
        pd = rej ? 0.f : 1.f;
        qd = -1.f;
      } else if (dok && !row_empty(ts.m)) {
        const char *trow = a.target + (long long)(r.t0 + i) * a.t_row_bytes;
        pd = ex2((load_elem(trow, a.tdt, d) - ts.m) * c) / ts.S;
        qd = draft_prob_at(a, r.d0 + i, d, c, ds);
        const float acc = qd <= pd ? 1.f : pd / qd;
        rej = !(uniform24(a.seed, (uint32_t)b, (uint32_t)(i + 1), 0) < acc);
      } else {
        pd = 0.f;
        qd = 0.f;
        rej = true;
      }
      if (a.out_pq) {
        a.out_pq[2LL * (r.d0 + i)] = pd;
        a.out_pq[2LL * (r.d0 + i) + 1] = qd;
      }
    }
    const unsigned bal = __ballot_sync(0xffffffffu, rej);
    if (n == K && bal) n = base + __ffs(bal) - 1;
  }
  for (int j = lane; j < W; j += 32) out[j] = j < n ? a.tokens[r.d0 + j] : -1;
  const RowStat tf = target_stat(a, r.t0 + n, c, lane);
  RowStat df{NO_MAX, 0.f, 0x7fffffff};
  if (sample && n < K && a.stream_draft) df = draft_stat(a, r.d0 + n, c, lane);
  __syncwarp();
  if (lane == 0) {
    a.out_accepted[b] = n;
    FinalInfo f{n, 0, 0.f, 0.f, 0.f, 0.f, {0, 0}};
    if (!sample) {
      out[n] = tf.idx;
    } else {
      f.kind = n < K ? 1 : 2;
      f.mt = tf.m;
      f.St = tf.S;
      f.md = df.m;
      f.Sd = df.S;
    }
    a.fin[b] = f;
  }
}

// --------------------------------------------------- final-token sampler
struct SampleSmem {
  float tsum[MAX_SAMPLE_TILES];
  float scratch[33];
  int s_idx[SPEC_TOPK];
  float s_prob[SPEC_TOPK];
  int n_sparse;
  int jstar;
  float carry, target, Z;
  int xmin, xlast;
};

// Weights of this thread's SAMPLE_EPT elements of tile j: the residual
// max(0, p - q) (kind 1) or p (kind 2).
template <int DK>
__device__ __forceinline__ void tile_weights(const LinearArgs &a, const SampleSmem &sh,
                                             const char *trow, bool tvec, const char *drow,
                                             bool dvec, int kind, float c, float mt,
                                             float invSt, float md, float invSd, int j,
                                             float *w) {
  const int x0 = j * SAMPLE_TILE + (int)threadIdx.x * SAMPLE_EPT;
  float z[SAMPLE_EPT];
  load_ept(trow, a.tdt, tvec, x0, a.V, -INFINITY, z);
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
__global__ void __launch_bounds__(SAMPLE_THREADS) k_sample(const LinearArgs a) {
  __shared__ SampleSmem sh;
  extern __shared__ float wsum[];   // [tiles][32 warps]
  const int b = blockIdx.x;
  const ReqInfo r = a.req[b];
  if (r.mode != MODE_SAMPLE) return;
  const FinalInfo f = a.fin[b];
  if (f.kind == 0) return;
  const int n = f.n;
  const float c = r.c;
  const char *trow = a.target + (long long)(r.t0 + n) * a.t_row_bytes;
  const bool tvec = ((uintptr_t)trow & 15) == 0;
  const char *drow = nullptr;
  bool dvec = false;
  if (f.kind == 1 && !a.sparse) {
    drow = a.draft + (long long)(r.d0 + n) * a.d_row_bytes;
    dvec = ((uintptr_t)drow & 15) == 0;
  }
  if (DK == SPEC_DRAFT_SPARSE128 && f.kind == 1) {
    // gather this row's sparse law and sort it by id (bitonic, 128 keys)
    const int t = threadIdx.x;
    if (t < SPEC_TOPK) {
      const int id = a.draft_idx[(long long)(r.d0 + n) * SPEC_TOPK + t];
      const bool ok = id >= 0 && id < a.V;
      sh.s_idx[t] = ok ? id : 0x7fffffff;
      sh.s_prob[t] = ok ? a.sparse_prob[(long long)(r.d0 + n) * SPEC_TOPK + t] : 0.f;
    }
    __syncthreads();
    for (int size = 2; size <= SPEC_TOPK; size <<= 1) {
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
  }
  __syncthreads();

  const float invSt = 1.f / f.St;
  const float invSd = f.Sd > 0.f ? 1.f / f.Sd : 0.f;
  const int ntiles = (a.V + SAMPLE_TILE - 1) / SAMPLE_TILE;
  int kind = f.kind;
  float u = uniform24(a.seed, (uint32_t)b, (uint32_t)(n + 1), kind == 1 ? 1u : 2u);
  float w[SAMPLE_EPT];
  for (int attempt = 0; attempt < 2; ++attempt) {
    // pass 1: per-warp sums of every tile, no block-wide sync inside the
    // streaming loop; then tile totals in a fixed order (warp 0)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll 2
    for (int j = 0; j < ntiles; ++j) {
      tile_weights<DK>(a, sh, trow, tvec, drow, dvec, kind, c, f.mt, invSt, f.md, invSd, j, w);
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < SAMPLE_EPT; ++k) s += w[k];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) wsum[j * 32 + warp] = s;
    }
    __syncthreads();
    if (warp == 0)
      for (int j = lane; j < ntiles; j += 32) {
        float t = 0.f;
        for (int q = 0; q < SAMPLE_THREADS / 32; ++q) t += wsum[j * 32 + q];
        sh.tsum[j] = t;
      }
    __syncthreads();
    if (threadIdx.x == 0) {
      float Z = 0.f;
      for (int j = 0; j < ntiles; ++j) Z += sh.tsum[j];
      sh.Z = Z;
      sh.target = u * Z;
      float carry = 0.f;
      int js = -1;
      for (int j = 0; j < ntiles; ++j) {
        const float nc = carry + sh.tsum[j];
        if (nc > sh.target) { js = j; break; }
        carry = nc;
      }
      if (js < 0)  // rounding left u*Z >= Z: the last tile with mass
        for (int j = ntiles - 1; j >= 0 && js < 0; --j)
          if (sh.tsum[j] > 0.f) js = j;
      sh.jstar = js;
      sh.carry = carry;
      sh.xmin = 0x7fffffff;
      sh.xlast = -1;
    }
    __syncthreads();
    if (sh.Z > 0.f || kind == 2) break;
    kind = 2;  // the residual has no mass (p == q): draw from p instead
  }
  const int js = sh.jstar;
  if (js >= 0) {
    tile_weights<DK>(a, sh, trow, tvec, drow, dvec, kind, c, f.mt, invSt, f.md, invSd, js, w);
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
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int x = sh.xmin != 0x7fffffff ? sh.xmin : sh.xlast;
    if (x < 0) {
      set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);  // a row without mass
      x = -1;
    }
    a.out_tokens[(long long)b * (a.max_k + 1) + n] = x;
  }
}

}  // namespace sv

using namespace sv;

extern "C" size_t spec_verify_linear_workspace(int B, int max_k, int V, int rule) {
  if (B < 0 || max_k < 0 || max_k > SPEC_MAX_K || V <= 0 || V > SPEC_MAX_V) return 0;
  if (rule < 0 || rule > 2) return 0;
  return linear_layout(B, max_k, V, rule).total;
}

extern "C" int spec_verify_linear(const void *target, int tdt, const void *draft, int ddt,
                                  int dk, const int32_t *draft_idx,
                                  const int32_t *draft_tokens, const int32_t *cu_draft,
                                  const float *temperature, int B, int V, int max_k,
                                  uint64_t seed, int rule, int32_t *out_tokens,
                                  int32_t *out_accepted, float *out_pq, void *workspace,
                                  size_t ws_bytes, spec_stream_t stream) {
  if (B < 0 || V <= 0 || V > SPEC_MAX_V || max_k < 0) return SPEC_ERR_INVALID_ARG;
  if (max_k > SPEC_MAX_K) return SPEC_ERR_UNSUPPORTED;
  if ((tdt != SPEC_F32 && tdt != SPEC_BF16) || (ddt != SPEC_F32 && ddt != SPEC_BF16))
    return SPEC_ERR_INVALID_ARG;
  if (dk < SPEC_DRAFT_LOGITS || dk > SPEC_DRAFT_SPARSE128) return SPEC_ERR_INVALID_ARG;
  if (rule < SPEC_RULE_STRICT || rule > SPEC_RULE_STRICT_TOP128) return SPEC_ERR_INVALID_ARG;
  if (rule == SPEC_RULE_STRICT_TOP128 && dk != SPEC_DRAFT_LOGITS) return SPEC_ERR_INVALID_ARG;
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
  a.out_tokens = out_tokens;
  a.out_accepted = out_accepted;
  a.out_pq = out_pq;
  a.hdr = reinterpret_cast<WsHeader *>(ws + L.hdr);
  a.req = reinterpret_cast<ReqInfo *>(ws + L.req);
  a.fin = reinterpret_cast<FinalInfo *>(ws + L.fin);
  a.list = reinterpret_cast<RowTask *>(ws + L.list);
  a.part = reinterpret_cast<Part *>(ws + L.part);
  a.t_row_bytes = (long long)V * (tdt == SPEC_BF16 ? 2 : 4);
  a.d_row_bytes = dk == SPEC_DRAFT_SPARSE128 ? (long long)SPEC_TOPK * 4
                                             : (long long)V * (ddt == SPEC_BF16 ? 2 : 4);
  a.nch_t = nchunks(V, tdt);
  a.nch_d = nchunks(V, ddt);
  a.nch_max = L.nch_max;
  a.rt_max = B * (max_k + 1);
  a.sparse = dk == SPEC_DRAFT_SPARSE128 || rule == SPEC_RULE_STRICT_TOP128;
  a.stream_draft = dk == SPEC_DRAFT_LOGITS && rule != SPEC_RULE_STRICT_TOP128;
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

  k_setup_linear<<<1, 1024, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (B == 0) return SPEC_OK;
  if (rule == SPEC_RULE_STRICT_TOP128) {
    const int rc = launch_topk128(draft, ddt, B * max_k, V, cu_draft, temperature, B,
                                  reinterpret_cast<int32_t *>(ws + L.tk_idx),
                                  reinterpret_cast<float *>(ws + L.tk_prob), a.hdr, st);
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
  rp.list = a.list;
  rp.hdr = a.hdr;
  rp.part = a.part;
  int rc = launch_row_pass(rp, st);
  if (rc != SPEC_OK) return rc;
  k_accept<<<(B + ACCEPT_WARPS - 1) / ACCEPT_WARPS, ACCEPT_WARPS * 32, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  const size_t wsum_bytes = sizeof(float) * 32 * ((V + SAMPLE_TILE - 1) / SAMPLE_TILE);
  void (*sampler)(LinearArgs) = a.sparse ? k_sample<SPEC_DRAFT_SPARSE128>
                                : dk == SPEC_DRAFT_PROBS ? k_sample<SPEC_DRAFT_PROBS>
                                                         : k_sample<SPEC_DRAFT_LOGITS>;
  if (wsum_bytes > 48 * 1024 &&
      cudaFuncSetAttribute(sampler, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)wsum_bytes) != cudaSuccess)
    return SPEC_ERR_CUDA;
  sampler<<<B, SAMPLE_THREADS, wsum_bytes, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}
