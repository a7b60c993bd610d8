// Cluster-resident linear verification: the position-lazy schedule with
// every needed row read from HBM once, and the final draws made from the
// copy already on chip.
//
// What it computes is the position-lazy linear verifier (nalar.dev
// "Penolakan memendekkan pekerjaan speculative": proposals after a rejected
// one are not read). Position j of request b needs target row p_{j+1} and,
// for a sampling request, draft row q_{j+1}; it is decided by the lossless
// coin ("Acceptance Is Not Speed", §6; "RheoSampling 2026", §4 step 1) or
// the greedy prefix match (nalar.dev "Semantik penerimaan"). A rejection
// ends the request with the inverse-CDF draw from norm(max(0, p - q))
// ("RheoSampling 2026", §4 step 3; from p itself when that has no mass), K
// acceptances with the bonus draw from p_{K+1}, a greedy request with the
// target argmax. Draws take the smallest id x with u*Z < C_x, C inclusive.
//
// How (GB300): a cluster of RC_CLUSTER CTAs verifies one request at a time
// with the rows of its current position resident in shared memory: CTA k
// holds slice k (1/8) of the position's target row and draft row (about
// 100 KB), so the residual draw after a rejection reads both rows from
// shared memory instead of HBM. Two CTAs share an SM, so each SM serves two
// requests, one copying its rows while the other decides.
//   - a position: lanes of warp 0 copy the CTA's two slices in RC_PIECES
//     TMA bulk copies each (completion on mbarriers); the CTA reduces them
//     to slice statistics (max, sum of 2^((z - m) c), lowest argmax) piece
//     by piece as they land, with packed bf16 maxima and one 2^x per element;
//   - the exchange: lane k of warp 0 stores the slice statistics into CTA
//     k's shared memory (DSMEM) and arrives on its barrier with release at
//     cluster scope; after the wait every thread merges the eight in rank
//     order and takes the decision, so all eight CTAs take the same decision
//     on the same bits;
//   - a residual draw: each CTA sums max(0, p - q) over its slices, the
//     eight totals are exchanged the same way, and the CTA whose slice holds
//     u*Z finds the token in its shared memory; a draw from p finds its
//     slice from the exchanged statistics alone.
// Requests come from a global counter; rank 0 takes the cluster's next one
// at the start of each request and sends it with its first statistics.
// Every wait is bounded (2 s of %globaltimer); on expiry the status word
// gets SPEC_ERR_TIMEOUT and the cluster stops.
#include <algorithm>
#include <mutex>
#include <utility>
#include <vector>
#include <climits>
#include <cstddef>

#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"
#include "linear.cuh"
#include "rowpass.cuh"

namespace sv {

namespace cg = cooperative_groups;

namespace {

constexpr int RC_CLUSTER = 8;                          // CTAs per cluster
constexpr int RC_WARPS = 8;
constexpr int RC_THREADS = 32 * RC_WARPS;              // one request (slot) per CTA
constexpr int RC_CTAS_PER_SM = 2;
constexpr int RC_PIECES = 4;                           // bulk copies per row slice
constexpr int RC_SLICE_MAX = 25600;                    // elements of a slice a CTA holds
constexpr int RC_MIN_V = 16384;                        // smaller rows: other schedules
constexpr size_t RC_DYN_SMEM = (size_t)2 * RC_SLICE_MAX * 2;   // target + draft slice, bf16

struct alignas(16) RcMsg {   // one CTA's slice statistics of a position (32 bytes), stored
                             // to peers as two 16-byte vectors: 16-byte aligned
  float tm, tS;       // target slice: max, sum of 2^((z - tm) c)
  int tidx;           // lowest index of the target slice's max
  float dm, dS;       // draft slice (sampling positions)
  int next;           // rank 0, first position: the slot's next request
  int pad[2];
};
static_assert(sizeof(RcMsg) == 32, "two 16-byte stores");

struct RcSmem {
  uint64_t full_t[RC_PIECES];             // target slice pieces landed
  uint64_t full_d[RC_PIECES];             // draft slice pieces landed
  uint64_t xch;                           // the 8 CTAs' statistics of a position
  uint64_t xch2;                          // the 8 CTAs' totals of a residual draw
  RcMsg msg[2][RC_CLUSTER];               // by exchange parity, then sender rank
  float tot[2][RC_CLUSTER];
  Part wt[RC_WARPS], wd[RC_WARPS];        // per-warp statistics
  float scan[RC_WARPS + 1];
  int xmin, xlast;
  int abort;
  int skip;
};
static_assert(offsetof(RcSmem, msg) % 16 == 0, "peer stores are 16-byte vectors");

// ------------------------------------------------------- cluster helpers
__device__ __forceinline__ uint32_t cluster_addr(const void *local, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Arrival on a peer's mbarrier; this thread's earlier stores to the cluster
// are visible to the peer once it has seen the phase complete.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for a phase completed by the cluster's arrivals.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t *bar, uint32_t parity,
                                                          volatile int *abort) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > WAIT_NS) return false;
  }
}

// Exclusive prefix of one float per thread over the CTA (warp scans, then
// the warps' totals in warp order); *total gets the CTA total.
__device__ __forceinline__ float cta_excl_scan(float v, float *scratch, int warp, int lane,
                                               float *total) {
  float x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  float xe = __shfl_up_sync(0xffffffffu, x, 1);
  if (lane == 0) xe = 0.f;
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  float off = 0.f, t = 0.f;
  for (int k = 0; k < RC_WARPS; ++k) {
    if (k == warp) off = t;
    t += scratch[k];
  }
  *total = t;
  __syncthreads();
  return off + xe;
}

// --------------------------------------------------------------- kernel
struct RcArgs {
  LinearArgs a;
  int slice;      // elements per CTA slice (a multiple of 8)
  int nbuf;       // one cluster per request: row-slice buffers per CTA
};

// The CTA's slice of a row: elements [e0, e0 + nel), as nvec 16-byte
// vectors; piece p holds vectors [piece_v0(p), piece_v0(p + 1)).
__device__ __forceinline__ int piece_v0(int nvec, int p) {
  return (int)((long long)nvec * p / RC_PIECES);
}

// Piece p of one slice into `buf`, completion on bar (one lane per piece).
__device__ __forceinline__ void load_piece(unsigned char *buf, const char *row, int e0, int nvec,
                                           int p, uint64_t *bar) {
  const int v0 = piece_v0(nvec, p), v1 = piece_v0(nvec, p + 1);
  const uint32_t nb = (uint32_t)(v1 - v0) * 16u;
  if (nb > 0) {
    mbar_arrive_tx(bar, nb);
    bulk_g2s(buf + 16LL * v0, row + 2LL * e0 + 16LL * v0, nb, bar);
  } else {
    mbar_arrive(bar);
  }
}

// Running statistics over this thread's vectors v0, v0 + RC_THREADS, ...
// below v1 of a bf16 slice (element index e0 + 8 v): four vectors at a time,
// their packed maximum checked once, one 2^x per element.
template <bool SOFTMAX>
__device__ __forceinline__ void consume_vectors(const unsigned char *buf, int v0, int v1, int e0,
                                                float c, RunState &st) {
  constexpr uint32_t NINF2 = 0xff80ff80u;   // (-inf, -inf)
  for (int v = v0; v < v1; v += 4 * RC_THREADS) {
    uint4 w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      w[k] = v + k * RC_THREADS < v1 ? lds128(buf + 16 * (v + k * RC_THREADS))
                                     : make_uint4(NINF2, NINF2, NINF2, NINF2);
    uint32_t m2 = bmax2(bmax2(w[0].x, w[0].y), bmax2(w[0].z, w[0].w));
#pragma unroll
    for (int k = 1; k < 4; ++k)
      m2 = bmax2(m2, bmax2(bmax2(w[k].x, w[k].y), bmax2(w[k].z, w[k].w)));
    const float vm = fmaxf(bf16lo(m2), bf16hi(m2));
    if (vm > st.m) {   // the lowest index holding vm (vectors in index order)
      int idx = INT_MAX;
#pragma unroll
      for (int k = 3; k >= 0; --k) {
        const uint32_t u4[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
        for (int q = 3; q >= 0; --q) {
          const int e = e0 + 8 * (v + k * RC_THREADS) + 2 * q;
          if (bf16hi(u4[q]) == vm) idx = e + 1;
          if (bf16lo(u4[q]) == vm) idx = e;
        }
      }
      if (SOFTMAX) {
        const float f = ex2((st.m - vm) * c);
        st.S2 = mul2(st.S2, pk2(f, f));
      }
      st.m = vm;
      st.idx = idx;
    }
    if (SOFTMAX) {
      const f32x2 c2 = pk2(c, c);
      f32x2 acc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t u4[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
        f32x2 s = pk2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const f32x2 t = mul2(bsub2(u4[q], st.m), c2);
          s = add2(s, pk2(ex2(lo2(t)), ex2(hi2(t))));
        }
        acc[k] = s;
      }
      st.S2 = add2(st.S2, add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])));
    }
  }
}

// p(x) or max(0, p(x) - q(x)) for the 8 elements of slice vector v.
__device__ __forceinline__ void slice_weights(const unsigned char *tb, const unsigned char *db,
                                              int v, float c, float mt, float invSt, float md,
                                              float invSd, float (&w)[8]) {
  const uint4 t4 = lds128(tb + 16 * v);
  const uint32_t tw[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    w[2 * q] = ex2((bf16lo(tw[q]) - mt) * c) * invSt;
    w[2 * q + 1] = ex2((bf16hi(tw[q]) - mt) * c) * invSt;
  }
  if (db != nullptr) {
    const uint4 d4 = lds128(db + 16 * v);
    const uint32_t dw[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      w[2 * q] = fmaxf(0.f, w[2 * q] - ex2((bf16lo(dw[q]) - md) * c) * invSd);
      w[2 * q + 1] = fmaxf(0.f, w[2 * q + 1] - ex2((bf16hi(dw[q]) - md) * c) * invSd);
    }
  }
}

// The CTA's share of a draw in its slice: weights of p (db null) or of
// max(0, p - q) over contiguous runs of vectors per thread. With `search`,
// the smallest element x with carry + C(x) > target (C the inclusive prefix
// over the slice), else the slice's last element of positive weight, -1 if
// none; without, -1 and only the slice total in *total. Every thread returns
// the same values.
template <class Smem>
__device__ int slice_draw(Smem &sh, int warp, int lane, const unsigned char *tb,
                          const unsigned char *db, int e0, int nvec, float c, float mt,
                          float invSt, float md, float invSd, bool search, float carry,
                          float target, float *total) {
  const int seg = (nvec + RC_THREADS - 1) / RC_THREADS;
  const int v0 = min(nvec, (int)threadIdx.x * seg), v1 = min(nvec, v0 + seg);
  float s = 0.f;
  for (int v = v0; v < v1; ++v) {
    float w[8];
    slice_weights(tb, db, v, c, mt, invSt, md, invSd, w);
#pragma unroll
    for (int k = 0; k < 8; ++k) s += w[k];
  }
  const float excl = cta_excl_scan(s, sh.scan, warp, lane, total);
  if (!search) return -1;
  if (threadIdx.x == 0) {
    sh.xmin = INT_MAX;
    sh.xlast = -1;
  }
  __syncthreads();
  float pre = 0.f;
  int cand = INT_MAX, last = -1;
  for (int v = v0; v < v1 && cand == INT_MAX; ++v) {
    float w[8];
    slice_weights(tb, db, v, c, mt, invSt, md, invSd, w);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      pre += w[k];
      if (cand == INT_MAX && carry + (excl + pre) > target) cand = e0 + 8 * v + k;
      if (w[k] > 0.f) last = e0 + 8 * v + k;
    }
  }
  if (cand != INT_MAX) atomicMin(&sh.xmin, cand);
  if (last >= 0) atomicMax(&sh.xlast, last);
  __syncthreads();
  const int x = sh.xmin != INT_MAX ? sh.xmin : sh.xlast;
  __syncthreads();
  return x;
}

__global__ void __cluster_dims__(RC_CLUSTER, 1, 1) __launch_bounds__(RC_THREADS, RC_CTAS_PER_SM)
    k_verify_resident(const RcArgs ra) {
  extern __shared__ __align__(128) unsigned char dsmem[];
  __shared__ RcSmem sh;
  const LinearArgs &a = ra.a;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int cid = (int)(blockIdx.x / RC_CLUSTER), ncl = (int)(gridDim.x / RC_CLUSTER);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int p = 0; p < RC_PIECES; ++p) {
      mbar_init(&sh.full_t[p], 1);
      mbar_init(&sh.full_d[p], 1);
    }
    mbar_init(&sh.xch, RC_CLUSTER);
    mbar_init(&sh.xch2, RC_CLUSTER);
    sh.abort = 0;
    sh.skip = *(volatile int *)&a.hdr->setup_bad;
    fence_mbar_init();
  }
  cluster.sync();   // barriers initialised everywhere before any remote arrival
  if (sh.skip) {    // inputs rejected by the setup: nothing is verified
    const int W = a.max_k + 1;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < (long long)a.B * W;
         i += (long long)gridDim.x * blockDim.x) {
      GST(a.out_tokens + (i), -1);
      if (i < a.B) GST(a.out_accepted + (i), -1);
    }
    cluster.sync();
    return;
  }

  const int V = a.V;
  const int e0 = min(V, rank * ra.slice);
  const int nel = min(V, e0 + ra.slice) - e0;
  const int nvec = nel / 8;
  unsigned char *tb = dsmem;
  unsigned char *db = dsmem + (size_t)RC_SLICE_MAX * 2;
  volatile int *abort = &sh.abort;
  const int W = a.max_k + 1;
  const uint64_t seed = seed_of(a);
  unsigned pos_ct = 0, dpos_ct = 0, xch_ct = 0, xch2_ct = 0;   // phases used so far
  bool failed = false;

  int b = cid;   // the first request of this cluster; then the leader's picks
  ReqInfo r{};
  if (b < a.B) r = GLD(a.req + (b));
  while (b < a.B && !failed) {
    const bool sample = r.mode == MODE_SAMPLE;
    const float c = r.c;
    const char *trow0 = a.target + (long long)r.t0 * a.t_row_bytes;
    const char *drow0 = a.draft + (long long)r.d0 * a.d_row_bytes;
    int n = r.K, par = 0, next = a.B;
    ReqInfo rn{};
    RowStat ts{NO_MAX, 0.f, INT_MAX}, ds{NO_MAX, 0.f, INT_MAX};
    for (int j = 0;; ++j) {
      const bool need_d = sample && j < r.K;
      // 1. the CTA's slices of position j's rows (lane p of warp 0 copies
      // target piece p, lane RC_PIECES + p draft piece p), and the decision
      // inputs, needed after the exchange
      if (warp == 0 && lane < RC_PIECES)
        load_piece(tb, trow0 + (long long)j * a.t_row_bytes, e0, nvec, lane, &sh.full_t[lane]);
      if (need_d && warp == 0 && lane >= RC_PIECES && lane < 2 * RC_PIECES)
        load_piece(db, drow0 + (long long)j * a.d_row_bytes, e0, nvec, lane - RC_PIECES,
                   &sh.full_d[lane - RC_PIECES]);
      int d = -1, nxt = -1;
      float zt = 0.f, zd = 0.f;
      if (j < r.K) {
        d = GLDG(a.tokens + r.d0 + j);
        zt = GLDCG(a.rank_thr + r.t0 + j);
        if (need_d) zd = GLDCG(a.zd_at + r.d0 + j);
      }
      if (threadIdx.x == 0 && j == 0 && rank == 0)
        nxt = ncl + (int)atomicAdd(&a.hdr->work, 1u);
      // 2. slice statistics, piece by piece as they land
      RunState st{NO_MAX, pk2(0.f, 0.f), INT_MAX, 0, 0u};
      RunState sd{NO_MAX, pk2(0.f, 0.f), INT_MAX, 0, 0u};
      for (int p = 0; p < RC_PIECES && !failed; ++p) {
        if (!mbar_wait_bounded(&sh.full_t[p], pos_ct & 1u, abort) ||
            (need_d && !mbar_wait_bounded(&sh.full_d[p], dpos_ct & 1u, abort))) {
          *abort = 1;
          failed = true;
          break;
        }
        const int v0 = piece_v0(nvec, p) + (int)threadIdx.x, v1 = piece_v0(nvec, p + 1);
        if (sample) {
          consume_vectors<true>(tb, v0, v1, e0, c, st);
          if (need_d) consume_vectors<true>(db, v0, v1, e0, c, sd);
        } else {
          consume_vectors<false>(tb, v0, v1, e0, c, st);
        }
      }
      ++pos_ct;
      if (need_d) ++dpos_ct;
      const Part pt = finish_row_chunk<false>(st, c);
      const Part pd = finish_row_chunk<false>(sd, c);
      if (lane == 0) {
        sh.wt[warp] = pt;
        sh.wd[warp] = pd;
      }
      failed = __syncthreads_or(failed);
      if (failed) break;
      // 3. exchange: lane k of warp 0 sends this CTA's slice statistics to
      // rank k (every lane merges the warps' statistics in warp order)
      par = (int)(xch_ct & 1u);
      if (warp == 0) {
        float tm = NO_MAX, tS = 0.f, dm = NO_MAX, dS = 0.f;
        int ti = INT_MAX, di = INT_MAX;
        for (int k = 0; k < RC_WARPS; ++k) {
          merge_stat(tm, tS, ti, sh.wt[k].m, sh.wt[k].S, sh.wt[k].idx, c);
          merge_stat(dm, dS, di, sh.wd[k].m, sh.wd[k].S, sh.wd[k].idx, c);
        }
        const int nx = __shfl_sync(0xffffffffu, nxt, 0);
        if (lane < RC_CLUSTER) {
          const uint32_t m = cluster_addr(&sh.msg[par][rank], lane);
          st_cluster_v4(m, make_uint4(__float_as_uint(tm), __float_as_uint(tS), (unsigned)ti,
                                      __float_as_uint(dm)));
          st_cluster_v4(m + 16, make_uint4(__float_as_uint(dS), (unsigned)nx, 0u, 0u));
          mbar_arrive_cluster(cluster_addr(&sh.xch, lane));
        }
      }
      failed = !mbar_wait_cluster_bounded(&sh.xch, xch_ct & 1u, abort);
      ++xch_ct;
      failed = __syncthreads_or(failed);
      if (failed) break;
      // 4. the row statistics (rank order: the same bits in every CTA) and
      // the decision, taken by every thread on the same values
      ts = RowStat{NO_MAX, 0.f, INT_MAX};
      ds = RowStat{NO_MAX, 0.f, INT_MAX};
      for (int k = 0; k < RC_CLUSTER; ++k) {
        const RcMsg &mk = sh.msg[par][k];
        merge_stat(ts.m, ts.S, ts.idx, mk.tm, mk.tS, mk.tidx, c);
        if (need_d) merge_stat(ds.m, ds.S, ds.idx, mk.dm, mk.dS, INT_MAX, c);
      }
      if (j == 0) {
        next = sh.msg[par][0].next;
        if (next < a.B) rn = GLD(a.req + (next));   // early: used after this request
      }
      if (j == r.K) {
        n = j;
        break;
      }
      const bool dok = (unsigned)d < (unsigned)V;
      float pdv, qdv;
      bool rej;
      if (!sample) {
        rej = !(dok && d == ts.idx);
        pdv = rej ? 0.f : 1.f;
        qdv = -1.f;
      } else if (dok && !row_empty(ts.m)) {
        pdv = ex2((zt - ts.m) * c) / ts.S;
        qdv = row_empty(ds.m) ? 0.f : ex2((zd - ds.m) * c) / ds.S;
        const float acc = qdv <= pdv ? 1.f : pdv / qdv;
        rej = !(uniform24(seed, (uint32_t)b, (uint32_t)(j + 1), 0) < acc);
      } else {
        pdv = qdv = 0.f;
        rej = true;
      }
      if (rank == 0 && threadIdx.x == 0) {
        if (!dok || row_empty(ts.m)) set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);
        if (a.out_pq) {
          GST(a.out_pq + (2LL * (r.d0 + j)), pdv);
          GST(a.out_pq + (2LL * (r.d0 + j) + 1), qdv);
        }
      }
      if (rej) {
        n = j;
        break;
      }
    }
    if (failed) break;
    // 5. commit: the accepted drafts, -1 after the final slot; positions
    // after n + 1 are not reported
    if (rank == 0) {
      int32_t *out = a.out_tokens + (long long)b * W;
      for (int jj = threadIdx.x; jj < W; jj += RC_THREADS)
        if (jj != n) GST(out + jj, jj < n ? GLD(a.tokens + (r.d0 + jj)) : -1);
      if (a.out_pq)
        for (int i = n + 1 + threadIdx.x; i < r.K; i += RC_THREADS) {
          GST(a.out_pq + (2LL * (r.d0 + i)), __int_as_float(0x7fc00000));
          GST(a.out_pq + (2LL * (r.d0 + i) + 1), __int_as_float(0x7fc00000));
        }
      if (threadIdx.x == 0) {
        GST(a.out_accepted + (b), n);
        if (!sample) GST(out + n, ts.idx);   // greedy: the target's argmax
      }
    }
    // 6. the final draw (sampling requests) from position n's slices, which
    // are still in shared memory
    if (sample) {
      const float invSt = 1.f / ts.S;
      int owner = -1, x = -1;
      float carry = 0.f, target = 0.f;
      bool from_p = true;
      const float u = uniform24(seed, (uint32_t)b, (uint32_t)(n + 1), n < r.K ? 1u : 2u);
      if (n < r.K) {
        // residual: slice totals of max(0, p - q), exchanged
        const float invSd = ds.S > 0.f ? 1.f / ds.S : 0.f;
        float R;
        slice_draw(sh, warp, lane, tb, db, e0, nvec, c, ts.m, invSt, ds.m, invSd, false, 0.f,
                   0.f, &R);
        const int p2 = (int)(xch2_ct & 1u);
        if (warp == 0 && lane < RC_CLUSTER) {
          st_cluster_f32(cluster_addr(&sh.tot[p2][rank], lane), R);
          mbar_arrive_cluster(cluster_addr(&sh.xch2, lane));
        }
        failed = !mbar_wait_cluster_bounded(&sh.xch2, xch2_ct & 1u, abort);
        ++xch2_ct;
        failed = __syncthreads_or(failed);
        if (failed) break;
        float Z = 0.f;
        int klast = -1;
        for (int k = 0; k < RC_CLUSTER; ++k) {
          Z += sh.tot[p2][k];
          if (sh.tot[p2][k] > 0.f) klast = k;
        }
        if (Z > 0.f) {
          target = u * Z;
          for (int k = 0; k < RC_CLUSTER; ++k) {
            const float nc = carry + sh.tot[p2][k];
            if (nc > target) {
              owner = k;
              break;
            }
            carry = nc;
          }
          if (owner < 0) owner = klast;
          from_p = false;
          if (owner == rank) {   // its slice total is positive: x >= 0
            float dummy;
            x = slice_draw(sh, warp, lane, tb, db, e0, nvec, c, ts.m, invSt, ds.m, invSd, true,
                           carry, target, &dummy);
          }
        }
      }
      if (from_p) {
        // a draw from p (bonus, or a residual without mass): the slice
        // masses from the exchanged statistics, then the owner's slice
        float Zp = 0.f, mk[RC_CLUSTER];
        int klast = -1;
        for (int k = 0; k < RC_CLUSTER; ++k) {
          const RcMsg &m = sh.msg[par][k];
          mk[k] = m.tS > 0.f ? m.tS * ex2((m.tm - ts.m) * c) * invSt : 0.f;
          Zp += mk[k];
          if (mk[k] > 0.f) klast = k;
        }
        target = u * Zp;
        for (int k = 0; k < RC_CLUSTER && Zp > 0.f; ++k) {
          const float nc = carry + mk[k];
          if (nc > target) {
            owner = k;
            break;
          }
          carry = nc;
        }
        if (owner < 0) owner = klast;
        if (owner == rank) {
          float dummy;
          x = slice_draw(sh, warp, lane, tb, nullptr, e0, nvec, c, ts.m, invSt, 0.f, 0.f, true,
                         carry, target, &dummy);
        }
        if (owner < 0) owner = 0;   // no mass anywhere: rank 0 reports it
      }
      if (owner == rank && threadIdx.x == 0) {
        if (x < 0) set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);   // a row without mass
        GST(a.out_tokens + ((long long)b * W + n), x);
      }
    }
    __syncthreads();   // the slices are free for the next request's copies
    b = next;
    r = rn;
  }
  if (failed && threadIdx.x == 0) set_status(a.hdr, SPEC_ERR_TIMEOUT, -6);
  cluster.sync();   // no CTA leaves while a peer may still write to it
}

// ------------------------------------------- small calls: whole requests
// Small calls with rows longer than the fused kernel takes (dense bf16
// logits, V % 8 == 0, at most RQ_MAX_K drafts, at most RQ_MAX_B requests):
// one launch, a cluster per request. Every CTA first validates the whole
// call. The request's rows (target rows 1..K+1, then draft rows 1..K) pass
// through a few row-slice buffers per CTA, as many rows at a time as there
// are buffers: lane i of warp 0 copies the CTA's slice of a row into buffer
// i, and one warp reduces each buffer. One exchange carries every
// position's slice statistics; every CTA then decides all positions on the
// same merged bits. The final draw copies the two rows it needs again (they
// are still in L2) and finds the token with one more exchange. Two
// exchanges per request, however many drafts it has; with few buffers
// (48 KB for V = 32000) four CTAs share an SM, so a call of up to about 76
// requests has all its clusters at once.
constexpr int RQ_MAX_K = 8;
constexpr int RQ_ROWS = 2 * RQ_MAX_K + 1;
// Row-slice buffers per CTA: as many slices as fit this many bytes (at least
// two, for the final draw's row pair), so that short rows run four CTAs per
// SM and every request of a call up to RQ_MAX_B has its cluster at once.
constexpr size_t RQ_BUF_BYTES = 48 * 1024;
constexpr int RQ_CTAS_PER_SM = 4;
// A cluster takes one request at a time, so the call's time grows with the
// rounds of requests per cluster: above this many requests the streaming
// and eager schedules, which spread every row over the whole GPU, are faster.
constexpr int RQ_MAX_B = 128;

struct RqSmem {
  uint64_t bar[RQ_ROWS];                  // row-slice buffer filled
  uint64_t xch, xch2;
  RcMsg msg[2][RC_CLUSTER][RQ_MAX_K + 1];  // by parity, sender, position
  float tot[2][RC_CLUSTER];
  Part rows[RQ_ROWS];                     // this CTA's slice statistics per row
  RowStat ts[RQ_MAX_K + 1], ds[RQ_MAX_K + 1];   // merged, per position
  int d[RQ_MAX_K];
  float zt[RQ_MAX_K], zd[RQ_MAX_K];
  float scan[RC_WARPS + 1];
  int xmin, xlast;
  int n, next;
  int abort;
};
static_assert(offsetof(RqSmem, msg) % 16 == 0, "peer stores are 16-byte vectors");

// Running statistics of one warp over vectors lane, lane + 32, ... of a
// bf16 slice (element index e0 + 8 v).
template <bool SOFTMAX>
__device__ __forceinline__ void warp_consume(const unsigned char *buf, int nvec, int lane, int e0,
                                             float c, RunState &st) {
  for (int v = lane; v < nvec; v += 32)
    consume_vec<SOFTMAX, true>(lds128(buf + 16 * v), e0 + 8 * v, c, st, INFINITY);
}

__global__ void __cluster_dims__(RC_CLUSTER, 1, 1) __launch_bounds__(RC_THREADS, RQ_CTAS_PER_SM)
    k_verify_cluster_small(const RcArgs ra) {
  extern __shared__ __align__(128) unsigned char dsmem[];
  __shared__ RqSmem sh;
  const LinearArgs &a = ra.a;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int cid = (int)(blockIdx.x / RC_CLUSTER), ncl = (int)(gridDim.x / RC_CLUSTER);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < RQ_ROWS; ++i) mbar_init(&sh.bar[i], 1);
    mbar_init(&sh.xch, RC_CLUSTER);
    mbar_init(&sh.xch2, RC_CLUSTER);
    sh.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();   // this CTA's barriers are ready for its own copies
  const int V = a.V, W = a.max_k + 1;
  const int e0 = min(V, rank * ra.slice);
  const int nvec = (min(V, e0 + ra.slice) - e0) / 8;
  const size_t rbytes = (size_t)ra.slice * 2;   // row stride in shared memory
  volatile int *abort = &sh.abort;
  const uint64_t seed = seed_of(a);
  // phase parities of each buffer's barrier, one bit per buffer: uses issued
  // and uses completed (a buffer has at most one copy in flight; every thread
  // keeps the same bits)
  unsigned par_issued = 0, par_done = 0;
  const int nb = ra.nbuf;
  unsigned xch_ct = 0, xch2_ct = 0;
  bool failed = false;
  // row i of request rq (target rows 0..K, then draft rows) into buffer q
  auto issue_row = [&](const ReqInfo &rq, int i, int q) {
    const bool tgt = i <= rq.K;
    const char *row = tgt ? a.target + (long long)(rq.t0 + i) * a.t_row_bytes
                          : a.draft + (long long)(rq.d0 + i - rq.K - 1) * a.d_row_bytes;
    const uint32_t nbytes = (uint32_t)nvec * 16u;
    if (nbytes > 0) {
      // the buffer was read by this CTA's threads before the last barrier
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_tx(&sh.bar[q], nbytes);
      bulk_g2s(dsmem + q * rbytes, row + 2LL * e0, nbytes, &sh.bar[q]);
    } else {
      mbar_arrive(&sh.bar[q]);
    }
  };
  auto rows_of = [](const ReqInfo &rq) {
    return rq.K + 1 + (rq.mode == MODE_SAMPLE ? rq.K : 0);
  };

  // The cluster's first request: when its record is valid (its rows are then
  // in bounds), its first rows are copied while the call is validated.
  int b = cid;
  ReqInfo r{};
  const bool pre = b < a.B && load_request(a, b, r);
  unsigned pre_used = 0;
  if (pre) {
    const int cnt = min(nb, rows_of(r));
    if (warp == 0 && lane < cnt) issue_row(r, lane, lane);
    pre_used = (1u << cnt) - 1u;
    par_issued ^= pre_used;
  }
  // Every CTA validates the whole call (B <= RQ_MAX_B requests: one record
  // and up to RQ_MAX_K tokens per thread), so every CTA reaches the same
  // verdict without a grid-wide barrier: with any request invalid, none is
  // verified.
  bool bad = false;
  for (int bb = threadIdx.x; bb < a.B; bb += RC_THREADS) {
    ReqInfo rq;
    if (!load_request(a, bb, rq)) {
      bad = true;
      continue;
    }
    for (int j = 0; j < rq.K; ++j)
      if ((unsigned)GLD(a.tokens + rq.d0 + j) >= (unsigned)a.V) {
        set_status(a.hdr, SPEC_ERR_INVALID_ARG, bb);
        bad = true;
      }
  }
  bad = __syncthreads_or(bad);
  cluster.sync();   // barriers initialised everywhere before any remote arrival
  if (bad) {
    // the first rows' copies in flight, waited for (bounded) before leaving
    volatile int never = 0;
    for (int q = 0; q < nb; ++q)
      if ((pre_used >> q) & 1u) mbar_wait_bounded(&sh.bar[q], 0u, &never);
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < (long long)a.B * W;
         i += (long long)gridDim.x * blockDim.x) {
      GST(a.out_tokens + i, -1);
      if (i < a.B) GST(a.out_accepted + i, -1);
    }
    cluster.sync();
    return;
  }

  bool first = pre;   // this request's first rows are already on their way
  while (b < a.B && !failed) {
    if (!first) load_request(a, b, r);   // valid: checked above
    const bool sample = r.mode == MODE_SAMPLE;
    const float c = r.c;
    const int K = r.K;
    const int nrows = rows_of(r);
    // 1. the decision inputs (the drafts and both logits at each draft); the
    // cluster's next request (rank 0)
    if (threadIdx.x < K) {
      const int j = threadIdx.x;
      const int d = GLD(a.tokens + r.d0 + j);
      sh.d[j] = d;
      sh.zt[j] = load_elem(a.target + (long long)(r.t0 + j) * a.t_row_bytes, a.tdt, d);
      sh.zd[j] = sample ? load_elem(a.draft + (long long)(r.d0 + j) * a.d_row_bytes, a.ddt, d)
                        : 0.f;
    }
    int nxt = -1;
    if (threadIdx.x == 0 && rank == 0) nxt = ncl + (int)atomicAdd(&a.hdr->work, 1u);
    // 2. slice statistics of every row: the rows pass through the nb
    // buffers, nb at a time (one bulk copy each), one warp per row
    for (int i0 = 0; i0 < nrows && !failed; i0 += nb) {
      const int cnt = min(nb, nrows - i0);
      const unsigned used = (1u << cnt) - 1u;
      if (first) {
        first = false;   // issued before the validation
      } else {
        if (warp == 0 && lane < cnt) issue_row(r, i0 + lane, lane);
        par_issued ^= used;
      }
      for (int q = warp; q < cnt; q += RC_WARPS) {
        if (!mbar_wait_bounded(&sh.bar[q], (par_done >> q) & 1u, abort)) {
          *abort = 1;
          failed = true;
          break;
        }
        RunState st{NO_MAX, pk2(0.f, 0.f), INT_MAX, 0, 0u};
        if (c != 0.f) warp_consume<true>(dsmem + q * rbytes, nvec, lane, e0, c, st);
        else warp_consume<false>(dsmem + q * rbytes, nvec, lane, e0, c, st);
        const Part p = finish_row_chunk<false>(st, c);
        if (lane == 0) sh.rows[i0 + q] = p;
      }
      failed = __syncthreads_or(failed);   // every buffer read before it is refilled
      if (!failed) par_done ^= used;
    }
    if (failed) break;
    // 3. one exchange: lane k of warp 0 sends every position's slice
    // statistics to rank k
    const int par = (int)(xch_ct & 1u);
    if (warp == 0) {
      const int nx = __shfl_sync(0xffffffffu, nxt, 0);
      if (lane < RC_CLUSTER) {
        for (int p = 0; p <= K; ++p) {
          const Part t = sh.rows[p];
          const Part d = sample && p < K ? sh.rows[K + 1 + p] : Part{NO_MAX, 0.f, INT_MAX, 0};
          const uint32_t m = cluster_addr(&sh.msg[par][rank][p], lane);
          st_cluster_v4(m, make_uint4(__float_as_uint(t.m), __float_as_uint(t.S), (unsigned)t.idx,
                                      __float_as_uint(d.m)));
          st_cluster_v4(m + 16, make_uint4(__float_as_uint(d.S), (unsigned)nx, 0u, 0u));
        }
        mbar_arrive_cluster(cluster_addr(&sh.xch, lane));
      }
    }
    failed = !mbar_wait_cluster_bounded(&sh.xch, xch_ct & 1u, abort);
    ++xch_ct;
    failed = __syncthreads_or(failed);
    if (failed) break;
    // 4. merged statistics per position (rank order: the same bits in every
    // CTA), then the decisions in order; p(d), q(d) for every position
    if ((int)threadIdx.x <= K) {
      const int p = threadIdx.x;
      RowStat ts{NO_MAX, 0.f, INT_MAX}, ds{NO_MAX, 0.f, INT_MAX};
      for (int k = 0; k < RC_CLUSTER; ++k) {
        const RcMsg &m = sh.msg[par][k][p];
        merge_stat(ts.m, ts.S, ts.idx, m.tm, m.tS, m.tidx, c);
        if (sample && p < K) merge_stat(ds.m, ds.S, ds.idx, m.dm, m.dS, INT_MAX, c);
      }
      sh.ts[p] = ts;
      sh.ds[p] = ds;
    }
    __syncthreads();
    if (warp == 0) {   // position j on lane j (K <= RQ_MAX_K < 32); the first rejection ends it
      bool rej = false;
      if (lane < K) {
        const int j = lane;
        const int d = sh.d[j];
        const RowStat ts = sh.ts[j], ds = sh.ds[j];
        const bool dok = (unsigned)d < (unsigned)V;
        float pdv, qdv;
        if (!sample) {
          rej = !(dok && d == ts.idx);
          pdv = rej ? 0.f : 1.f;
          qdv = -1.f;
        } else if (dok && !row_empty(ts.m)) {
          pdv = ex2((sh.zt[j] - ts.m) * c) / ts.S;
          qdv = row_empty(ds.m) ? 0.f : ex2((sh.zd[j] - ds.m) * c) / ds.S;
          const float acc = qdv <= pdv ? 1.f : pdv / qdv;
          rej = !(uniform24(seed, (uint32_t)b, (uint32_t)(j + 1), 0) < acc);
        } else {
          pdv = qdv = 0.f;
          rej = true;
        }
        if (rank == 0) {
          if (!dok || row_empty(ts.m)) set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);
          if (a.out_pq) {
            GST(a.out_pq + 2LL * (r.d0 + j), pdv);
            GST(a.out_pq + 2LL * (r.d0 + j) + 1, qdv);
          }
        }
      }
      const unsigned rm = __ballot_sync(0xffffffffu, rej);
      if (lane == 0) {
        if (rank == 0 && row_empty(sh.ts[K].m)) set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);
        sh.n = rm ? __ffs(rm) - 1 : K;
        sh.next = sh.msg[par][0][0].next;
      }
    }
    __syncthreads();
    const int n = sh.n, next = sh.next;
    // 5. commit: the accepted drafts, then -1 after the final slot
    if (rank == 0) {
      int32_t *out = a.out_tokens + (long long)b * W;
      for (int jj = threadIdx.x; jj < W; jj += RC_THREADS)
        if (jj != n) GST(out + jj, jj < n ? sh.d[jj] : -1);
      if (threadIdx.x == 0) {
        GST(a.out_accepted + b, n);
        if (!sample) GST(out + n, sh.ts[n].idx);   // greedy: the target's argmax
      }
    }
    // 6. the final draw from position n's rows, copied again (from L2) into
    // buffers 0 and 1
    if (sample) {
      const int nfin = n < K ? 2 : 1;
      const unsigned used = (1u << nfin) - 1u;
      if (warp == 0 && lane < nfin) issue_row(r, lane == 0 ? n : K + 1 + n, lane);
      par_issued ^= used;
      for (int q = 0; q < nfin && !failed; ++q)
        failed = !mbar_wait_bounded(&sh.bar[q], (par_done >> q) & 1u, abort);
      failed = __syncthreads_or(failed);
      if (failed) break;
      par_done ^= used;
      const RowStat ts = sh.ts[n], ds = sh.ds[n];
      const unsigned char *tb = dsmem;
      const unsigned char *db = dsmem + rbytes;
      const float invSt = 1.f / ts.S;
      int owner = -1, x = -1;
      float carry = 0.f, target = 0.f;
      bool from_p = true;
      const float u = uniform24(seed, (uint32_t)b, (uint32_t)(n + 1), n < K ? 1u : 2u);
      if (n < K) {
        const float invSd = ds.S > 0.f ? 1.f / ds.S : 0.f;
        float R;
        slice_draw(sh, warp, lane, tb, db, e0, nvec, c, ts.m, invSt, ds.m, invSd, false, 0.f,
                      0.f, &R);
        const int p2 = (int)(xch2_ct & 1u);
        if (warp == 0 && lane < RC_CLUSTER) {
          st_cluster_f32(cluster_addr(&sh.tot[p2][rank], lane), R);
          mbar_arrive_cluster(cluster_addr(&sh.xch2, lane));
        }
        failed = !mbar_wait_cluster_bounded(&sh.xch2, xch2_ct & 1u, abort);
        ++xch2_ct;
        failed = __syncthreads_or(failed);
        if (failed) break;
        float Z = 0.f;
        int klast = -1;
        for (int k = 0; k < RC_CLUSTER; ++k) {
          Z += sh.tot[p2][k];
          if (sh.tot[p2][k] > 0.f) klast = k;
        }
        if (Z > 0.f) {
          target = u * Z;
          for (int k = 0; k < RC_CLUSTER; ++k) {
            const float nc = carry + sh.tot[p2][k];
            if (nc > target) {
              owner = k;
              break;
            }
            carry = nc;
          }
          if (owner < 0) owner = klast;
          from_p = false;
          if (owner == rank) {   // its slice total is positive: x >= 0
            float dummy;
            x = slice_draw(sh, warp, lane, tb, db, e0, nvec, c, ts.m, invSt, ds.m, invSd,
                              true, carry, target, &dummy);
          }
        }
      }
      if (from_p) {   // bonus, or a residual without mass: p by slice masses
        float Zp = 0.f, mk[RC_CLUSTER];
        int klast = -1;
        for (int k = 0; k < RC_CLUSTER; ++k) {
          const RcMsg &m = sh.msg[par][k][n];
          mk[k] = m.tS > 0.f ? m.tS * ex2((m.tm - ts.m) * c) * invSt : 0.f;
          Zp += mk[k];
          if (mk[k] > 0.f) klast = k;
        }
        target = u * Zp;
        for (int k = 0; k < RC_CLUSTER && Zp > 0.f; ++k) {
          const float nc = carry + mk[k];
          if (nc > target) {
            owner = k;
            break;
          }
          carry = nc;
        }
        if (owner < 0) owner = klast;
        if (owner == rank) {
          float dummy;
          x = slice_draw(sh, warp, lane, tb, nullptr, e0, nvec, c, ts.m, invSt, 0.f, 0.f, true,
                            carry, target, &dummy);
        }
        if (owner < 0) owner = 0;   // no mass anywhere: rank 0 reports it
      }
      if (owner == rank && threadIdx.x == 0) {
        if (x < 0) set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);   // a row without mass
        GST(a.out_tokens + (long long)b * W + n, x);
      }
    }
    __syncthreads();   // the buffers are free for the next request's copies
    b = next;
  }
  if (failed) {
    if (threadIdx.x == 0) set_status(a.hdr, SPEC_ERR_TIMEOUT, -7);
    // this CTA's copies still in flight: wait for them (bounded) before leaving
    volatile int never = 0;
    for (int q = 0; q < nb; ++q)
      if (((par_done ^ par_issued) >> q) & 1u) mbar_wait_bounded(&sh.bar[q], (par_done >> q) & 1u, &never);
  }
  cluster.sync();   // no CTA leaves while a peer may still write to it
}

}  // namespace

bool cluster_small_supported(const LinearArgs &a, const spec_linear_ext *ext,
                             size_t limit_bytes) {
  if (limit_bytes == 0 || a.B > RQ_MAX_B) return false;
  if (ext != nullptr && (ext->flags != 0 || ext->out_kl != nullptr || ext->out_rank != nullptr))
    return false;
  if ((a.rule != SPEC_RULE_STRICT && a.rule != SPEC_RULE_GREEDY) || a.dk != SPEC_DRAFT_LOGITS ||
      a.tdt != SPEC_BF16 || a.ddt != SPEC_BF16 || a.V % 8 != 0 || a.max_k > RQ_MAX_K)
    return false;
  const size_t slice = (size_t)(a.V / 8 + RC_CLUSTER - 1) / RC_CLUSTER * 8;
  return (size_t)(2 * a.max_k + 1) * slice * 2 <= RC_DYN_SMEM;
}

// Co-resident clusters of the cluster-resident kernel on the current device
// (asked once per device).
static int cluster_count(const void *kernel) {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  int *c = &cache[dev];
  if (*c <= 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(RC_CLUSTER * num_sms(), 1, 1);
    cfg.blockDim = dim3(RC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = RC_DYN_SMEM;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = RC_CLUSTER;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) return -1;
    *c = n;
  }
  return *c;
}

int launch_setup_stream(const LinearArgs &a, cudaStream_t stream);

// Co-resident clusters of the one-cluster-per-request kernel with `smem`
// bytes of buffers per CTA on the current device (asked once per device and
// size).
static int cluster_small_count(size_t smem) {
  static std::mutex mu;
  static std::vector<std::pair<std::pair<int, size_t>, int>> known;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto &k : known)
    if (k.first.first == dev && k.first.second == smem) return k.second;
  if (cudaFuncSetAttribute(k_verify_cluster_small, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(RC_CLUSTER * num_sms(), 1, 1);
  cfg.blockDim = dim3(RC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = RC_CLUSTER;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (const void *)k_verify_cluster_small, &cfg) !=
          cudaSuccess ||
      n <= 0)
    return -1;
  known.push_back({{dev, smem}, n});
  return n;
}

int launch_verify_cluster_small(const LinearArgs &a, cudaStream_t stream) {
  if (check_upload(stream) != SPEC_OK) return SPEC_ERR_CUDA;
  RcArgs ra;
  ra.a = a;
  ra.slice = (a.V / 8 + RC_CLUSTER - 1) / RC_CLUSTER * 8;
  const size_t slice_bytes = (size_t)ra.slice * 2;
  ra.nbuf = (int)std::min<size_t>(std::max<size_t>(RQ_BUF_BYTES / slice_bytes, 2),
                                  (size_t)(2 * a.max_k + 1));
  const size_t smem = (size_t)ra.nbuf * slice_bytes;
  const int n = cluster_small_count(smem);
  if (n <= 0) return SPEC_ERR_CUDA;
  if (cudaFuncSetAttribute(k_verify_cluster_small, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return SPEC_ERR_CUDA;
  const int grid_clusters = std::min(n, a.B);
  cudaEvent_t before, after;
  take_row_pass_events(&before, &after);
  if (before && cudaEventRecord(before, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  k_verify_cluster_small<<<RC_CLUSTER * grid_clusters, RC_THREADS, smem, stream>>>(ra);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (after && cudaEventRecord(after, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

bool resident_supported(const LinearArgs &a) {
  return a.dk == SPEC_DRAFT_LOGITS && a.rule == SPEC_RULE_STRICT && !a.want_kl &&
         !a.want_rank && a.out_rank == nullptr && a.tdt == SPEC_BF16 && a.ddt == SPEC_BF16 &&
         a.V % 8 == 0 && a.V >= RC_MIN_V &&
         (a.V / 8 + RC_CLUSTER - 1) / RC_CLUSTER * 8 <= RC_SLICE_MAX;
}

int launch_verify_resident(const LinearArgs &a, cudaStream_t stream) {
  if (check_upload(stream) != SPEC_OK) return SPEC_ERR_CUDA;
  const size_t smem = RC_DYN_SMEM;
  if (cudaFuncSetAttribute(k_verify_resident, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return SPEC_ERR_CUDA;
  const int clusters = cluster_count((const void *)k_verify_resident);
  if (clusters <= 0) return SPEC_ERR_CUDA;
  const int rc = launch_setup_stream(a, stream);
  if (rc != SPEC_OK) return rc;
  RcArgs ra;
  ra.a = a;
  ra.slice = (a.V / 8 + RC_CLUSTER - 1) / RC_CLUSTER * 8;
  ra.nbuf = 0;   // (the small-call kernel's)
  cudaEvent_t before, after;
  take_row_pass_events(&before, &after);
  if (before && cudaEventRecord(before, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  k_verify_resident<<<RC_CLUSTER * clusters, RC_THREADS, smem, stream>>>(ra);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (after && cudaEventRecord(after, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

}  // namespace sv
