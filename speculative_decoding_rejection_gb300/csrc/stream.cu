// Streaming verifier: position-lazy linear verification in one persistent
// kernel.
//
// What it computes is the position-lazy schedule of the linear verifier
// (nalar.dev "Penolakan memendekkan pekerjaan speculative": proposals after
// a rejected one do not continue the committed prefix, so their rows are not
// needed). Position j of request b is decided once its target row p_{j+1}
// and, when the request samples, its draft row q_{j+1} are reduced and
// position j-1 was accepted: the lossless coin ("Acceptance Is Not Speed",
// §6; "RheoSampling 2026", §4 step 1), the CACTUS rule with its low-support
// guard, or the greedy prefix match (nalar.dev "Semantik penerimaan"). A
// rejection ends the request with the draw from norm(max(0, p - q))
// ("RheoSampling 2026", §4 step 3), K acceptances with the bonus draw from
// p_{K+1}, a greedy request with the target argmax.
//
// How (GB300): the CTA shape of the TMA row pass (one producer lane and four
// consumer warps over a two-stage ring of 16 KB bulk copies, six CTAs per
// SM), plus one service warp, over two work sources.
//   - The static list holds every position's rows in layer order: position 1
//     of every request, then position 2, and so on, each row split into
//     chunks. A producer skips a chunk of request b at position j once
//     b is known to have rejected an earlier position; by the time a layer
//     comes up the previous layer's decisions are mostly known, so the rows
//     after a rejection are mostly never read.
//   - Rows are split in 128 KB chunks (smaller chunks measured slower; the
//     residual's second read mostly misses L2 at every chunk size tried:
//     it comes long after the first read, once the position is decided).
//   - Chunk ends go to a service warp: each consumer warp leaves its partial
//     in a shared-memory queue record and goes on streaming; the CTA's sixth
//     warp publishes the four partials and counts one completion of the
//     position with a release atomic, off the consumers' path.
//   - A position is decided by whichever of two events comes second: its
//     rows complete, or the previous position accepted (an atomic join). An
//     acceptance whose next position is already complete decides that one
//     too, in the same service warp.
//   - A rejection of a sampling request appends its residual entry: the two
//     rows just decided on, streamed once more as tile pairs whose sums of
//     max(0, p - q) land in the job's tile-sum slots. Producers serve these
//     entries first, so the re-read follows the first read closely. The
//     final draws (these and the bonus draws) are queued as jobs for the
//     final-draw kernel, which runs after this kernel as in the multi-launch
//     schedule.
// Partials written by other CTAs are read through L2 (ld.global.cg) after an
// acquire; entries are published with a release store of their ready flag.
// Every wait is bounded (2 s of %globaltimer): on expiry the status word
// gets SPEC_ERR_TIMEOUT, producers stop issuing, and each CTA drains its own
// copies and returns.
#include <limits.h>

#include "common.cuh"
#include "internal.h"
#include "linear.cuh"
#include "rowpass.cuh"

namespace sv {

struct StreamEntry {   // the residual tile pairs of a rejected position
  int b;               // request
  int trow, drow;      // the rejected position's target and draft rows
  int job;             // index of the final-draw job (its tile-sum slots)
  float c;             // log2(e)/T
  int pad[3];
};
static_assert(sizeof(StreamEntry) == 32, "entries are two 16-byte words");

// Stage flags (m0.w).
constexpr int F_NVEC = 0xfff;       // 16-byte vectors in the stage (row stages)
constexpr int F_LAST = 1 << 12;     // last stage of its chunk / residual item
constexpr int F_DRAFT = 1 << 13;    // the draft tensor
constexpr int F_RES = 1 << 14;      // a residual tile pair
// bits 16-19 / 20-23: unaligned head / tail elements of the chunk

// CTA of the streaming verifier: the producer warp (lane 0 issues copies),
// four consumer warps, the service warp.
constexpr int ST_SERVICE_WARP = 1 + RS_CONS_WARPS;
constexpr int ST_THREADS = 32 * (2 + RS_CONS_WARPS);
constexpr int ST_CTAS_PER_SM = 6;
constexpr int ST_RANK_CTAS_PER_SM = 5;
constexpr int NQ = 8;   // chunk-end records in flight per CTA

struct StreamSmem {
  uint64_t full[NSTAGE];
  uint64_t empty[NSTAGE];
  int4 m0[NSTAGE];     // {part slot (-1: end of work), chunk or tile, first element, flags}
  int4 m1[NSTAGE];     // {c bits, row (residual: elements), head element (residual: first
                       //  tile of the item), tail element (residual: tiles in the item)}
  int4 m2[NSTAGE];     // rows: {request, items of the position, j | K << 16, target row};
                       // residual: {request, items of the entry, job, first tile}
  float4 law[NSTAGE];  // residual stages: m_t, 1/S_t, m_d, 1/S_d
  float thr[NSTAGE];   // rank threshold of a target row (+inf: none)
  // chunk-end queue, consumers to the service warp: record e sits in slot
  // e % NQ; every consumer warp leaves its partial (row chunks) or its tile
  // sums (residual items) there and arrives on qfull, the service warp
  // arrives on qempty once it has taken the record
  uint64_t qfull[NQ];
  uint64_t qempty[NQ];
  int4 qm0[NQ], qm1[NQ], qm2[NQ];   // the chunk's last stage's m0, m1, m2 (m0.x < 0: end)
  Part qp[NQ][RS_CONS_WARPS];
  float qt[NQ][RS_CONS_WARPS][RES_TILES_PER_ITEM];
  int abort;
  int skip;            // the setup rejected the inputs: no work
};

// ---------------------------------------------------------- memory order
// Returns the old value; this thread's earlier writes are visible to any
// thread that acquires the new one.
__device__ __forceinline__ int atom_add_release(int *p, int v) {
  if (!GCHK(p, 4)) return -1;
  int old;
  asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}
__device__ __forceinline__ void fence_acquire() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ void st_release(int *p, int v) {
  if (!GCHK(p, 4)) return;
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int *p) {
  if (!GCHK(p, 4)) return 0;
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ StreamEntry ldcg_entry(const StreamEntry *e) {
  const int4 *p = reinterpret_cast<const int4 *>(e);
  const int4 x = GLDCG(p), y = GLDCG(p + 1);
  return StreamEntry{x.x, x.y, x.z, x.w, __int_as_float(y.x), {0, 0, 0}};
}
__device__ __forceinline__ void st_entry(StreamEntry *e, const StreamEntry &v) {
  int4 *p = reinterpret_cast<int4 *>(e);
  GST(p, make_int4(v.b, v.trow, v.drow, v.job));
  GST(p + 1, make_int4(__float_as_int(v.c), 0, 0, 0));
}
__device__ __forceinline__ Job ldcg_job(const Job *j) {
  const int4 *p = reinterpret_cast<const int4 *>(j);
  const int4 x = GLDCG(p), y = GLDCG(p + 1);
  return Job{x.x, x.y, x.z, x.w, __int_as_float(y.x), __int_as_float(y.y), __int_as_float(y.z),
             __int_as_float(y.w)};
}

// ------------------------------------------------------------------ setup
// One thread per (request b, position j): position j's counters (position 0
// needs no acceptance) and, for a draft position, the draft token's logits
// z_t(d_j) (also the rank count's threshold) and z_d(d_j), gathered once so
// a decision needs no dependent load; thread (b, 0) also writes the
// request's record, its first rejection (none) and its residual entry's
// flag and count. Every draft token must be a vocabulary id (the eager
// schedule checks them all, so this one does too).
constexpr int SETUP_STREAM_THREADS = 128;

__global__ void __launch_bounds__(SETUP_STREAM_THREADS) k_setup_stream(const LinearArgs a) {
  const int W = a.max_k + 1;
  const long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (g >= (long long)a.B * W) return;
  const int b = (int)(g / W), j = (int)(g % W);
  GST(a.pos_done + (g), 0);
  GST(a.pos_join + (g), j == 0);
  ReqInfo r;
  const bool ok = load_request(a, b, r);   // every thread of b: the same record
  if (j == 0) {
    GST(a.ready_d + (b), 0);
    GST(a.ready_d + (a.cap_d + b), 0);
    GST(a.rej_at + (b), INT_MAX);
    GST(a.req + (b), r);
    if (!ok) a.hdr->setup_bad = 1;
  }
  if (!ok || j > r.K) return;
  if (j == r.K) {
    GST(a.rank_thr + (r.t0 + r.K), INFINITY);
    return;
  }
  const bool drow = r.mode == MODE_SAMPLE && a.stream_draft;
  const int d = GLD(a.tokens + (r.d0 + j));
  const bool dok = (unsigned)d < (unsigned)a.V;
  if (!dok) {
    set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);
    a.hdr->setup_bad = 1;
  }
  GST(a.rank_thr + (r.t0 + j), dok ? load_elem(a.target + (long long)(r.t0 + j) * a.t_row_bytes, a.tdt, d) : INFINITY);
  if (drow)
    GST(a.zd_at + (r.d0 + j), dok ? load_elem(a.draft + (long long)(r.d0 + j) * a.d_row_bytes, a.ddt, d) : 0.f);
}

// --------------------------------------------------------------- producer
__device__ __forceinline__ bool acquire_stage(StreamSmem &sh, long long it, volatile int *abort) {
  const int s = (int)(it % NSTAGE);
  const long long use = it / NSTAGE;
  return use == 0 || mbar_wait_bounded(&sh.empty[s], (uint32_t)((use - 1) & 1), abort);
}

// The producer's held ticket of the dynamic queue (residual items).
struct DynTicket {
  unsigned long long t, n;   // the ticket, and the number of tickets in all
};

__device__ bool issue_res_item(const LinearArgs &a, StreamSmem &sh, unsigned char *stage_buf,
                               long long &it, volatile int *abort, const StreamEntry &E, int g);

// Serves the held residual ticket if its entry is published (a relaxed poll,
// then an acquire), and takes the next ticket. False when a wait gave up.
__device__ __forceinline__ bool serve_ready_ticket(const LinearArgs &a, StreamSmem &sh,
                                                   unsigned char *stage_buf, long long &it,
                                                   volatile int *abort, DynTicket &dy,
                                                   bool &served) {
  served = false;
  if (dy.t >= dy.n) return true;
  const int e = (int)(dy.t / (unsigned)a.n_res_items);
  if (!GCHK(a.ready_d + e, 4) || !*(volatile int *)(a.ready_d + e)) return true;
  fence_acquire();
  const StreamEntry E = ldcg_entry(a.ent_d + e);
  if (!issue_res_item(a, sh, stage_buf, it, abort, E, (int)(dy.t % (unsigned)a.n_res_items)))
    return false;
  dy.t = atomicAdd(&a.hdr->work_d, 1ull);
  served = true;
  return true;
}

// Streams chunk `chunk` of one row into the ring: its 16-byte aligned
// interior in TMA bulk copies of up to 16 KB, the unaligned head and tail
// left to the consumers' scalar loads. m2 travels with every stage.
template <bool RANK>
__device__ bool issue_row_chunk(const LinearArgs &a, StreamSmem &sh, unsigned char *stage_buf,
                                long long &it, volatile int *abort, int slot, bool draft,
                                int row, int chunk, float c, int4 m2) {
  const long long rbytes = draft ? a.d_row_bytes : a.t_row_bytes;
  const int esz = dtype_size(draft ? a.ddt : a.tdt);
  const uint64_t row0 = (uint64_t)((draft ? a.draft : a.target) + (long long)row * rbytes);
  const uint64_t cb0 = row0 + (uint64_t)chunk * a.chunk_bytes;
  const uint64_t cb1 = min(row0 + (uint64_t)rbytes, cb0 + (uint64_t)a.chunk_bytes);
  uint64_t A0 = (cb0 + 15) & ~15ull, A1 = cb1 & ~15ull;
  if (A1 <= A0) A0 = A1 = cb1;   // no aligned interior: all scalar
  const int ntile = A1 > A0 ? (int)((A1 - A0 + TILE_BYTES - 1) / TILE_BYTES) : 1;
  const int head_n = (int)((A0 - cb0) / esz), tail_n = (int)((cb1 - A1) / esz);
  const float thr = RANK && !draft ? GLD(a.rank_thr + (row)) : INFINITY;
  for (int tl = 0; tl < ntile; ++tl) {
    if (!acquire_stage(sh, it, abort)) return false;
    const int s = (int)(it % NSTAGE);
    const uint64_t off = A0 + (uint64_t)tl * TILE_BYTES;
    const uint32_t nb = (uint32_t)min((uint64_t)TILE_BYTES, A1 - off);
    sh.m0[s] = make_int4(slot, chunk, (int)((off - row0) / esz),
                         (int)(nb / 16) | (tl == ntile - 1 ? F_LAST : 0) | (draft ? F_DRAFT : 0) |
                             (head_n << 16) | (tail_n << 20));
    sh.m1[s] = make_int4(__float_as_int(c), row, (int)((cb0 - row0) / esz),
                         (int)((A1 - row0) / esz));
    sh.m2[s] = m2;
    if (RANK) sh.thr[s] = thr;
    if (nb > 0) {
      mbar_arrive_tx(&sh.full[s], nb);
      bulk_g2s(stage_buf + (size_t)s * TILE_BYTES, (const void *)off, nb, &sh.full[s]);
    } else {
      mbar_arrive(&sh.full[s]);
    }
    ++it;
  }
  return true;
}

// Static ticket t: position j of request b (layer order), chunk k of its
// target row, then of its draft row. Skipped when the position does not
// exist, when b already rejected an earlier position (a stale view only
// costs a read that turns out unneeded), or when k names no chunk. Partial
// slots are by absolute row: target row r at slot r, draft row r at slot
// rt_max + r.
template <bool RANK>
__device__ bool issue_static(const LinearArgs &a, StreamSmem &sh, unsigned char *stage_buf,
                             long long &it, volatile int *abort, unsigned long long t) {
  const unsigned long long e = t / (unsigned)a.stride;
  const int k = (int)(t % (unsigned)a.stride);
  const int j = (int)(e / (unsigned)a.B), b = (int)(e % (unsigned)a.B);
  const ReqInfo r = GLD(a.req + (b));
  const int rej = GLDCG(a.rej_at + b);
  if (r.mode == MODE_SKIP || j > r.K || j > rej) return true;
  const bool drow = r.mode == MODE_SAMPLE && a.stream_draft && j < r.K;
  const int4 m2 = make_int4(b, a.nch_t + (drow ? a.nch_d : 0), j | (r.K << 16), r.t0 + j);
  if (k < a.nch_t)
    return issue_row_chunk<RANK>(a, sh, stage_buf, it, abort, r.t0 + j, false, r.t0 + j, k, r.c,
                                 m2);
  if (drow && k - a.nch_t < a.nch_d)
    return issue_row_chunk<RANK>(a, sh, stage_buf, it, abort, a.rt_max + r.d0 + j, true,
                                 r.d0 + j, k - a.nch_t, r.c, m2);
  return true;
}

// Residual item g of entry E: up to RES_TILES_PER_ITEM tiles, each
// SAMPLE_TILE bf16 of the target row and the same elements of the draft row
// side by side in one stage.
__device__ bool issue_res_item(const LinearArgs &a, StreamSmem &sh, unsigned char *stage_buf,
                               long long &it, volatile int *abort, const StreamEntry &E, int g) {
  if (g >= a.n_res_items) return true;
  const Job job = ldcg_job(a.jobs_a + E.job);
  const float4 law = make_float4(job.mt, 1.f / job.St, job.md, job.Sd > 0.f ? 1.f / job.Sd : 0.f);
  const uint64_t trow = (uint64_t)(a.target + (long long)E.trow * a.t_row_bytes);
  const uint64_t drow = (uint64_t)(a.draft + (long long)E.drow * a.d_row_bytes);
  const int j0 = g * RES_TILES_PER_ITEM, j1 = min(a.ntiles, j0 + RES_TILES_PER_ITEM);
  for (int j = j0; j < j1; ++j) {
    if (!acquire_stage(sh, it, abort)) return false;
    const int s = (int)(it % NSTAGE);
    const int e0 = j * SAMPLE_TILE;
    const int ne = min(SAMPLE_TILE, a.V - e0);
    const uint32_t nb = (uint32_t)ne * 2;
    sh.m0[s] = make_int4(E.b, j, e0, F_RES | (j == j1 - 1 ? F_LAST : 0));
    sh.m1[s] = make_int4(__float_as_int(E.c), ne, j0, j1 - j0);
    sh.m2[s] = make_int4(E.b, a.n_res_items, E.job, j0);
    sh.law[s] = law;
    mbar_arrive_tx(&sh.full[s], 2 * nb);
    unsigned char *dst = stage_buf + (size_t)s * TILE_BYTES;
    bulk_g2s(dst, (const void *)(trow + 2ull * e0), nb, &sh.full[s]);
    bulk_g2s(dst + TILE_BYTES / 2, (const void *)(drow + 2ull * e0), nb, &sh.full[s]);
    ++it;
  }
  return true;
}

// ------------------------------------------------------- request progress
// Request b's final token is written (or queued as a final-draw job). The
// last request to finish moves the errors the decisions reported (empty
// rows) into the status word.
__device__ void finish_one(const LinearArgs &a, int lane) {
  if (lane == 0) {
    __threadfence();
    const int old = atomicAdd(&a.hdr->n_done, 1);
    if (old + 1 == a.B) {
      const int st = *(volatile int *)&a.err->status;
      if (st != SPEC_OK) set_status(a.hdr, st, *(volatile int *)&a.err->detail);
    }
  }
  __syncwarp();
}

// Row statistics of at most 32 chunk partials held one per lane, merged in
// the order of warp_row_stat (the same bits).
__device__ __forceinline__ RowStat lane_parts_stat(const Part &p, bool have, float c) {
  float m = NO_MAX, S = 0.f;
  int idx = 0x7fffffff;
  if (have) merge_stat(m, S, idx, p.m, p.S, p.idx, c);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float S2 = __shfl_xor_sync(0xffffffffu, S, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    merge_stat(m, S, idx, m2, S2, i2, c);
  }
  return RowStat{m, S, idx};
}

// Adds one event to position j's join (rows complete, previous position
// accepted); true for the second of the two.
__device__ __forceinline__ bool join_second(const LinearArgs &a, int b, int j) {
  int *pj = a.pos_join + b * (a.max_k + 1) + j;
  const bool second = GCHK(pj, 4) && atomicAdd(pj, 1) == 1;
  if (second) __threadfence();
  return second;
}

// Decisions on request b from position j on (target rows from t0, K
// drafts, c = log2(e)/T, 0 for greedy): both of position j's events are in.
// Every input of a decision comes from one round of independent loads: the
// chunk partials, the token and the gathered logits z_t(d), z_d(d). An
// accepted position whose successor's rows are already complete goes on to
// decide the successor.
__device__ __noinline__ void stream_decide(const LinearArgs &a, int b, int j, int K, int t0,
                                           float c, int lane) {
  ReqInfo r;
  r.t0 = t0;
  r.d0 = t0 - b;
  r.K = K;
  r.mode = c != 0.f ? MODE_SAMPLE : MODE_GREEDY;
  r.c = c;
  r.n = 0;
  r.pad[0] = r.pad[1] = 0;
  const bool sample = r.mode == MODE_SAMPLE;
  const bool fast = a.nch_t * RS_CONS_WARPS <= 32 && a.nch_d * RS_CONS_WARPS <= 32;
  while (true) {
    const bool drow = sample && a.stream_draft && j < K;
    const int tslot = r.t0 + j, dslot = a.rt_max + r.d0 + j;
    const bool th = lane < a.nch_t * RS_CONS_WARPS, dh = drow && lane < a.nch_d * RS_CONS_WARPS;
    Part tp{}, dp{};
    int d = -1;
    float zt = 0.f, zd = 0.f;
    if (fast && th) tp = ldcg_part(a.part + (long long)tslot * a.nch_max * RS_CONS_WARPS + lane);
    if (fast && dh) dp = ldcg_part(a.part + (long long)dslot * a.nch_max * RS_CONS_WARPS + lane);
    if (j < K) {
      d = GLD(a.tokens + (r.d0 + j));
      zt = GLDCG(a.rank_thr + r.t0 + j);
      if (drow) zd = GLDCG(a.zd_at + r.d0 + j);
    }
    const RowStat ts = fast ? lane_parts_stat(tp, th, c) : target_stat(a, tslot, c, lane);
    RowStat ds{NO_MAX, 0.f, 0x7fffffff};
    int n = K;
    if (j < K) {
      int rank = 0;
      if (a.want_rank) {
        if (fast) {
          rank = th ? tp.cnt : 0;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
          rank += 1;
        } else {
          rank = 1 + warp_row_count(a, tslot, lane);
        }
      }
      if (drow) ds = fast ? lane_parts_stat(dp, dh, c) : draft_stat(a, dslot, c, lane);
      const bool rej = __shfl_sync(
          0xffffffffu,
          lane == 0 && position_rejects_z(a, b, r, j, sample, ts, ds, rank, d, zt, zd, false), 0);
      if (!rej) {   // accepted: position j + 1 is decided once its rows are complete
        const bool go = __shfl_sync(0xffffffffu, lane == 0 && join_second(a, b, j + 1), 0);
        if (!go) return;
        ++j;
        continue;
      }
      n = j;
      if (lane == 0) GST(a.rej_at + (b), j);   // later positions' rows are no longer read
    }
    // positions after n+1 are not reported
    for (int i = n + 1 + lane; i < K; i += 32) {
      if (a.out_pq) {
        GST(a.out_pq + (2LL * (r.d0 + i)), __int_as_float(0x7fc00000));
        GST(a.out_pq + (2LL * (r.d0 + i) + 1), __int_as_float(0x7fc00000));
      }
      if (a.out_rank) GST(a.out_rank + (r.d0 + i), -1);
    }
    const int W = a.max_k + 1;
    int32_t *out = a.out_tokens + (long long)b * W;
    for (int jj = lane; jj < W; jj += 32) GST(out + jj, jj < n ? GLD(a.tokens + (r.d0 + jj)) : -1);
    if (lane == 0) GST(a.out_accepted + (b), n);
    __syncwarp();
    if (!sample) {   // greedy: the target's argmax replaces the rejected draft
      if (lane == 0) GST(out + n, ts.idx);
      finish_one(a, lane);
      return;
    }
    const bool residual = n < K && a.stream_draft;
    if (lane == 0) {
      if (residual) {
        // the residual's tile sums are summed in this kernel, the draw after it
        const int ja = atomicAdd(&a.hdr->n_jobs_a, 1);
        GST(a.jobs_a + (ja), Job{b, n, 1, 0, ts.m, ts.S, ds.m, ds.S});
        const int e = atomicAdd(&a.hdr->n_alloc_d, 1);   // < B: one per request
        st_entry(a.ent_d + e, StreamEntry{b, r.t0 + n, r.d0 + n, ja, c, {0, 0, 0}});
        __threadfence();
        st_release(a.ready_d + e, 1);
      } else {   // bonus draw from p_{K+1}, after this kernel
        GST(a.jobs_b + (atomicAdd(&a.hdr->n_jobs_b, 1)), Job{b, n, 2, 0, ts.m, ts.S, 0.f, 0.f});
      }
    }
    if (!residual) finish_one(a, lane);
    __syncwarp();
    return;
  }
}

// The service warp on chunk-end record q (a row chunk, or a residual item):
// the four consumer warps' results to global memory, the record's slot back
// to the consumers, one completion of the position's rows (or of the
// residual entry), and, for the last completion, the position's join (its
// decision when the previous position was accepted) or the end of the
// request. Only this warp waits on global memory.
__device__ __forceinline__ void service_record(const LinearArgs &a, StreamSmem &sh, int q,
                                               int lane, const int4 m0, const int4 m1,
                                               const int4 m2) {
  const bool res = (m0.w & F_RES) != 0;
  int go = 0;
  if (lane == 0) {
    int *count;
    if (res) {   // m2.z: job, m2.w: first tile, m1.w: tiles in the item
      for (int t = 0; t < m1.w; ++t)
        GST(reinterpret_cast<float4 *>(a.tsum) + (long long)m2.z * a.ntiles + m2.w + t,
            make_float4(sh.qt[q][0][t], sh.qt[q][1][t], sh.qt[q][2][t], sh.qt[q][3][t]));
      count = a.ready_d + a.cap_d + m2.x;   // the residual entry's own count
    } else {
      Part *dst = a.part + ((long long)m0.x * a.nch_max + m0.y) * RS_CONS_WARPS;
#pragma unroll
      for (int w = 0; w < RS_CONS_WARPS; ++w) GST(dst + w, sh.qp[q][w]);
      count = a.pos_done + m2.x * (a.max_k + 1) + (m2.z & 0xffff);
    }
    mbar_arrive(&sh.qempty[q]);   // the record is in registers and global memory
    if (atom_add_release(count, 1) + 1 == m2.y) {
      fence_acquire();
      go = res ? 1 : join_second(a, m2.x, m2.z & 0xffff);
    }
  }
  if (!__shfl_sync(0xffffffffu, go, 0)) return;
  if (res) finish_one(a, lane);
  else stream_decide(a, m2.x, m2.z & 0xffff, m2.z >> 16, m2.w - (m2.z & 0xffff),
                     __int_as_float(m1.x), lane);
}

// A consumer warp at chunk end e (row partial p, or residual tile sums rs):
// waits until record slot e % NQ is free, leaves its result there (warp 0 of
// the consumers also the stage's metadata) and arrives on the slot. False
// when the wait gave up.
__device__ __forceinline__ bool push_record(StreamSmem &sh, unsigned e, int cw, int lane,
                                            volatile int *abort, bool res, const Part &p,
                                            const float (&rs)[RES_TILES_PER_ITEM], const int4 m0,
                                            const int4 m1, const int4 m2) {
  const int q = (int)(e % NQ);
  if (e >= NQ && !mbar_wait_bounded(&sh.qempty[q], (uint32_t)((e / NQ - 1) & 1), abort))
    return false;
  if (lane == 0) {
    if (res) {
#pragma unroll
      for (int t = 0; t < RES_TILES_PER_ITEM; ++t) sh.qt[q][cw][t] = rs[t];
    } else {
      sh.qp[q][cw] = p;
    }
    if (cw == 0) {
      sh.qm0[q] = m0;
      sh.qm1[q] = m1;
      sh.qm2[q] = m2;
    }
    mbar_arrive(&sh.qfull[q]);
  }
  __syncwarp();
  return true;
}

// ------------------------------------------------------------------ kernel
template <bool RANK>
__global__ void __launch_bounds__(ST_THREADS, RANK ? ST_RANK_CTAS_PER_SM : ST_CTAS_PER_SM)
    k_verify_stream(const LinearArgs a) {
  extern __shared__ __align__(128) unsigned char dsmem[];
  __shared__ StreamSmem sh;
  unsigned char *stage_buf = dsmem;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], RS_CONS_WARPS);
    }
    for (int q = 0; q < NQ; ++q) {
      mbar_init(&sh.qfull[q], RS_CONS_WARPS);
      mbar_init(&sh.qempty[q], 1);
    }
    sh.abort = 0;
    // the setup's verdict (fixed before this kernel starts); errors found
    // while it runs go to the status word without stopping the other requests
    sh.skip = *(volatile int *)&a.hdr->setup_bad;
    fence_mbar_init();
  }
  __syncthreads();
  if (sh.skip) {   // inputs rejected by the setup: nothing is verified
    const int W = a.max_k + 1;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < (long long)a.B * W;
         i += (long long)gridDim.x * blockDim.x) {
      GST(a.out_tokens + (i), -1);
      if (i < a.B) GST(a.out_accepted + (i), -1);
    }
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int *abort = &sh.abort;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    long long it = 0;
    bool ok = true;
    const unsigned long long n_static =
        (unsigned long long)(a.max_k + 1) * (unsigned)a.B * (unsigned)a.stride;
    const unsigned long long n_dyn = (unsigned long long)a.cap_d * a.n_res_items;
    unsigned long long st_t = atomicAdd(&a.hdr->work_s, 1ull);
    DynTicket dy{atomicAdd(&a.hdr->work_d, 1ull), n_dyn};
    while (true) {
      // 1. the held residual ticket, once its entry exists
      bool served;
      if (!serve_ready_ticket(a, sh, stage_buf, it, abort, dy, served)) {
        ok = false;
        break;
      }
      if (served) continue;
      // 2. the static list meanwhile
      if (st_t < n_static) {
        const unsigned long long next = atomicAdd(&a.hdr->work_s, 1ull);
        if (!issue_static<RANK>(a, sh, stage_buf, it, abort, st_t)) {
          ok = false;
          break;
        }
        st_t = next;
        continue;
      }
      // 3. nothing else: wait for the ticket's entry, the last request or an error
      // (1: entry ready, 2: every request finished, 3: give up)
      const int e = (int)(dy.t / (unsigned)a.n_res_items);
      const int outcome = poll_bounded(
          [&]() -> int {
            if (dy.t < n_dyn && ld_acquire(a.ready_d + e)) return 1;
            if (*(volatile int *)&a.hdr->n_done >= a.B) return 2;
            if (*(volatile int *)&a.hdr->status == SPEC_ERR_TIMEOUT || *abort) return 3;
            return 0;
          },
          3, WAIT_NS);
      if (outcome == 1) continue;
      ok = outcome == 2;
      break;
    }
    if (ok && acquire_stage(sh, it, abort)) {   // end marker
      const int s = (int)(it % NSTAGE);
      sh.m0[s] = make_int4(-1, 0, 0, 0);
      mbar_arrive(&sh.full[s]);
      return;
    }
    // gave up: record it, tell the consumers, then wait (bounded) for this
    // CTA's copies in flight
    set_status(a.hdr, SPEC_ERR_TIMEOUT, -2);
    *abort = 1;
    for (int s = 0; s < NSTAGE; ++s) {
      const long long issued = (it - s + NSTAGE - 1) / NSTAGE;   // uses of stage s
      if (issued > 0) {
        volatile int never = 0;
        mbar_wait_bounded(&sh.full[s], (uint32_t)((issued - 1) & 1), &never);
      }
    }
    return;
  }

  if (warp == ST_SERVICE_WARP) {
    // ------------------------------------------------------------- service
    for (unsigned e = 0;; ++e) {
      const int q = (int)(e % NQ);
      if (!mbar_wait_bounded(&sh.qfull[q], (uint32_t)((e / NQ) & 1), abort)) {
        if (!*abort) set_status(a.hdr, SPEC_ERR_TIMEOUT, -4);
        *abort = 1;
        return;
      }
      const int4 m0 = sh.qm0[q];
      if (m0.x < 0) return;   // the consumers reached the end marker
      service_record(a, sh, q, lane, m0, sh.qm1[q], sh.qm2[q]);
    }
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1;
  const int ctid = threadIdx.x - 32;
  RunState st{NO_MAX, pk2(0.f, 0.f), 0x7fffffff, 0, 0u};
  float rsum[RES_TILES_PER_ITEM] = {};
  unsigned ends = 0;   // chunk-end records pushed (the same count in every consumer warp)
  for (long long it = 0;; ++it) {
    const int s = (int)(it % NSTAGE);
    if (!mbar_wait_bounded(&sh.full[s], (uint32_t)((it / NSTAGE) & 1), abort)) {
      if (!*abort) set_status(a.hdr, SPEC_ERR_TIMEOUT, -3);
      *abort = 1;
      return;
    }
    const int4 m0 = sh.m0[s];
    if (m0.x < 0) {   // end of work: an end record tells the service warp
      push_record(sh, ends, cw, lane, abort, false, Part{}, rsum, m0, m0, m0);
      return;
    }
    const int4 m1 = sh.m1[s];
    const int4 m2 = sh.m2[s];
    const unsigned char *buf = stage_buf + (size_t)s * TILE_BYTES;
    const bool res = (m0.w & F_RES) != 0;
    const bool last = (m0.w & F_LAST) != 0;
    Part p{};
    if (res) {   // residual tile pair: tile m0.y, the item's tiles start at m1.z
      const float4 lw = sh.law[s];
      const ResLaw L{lw.x, lw.y, lw.z, lw.w, __int_as_float(m1.x)};
      const int ne = m1.y;
      float r = ne == SAMPLE_TILE ? consume_res_full(buf, ctid, L)
                                  : consume_res_partial(buf, ctid, ne, L);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
#pragma unroll
      for (int q = 0; q < RES_TILES_PER_ITEM; ++q)
        if (q == m0.y - m1.z) rsum[q] = r;
    } else {
      const int nvec = m0.w & F_NVEC;
      const bool draft = (m0.w & F_DRAFT) != 0;
      const int dt = draft ? a.ddt : a.tdt;
      const float c = __int_as_float(m1.x);
      const float thr = RANK ? sh.thr[s] : INFINITY;
      consume_row_stage<RANK>(buf, nvec, m0.z, c, dt == SPEC_BF16, thr, ctid, st);
      if (last) {
        if (cw == 0) {
          const char *row = (draft ? a.draft : a.target) +
                            (long long)m1.y * (draft ? a.d_row_bytes : a.t_row_bytes);
          consume_head_tail(row, dt, m0.w, m1.z, m1.w, c, thr, lane, st);
        }
        p = finish_row_chunk<RANK>(st, c);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
    if (last) {
      if (!push_record(sh, ends, cw, lane, abort, res, p, rsum, m0, m1, m2)) {
        if (!*abort) set_status(a.hdr, SPEC_ERR_TIMEOUT, -5);
        *abort = 1;
        return;
      }
      ++ends;
    }
  }
}

// The streaming setup on its own (the cluster-resident verifier uses its
// request records and gathered draft logits).
int launch_setup_stream(const LinearArgs &a, cudaStream_t stream) {
  if (check_upload(stream) != SPEC_OK) return SPEC_ERR_CUDA;
  const long long n_setup = (long long)a.B * (a.max_k + 1);
  k_setup_stream<<<(unsigned)((n_setup + SETUP_STREAM_THREADS - 1) / SETUP_STREAM_THREADS),
                   SETUP_STREAM_THREADS, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

bool stream_supported(const LinearArgs &a) {
  return a.dk == SPEC_DRAFT_LOGITS && a.rule != SPEC_RULE_STRICT_TOP128 && !a.want_kl &&
         a.tdt == SPEC_BF16 && a.ddt == SPEC_BF16 && a.V % 8 == 0;
}

int launch_verify_stream(const LinearArgs &a, cudaStream_t stream) {
  if (check_upload(stream) != SPEC_OK) return SPEC_ERR_CUDA;
  const int sms = num_sms();
  if (sms <= 0) return SPEC_ERR_CUDA;
  const long long n_setup = (long long)a.B * (a.max_k + 1);
  k_setup_stream<<<(unsigned)((n_setup + SETUP_STREAM_THREADS - 1) / SETUP_STREAM_THREADS),
                   SETUP_STREAM_THREADS, 0, stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  const size_t smem = (size_t)NSTAGE * TILE_BYTES;
  auto kern = a.want_rank ? k_verify_stream<true> : k_verify_stream<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return SPEC_ERR_CUDA;
  cudaEvent_t before, after;
  take_row_pass_events(&before, &after);
  if (before && cudaEventRecord(before, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  kern<<<(a.want_rank ? ST_RANK_CTAS_PER_SM : ST_CTAS_PER_SM) * sms, ST_THREADS, smem, stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (after && cudaEventRecord(after, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

}  // namespace sv
