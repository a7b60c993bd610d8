// Row-statistics pass: one streaming read of every listed vocabulary row.
//
// For each row it produces, per chunk and consumer warp, the max logit m,
// S = sum_x 2^((z_x - m) c) with c = log2(e)/T (the softmax normaliser of
// softmax(z/T) up to the factor 2^(m c)), and the lowest index attaining m.
// These give p(d) = 2^((z_d - m) c) / S and the greedy argmax without a
// second read ("RheoSampling 2026", §1 and §7: temperature applies to the
// verification softmax; nalar.dev "Semantik penerimaan": greedy compares the
// draft with the target's argmax).
//
// Design: a persistent grid (2 CTAs per SM). Warp 0 lane 0 is the producer:
// it takes work items (row, 64 KB chunk) from a global counter and streams
// each chunk into a ring of NSTAGE 16 KB shared-memory stages with 1-D TMA
// bulk copies, completion tracked by mbarriers. Warps 1..8 consume stages
// with 128-bit shared loads; one 2^x (MUFU) per element for softmax rows,
// none for argmax-only rows. No cross-warp barrier: each consumer warp writes
// its own partial. Every wait is bounded; on expiry the status word gets
// SPEC_ERR_TIMEOUT and the CTA drains its own copies and returns.
#include "common.cuh"
#include "internal.h"

namespace sv {

// With RANK, the consumers of a target row also count the logits strictly
// above the row's threshold (the draft token's own logit): the draft token's
// target rank minus one ("Acceptance Is Not Speed", §6 rule 1, the
// low-support guard on target rank), one packed bf16 compare per two
// elements.
//
// Stage metadata, two 16-byte records read with one shared load each:
//   m0 = {slot (-1: no more work), chunk, e_first, flags}
//   m1 = {c (float bits), row, head_e, tail_e}
// flags: nvec (bits 0-11), last stage of its chunk (bit 12), draft tensor
// (bit 13), head_n (bits 16-19), tail_n (bits 20-23).
struct RowPassSmem {
  uint64_t full[NSTAGE];
  uint64_t empty[NSTAGE];
  int4 m0[NSTAGE];
  int4 m1[NSTAGE];
  float thr[NSTAGE];   // rank threshold of the stage's row (+inf: none)
  int abort;
};

constexpr int FULL_NVEC = TILE_BYTES / 16;            // vectors in a full stage
constexpr int NCT = RS_CONS_WARPS * 32;               // consumer threads
constexpr int VEC_PER_THREAD = FULL_NVEC / NCT;       // 4
static_assert(FULL_NVEC % NCT == 0, "full stages split evenly");
static_assert((VEC_PER_THREAD & (VEC_PER_THREAD - 1)) == 0, "power-of-two vectors per thread");

// Running state of one consumer thread over a chunk: max logit m, the
// normaliser as a packed pair S2 (its two lanes summed at the chunk end) and
// the lowest index attaining m.
struct RunState {
  float m;
  f32x2 S2;
  int idx;
  int cnt;        // rank count (generic path)
  uint32_t cnt2;  // rank count, two 16-bit lanes (packed bf16 path)
};

__device__ __forceinline__ void rescale(RunState &st, float m_new, float c) {
  const float f = ex2((st.m - m_new) * c);
  st.S2 = mul2(st.S2, pk2(f, f));
  st.m = m_new;
}

__device__ __forceinline__ void scalar_update(float x, int e, float c, RunState &st,
                                              float thr) {
  st.cnt += x > thr;
  if (x > st.m) {
    if (c != 0.f) rescale(st, x, c);
    st.m = x;
    st.idx = e;
  } else if (x == st.m && e < st.idx) {
    st.idx = e;
  }
  if (c != 0.f) st.S2 = add2(st.S2, pk2(ex2((x - st.m) * c), 0.f));
}

// Generic path: one 16-byte vector (partial stages and fp32 rows).
template <bool SOFTMAX, bool BF16>
__device__ __forceinline__ void consume_vec(const uint4 w, int e, float c, RunState &st,
                                            float thr) {
  constexpr int N = BF16 ? 8 : 4;
  float x[N];
  if (BF16) {
    x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
    x[4] = bf16lo(w.z); x[5] = bf16hi(w.z); x[6] = bf16lo(w.w); x[7] = bf16hi(w.w);
  } else {
    x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
  }
  float vm = x[0];
#pragma unroll
  for (int k = 1; k < N; ++k) vm = fmaxf(vm, x[k]);
#pragma unroll
  for (int k = 0; k < N; ++k) st.cnt += x[k] > thr;
  if (vm > st.m) {
    int j = N - 1;
#pragma unroll
    for (int k = N - 2; k >= 0; --k)
      if (x[k] == vm) j = k;
    if (SOFTMAX) rescale(st, vm, c);
    st.m = vm;
    st.idx = e + j;
  }
  if (SOFTMAX) {
    const f32x2 c2 = pk2(c, c), nm = pk2(-st.m, -st.m);
    f32x2 acc = pk2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < N; k += 2) {
      const f32x2 t = mul2(add2(pk2(x[k], x[k + 1]), nm), c2);
      acc = add2(acc, pk2(ex2(lo2(t)), ex2(hi2(t))));
    }
    st.S2 = add2(st.S2, acc);
  }
}

// Lowest element index holding `vm` among this thread's bf16 vectors of a
// full stage (vector k sits at element e0 + 8 * NCT * k).
__device__ __forceinline__ int first_index_of(const uint4 (&v)[VEC_PER_THREAD], float vm, int e0) {
  int found = e0;
  bool done = false;
#pragma unroll
  for (int k = 0; k < VEC_PER_THREAD; ++k) {
    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e = e0 + 8 * NCT * k + 2 * q;
      if (!done && bf16lo(w[q]) == vm) { found = e; done = true; }
      if (!done && bf16hi(w[q]) == vm) { found = e + 1; done = true; }
    }
  }
  return found;
}

// Fast path: a full bf16 stage, 32 elements per thread. The max goes through
// packed bf16 compares and is checked once; exponents are formed with
// mixed-precision subtracts and packed multiplies, one 2^x per element, and
// the 32 terms are summed as a packed pairwise tree.
template <bool SOFTMAX, bool RANK>
__device__ __forceinline__ void consume_full_bf16(const unsigned char *buf, int ctid, int e_first,
                                                  float c, RunState &st, uint32_t thr2) {
  uint4 v[VEC_PER_THREAD];
#pragma unroll
  for (int k = 0; k < VEC_PER_THREAD; ++k) v[k] = lds128(buf + 16 * (ctid + NCT * k));
  if (RANK) {
#pragma unroll
    for (int k = 0; k < VEC_PER_THREAD; ++k)
      st.cnt2 += (bgt2(v[k].x, thr2) & 0x00010001u) + (bgt2(v[k].y, thr2) & 0x00010001u) +
                 (bgt2(v[k].z, thr2) & 0x00010001u) + (bgt2(v[k].w, thr2) & 0x00010001u);
  }
  uint32_t a[2 * VEC_PER_THREAD];
#pragma unroll
  for (int k = 0; k < VEC_PER_THREAD; ++k) {
    a[2 * k] = bmax2(v[k].x, v[k].y);
    a[2 * k + 1] = bmax2(v[k].z, v[k].w);
  }
#pragma unroll
  for (int s = VEC_PER_THREAD; s > 0; s >>= 1)
#pragma unroll
    for (int i = 0; i < s; ++i) a[i] = bmax2(a[i], a[i + s]);
  const float vm = fmaxf(bf16lo(a[0]), bf16hi(a[0]));
  if (vm > st.m) {
    const int e = first_index_of(v, vm, e_first + 8 * ctid);
    if (SOFTMAX) rescale(st, vm, c);
    st.m = vm;
    st.idx = e;
  }
  if (SOFTMAX) {
    const f32x2 c2 = pk2(c, c);
    f32x2 e[4 * VEC_PER_THREAD];
#pragma unroll
    for (int k = 0; k < VEC_PER_THREAD; ++k) {
      const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const f32x2 t = mul2(bsub2(w[q], st.m), c2);
        e[4 * k + q] = pk2(ex2(lo2(t)), ex2(hi2(t)));
      }
    }
#pragma unroll
    for (int s = 2 * VEC_PER_THREAD; s > 0; s >>= 1)
#pragma unroll
      for (int i = 0; i < s; ++i) e[i] = add2(e[i], e[i + s]);
    st.S2 = add2(st.S2, e[0]);
  }
}

// Residual mode, full tile: the stage holds SAMPLE_TILE bf16 of the target row
// (first half) and the same elements of the draft row (second half). Returns
// this thread's sum of max(0, p - q) over its 32 elements.
constexpr int RES_VPT = SAMPLE_TILE / 8 / NCT;   // vectors per thread per row
static_assert(RES_VPT * 8 * NCT == SAMPLE_TILE, "residual tiles split evenly");
static_assert(2 * SAMPLE_TILE * 2 <= TILE_BYTES, "a residual tile pair fits one stage");

struct ResLaw { float mt, invSt, md, invSd, c; };

__device__ __forceinline__ float consume_res_full(const unsigned char *buf, int ctid,
                                                  const ResLaw &L) {
  const f32x2 c2 = pk2(L.c, L.c), it2 = pk2(L.invSt, L.invSt), id2 = pk2(L.invSd, L.invSd);
  f32x2 e[4 * RES_VPT];
#pragma unroll
  for (int k = 0; k < RES_VPT; ++k) {
    const uint4 vt = lds128(buf + 16 * (ctid + NCT * k));
    const uint4 vd = lds128(buf + TILE_BYTES / 2 + 16 * (ctid + NCT * k));
    const uint32_t wt[4] = {vt.x, vt.y, vt.z, vt.w}, wd[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const f32x2 tt = mul2(bsub2(wt[q], L.mt), c2), td = mul2(bsub2(wd[q], L.md), c2);
      const f32x2 p2 = mul2(pk2(ex2(lo2(tt)), ex2(hi2(tt))), it2);
      const f32x2 q2 = mul2(pk2(ex2(lo2(td)), ex2(hi2(td))), id2);
      const f32x2 d2 = add2(p2, q2 ^ 0x8000000080000000ull);
      e[4 * k + q] = pk2(fmaxf(lo2(d2), 0.f), fmaxf(hi2(d2), 0.f));
    }
  }
#pragma unroll
  for (int s = 2 * RES_VPT; s > 0; s >>= 1)
#pragma unroll
    for (int i = 0; i < s; ++i) e[i] = add2(e[i], e[i + s]);
  return lo2(e[0]) + hi2(e[0]);
}

// Residual mode, last (partial) tile of a row: ne < SAMPLE_TILE elements.
__device__ __forceinline__ float consume_res_partial(const unsigned char *buf, int ctid, int ne,
                                                     const ResLaw &L) {
  float s = 0.f;
  for (int v = ctid; v * 8 < ne; v += NCT) {
    const uint4 vt = lds128(buf + 16 * v);
    const uint4 vd = lds128(buf + TILE_BYTES / 2 + 16 * v);
    const uint32_t wt[4] = {vt.x, vt.y, vt.z, vt.w}, wd[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (8 * v + 2 * q < ne) {
        s += fmaxf(0.f, ex2((bf16lo(wt[q]) - L.mt) * L.c) * L.invSt -
                            ex2((bf16lo(wd[q]) - L.md) * L.c) * L.invSd);
        s += fmaxf(0.f, ex2((bf16hi(wt[q]) - L.mt) * L.c) * L.invSt -
                            ex2((bf16hi(wd[q]) - L.md) * L.c) * L.invSd);
      }
    }
  }
  return s;
}

// Row pairs (KL mode): running statistics of a target row and its draft row
// over the same elements, plus A = sum 2^((zt - mt) c) (zt - zd) relative to
// the running target max: with the row totals it gives KL(p || q) ("Test-Time
// Speculation", §2 step 3) without a second read.
struct PairState {
  float mt, St, A;
  int idx, cnt;
  float md, Sd;
};

template <bool BF16, bool RANK>
__device__ __forceinline__ void consume_pair_vec(const uint4 wt, const uint4 wd, int e, float c,
                                                 PairState &ps, float thr) {
  constexpr int N = BF16 ? 8 : 4;
  float xt[N], xd[N];
  const uint32_t ut[4] = {wt.x, wt.y, wt.z, wt.w}, ud[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (BF16) {
      xt[2 * q] = bf16lo(ut[q]); xt[2 * q + 1] = bf16hi(ut[q]);
      xd[2 * q] = bf16lo(ud[q]); xd[2 * q + 1] = bf16hi(ud[q]);
    } else {
      xt[q] = __uint_as_float(ut[q]);
      xd[q] = __uint_as_float(ud[q]);
    }
  }
  float vmt = xt[0], vmd = xd[0];
#pragma unroll
  for (int k = 1; k < N; ++k) {
    vmt = fmaxf(vmt, xt[k]);
    vmd = fmaxf(vmd, xd[k]);
  }
  if (RANK) {
#pragma unroll
    for (int k = 0; k < N; ++k) ps.cnt += xt[k] > thr;
  }
  if (vmt > ps.mt) {
    int j = N - 1;
#pragma unroll
    for (int k = N - 2; k >= 0; --k)
      if (xt[k] == vmt) j = k;
    const float f = ex2((ps.mt - vmt) * c);
    ps.St *= f;
    if (!isinf(ps.A)) ps.A *= f;
    ps.mt = vmt;
    ps.idx = e + j;
  }
  if (vmd > ps.md) {
    ps.Sd *= ex2((ps.md - vmd) * c);
    ps.md = vmd;
  }
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const float et = ex2((xt[k] - ps.mt) * c);
    ps.St += et;
    ps.Sd += ex2((xd[k] - ps.md) * c);
    // zt - zd; -inf on both sides (NaN) or on the target side weighs 0
    if (et > 0.f) ps.A += et * fmaxf(xt[k] - xd[k], NO_MAX);
  }
}

// The rank count needs a few more registers than 6 CTAs per SM leave.
constexpr int RS_RANK_CTAS_PER_SM = 4;

template <bool RANK, bool PAIR>
__global__ void __launch_bounds__(RS_THREADS,
                                  RANK || PAIR ? RS_RANK_CTAS_PER_SM : RS_CTAS_PER_SM)
    k_row_pass(const RowPassArgs a) {
  extern __shared__ __align__(128) unsigned char dsmem[];
  __shared__ RowPassSmem sh;
  unsigned char *stage_buf = dsmem;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], RS_CONS_WARPS);
    }
    sh.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int *abort = &sh.abort;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane != 0) return;
    // nothing to stream once the setup rejected the inputs
    const int ipj = (a.ntiles + RES_TILES_PER_ITEM - 1) / RES_TILES_PER_ITEM;
    const long long n_items =
        a.hdr->status != SPEC_OK ? 0
        : a.residual             ? (long long)a.hdr->n_jobs_a * ipj
                                 : (long long)a.hdr->n_list * a.nch_max;
    long long it = 0;  // stages issued so far
    bool ok = true;
    unsigned int *counter = a.residual ? &a.hdr->work2 : &a.hdr->work;
    long long item = atomicAdd(counter, 1u);
    while (ok && a.residual && item < n_items) {
      const long long next = atomicAdd(counter, 1u);
      const int ja = (int)(item / ipj);
      const int g = (int)(item % ipj);
      const Job job = a.jobs[ja];
      const ReqInfo r = a.req[job.b];
      const uint64_t trow = (uint64_t)(a.base[0] + (long long)(r.t0 + job.n) * a.row_bytes[0]);
      const uint64_t drow = (uint64_t)(a.base[1] + (long long)(r.d0 + job.n) * a.row_bytes[1]);
      const int j1 = min(a.ntiles, (g + 1) * RES_TILES_PER_ITEM);
      for (int j = g * RES_TILES_PER_ITEM; j < j1; ++j) {
        const int s = (int)(it % NSTAGE);
        const long long use = it / NSTAGE;
        if (use > 0 && !mbar_wait_bounded(&sh.empty[s], (uint32_t)((use - 1) & 1), abort)) {
          ok = false;
          break;
        }
        const int e0 = j * SAMPLE_TILE;
        const int ne = min(SAMPLE_TILE, a.V - e0);
        const uint32_t nb = (uint32_t)ne * 2;
        sh.m0[s] = make_int4(ja, j, e0, ne | (1 << 14));
        sh.m1[s] = make_int4(__float_as_int(r.c), 0, 0, 0);
        mbar_arrive_tx(&sh.full[s], 2 * nb);
        unsigned char *dst = stage_buf + (size_t)s * TILE_BYTES;
        bulk_g2s(dst, (const void *)(trow + 2ull * e0), nb, &sh.full[s]);
        bulk_g2s(dst + TILE_BYTES / 2, (const void *)(drow + 2ull * e0), nb, &sh.full[s]);
        ++it;
      }
      item = next;
    }
    while (ok && !a.residual && item < n_items) {
      const long long next = atomicAdd(counter, 1u);  // one item ahead
      const int entry = (int)(item / a.nch_max);
      const int chunk = (int)(item % a.nch_max);
      const RowTask t = a.list[entry];
      const int w = t.which;
      const float thr = RANK && w != 1 && t.slot >= 0 ? a.rank_thr[t.row] : INFINITY;
      if (PAIR && w == ROW_PAIR) {
        // target row and draft row side by side: each stage holds up to
        // TILE_BYTES/2 of both (same dtype, 16-byte aligned rows)
        if (t.slot >= 0 && chunk < a.nch[0]) {
          const long long rbytes = a.row_bytes[0];
          const int esz = dtype_size(a.dtype[0]);
          const uint64_t trow = (uint64_t)(a.base[0] + (long long)t.row * rbytes);
          const uint64_t drow = (uint64_t)(a.base[1] + (long long)t.drow * rbytes);
          const uint64_t off0 = (uint64_t)chunk * a.chunk_bytes;
          const uint64_t off1 = min((uint64_t)rbytes, off0 + (uint64_t)a.chunk_bytes);
          const int ntile = (int)((off1 - off0 + TILE_BYTES / 2 - 1) / (TILE_BYTES / 2));
          for (int tl = 0; tl < ntile && ok; ++tl) {
            const int s = (int)(it % NSTAGE);
            const long long use = it / NSTAGE;
            if (use > 0 && !mbar_wait_bounded(&sh.empty[s], (uint32_t)((use - 1) & 1), abort)) {
              ok = false;
              break;
            }
            const uint64_t off = off0 + (uint64_t)tl * (TILE_BYTES / 2);
            const uint32_t nb = (uint32_t)min((uint64_t)(TILE_BYTES / 2), off1 - off);
            sh.m0[s] = make_int4(t.slot, chunk, (int)(off / esz),
                                 (int)(nb / 16) | ((tl == ntile - 1) << 12) | (1 << 15));
            sh.m1[s] = make_int4(__float_as_int(t.c), t.row, t.dslot, 0);
            if (RANK) sh.thr[s] = thr;
            mbar_arrive_tx(&sh.full[s], 2 * nb);
            unsigned char *dst = stage_buf + (size_t)s * TILE_BYTES;
            bulk_g2s(dst, (const void *)(trow + off), nb, &sh.full[s]);
            bulk_g2s(dst + TILE_BYTES / 2, (const void *)(drow + off), nb, &sh.full[s]);
            ++it;
          }
        }
        item = next;
        continue;
      }
      const long long rbytes = w ? a.row_bytes[1] : a.row_bytes[0];
      if (t.slot >= 0 && chunk < (w ? a.nch[1] : a.nch[0])) {
        const int esz = dtype_size(w ? a.dtype[1] : a.dtype[0]);
        const uint64_t row0 = (uint64_t)((w ? a.base[1] : a.base[0]) + (long long)t.row * rbytes);
        const uint64_t cb0 = row0 + (uint64_t)chunk * a.chunk_bytes;
        const uint64_t cb1 = min(row0 + (uint64_t)rbytes, cb0 + (uint64_t)a.chunk_bytes);
        uint64_t A0 = (cb0 + 15) & ~15ull, A1 = cb1 & ~15ull;
        if (A1 <= A0) A0 = A1 = cb1;  // no aligned interior: all scalar
        const int ntile = A1 > A0 ? (int)((A1 - A0 + TILE_BYTES - 1) / TILE_BYTES) : 1;
        const int head_n = (int)((A0 - cb0) / esz), tail_n = (int)((cb1 - A1) / esz);
        for (int tl = 0; tl < ntile; ++tl) {
          const int s = (int)(it % NSTAGE);
          const long long use = it / NSTAGE;
          if (use > 0 && !mbar_wait_bounded(&sh.empty[s], (uint32_t)((use - 1) & 1), abort)) {
            ok = false;
            break;
          }
          const uint64_t off = A0 + (uint64_t)tl * TILE_BYTES;
          const uint32_t nb = (uint32_t)min((uint64_t)TILE_BYTES, A1 - off);
          const int flags = (int)(nb / 16) | ((tl == ntile - 1) << 12) | (w << 13) |
                            (head_n << 16) | (tail_n << 20);
          sh.m0[s] = make_int4(t.slot, chunk, (int)((off - row0) / esz), flags);
          sh.m1[s] = make_int4(__float_as_int(t.c), t.row, (int)((cb0 - row0) / esz),
                               (int)((A1 - row0) / esz));
          if (RANK) sh.thr[s] = thr;
          if (nb > 0) {
            mbar_arrive_tx(&sh.full[s], nb);
            bulk_g2s(stage_buf + (size_t)s * TILE_BYTES, (const void *)off, nb, &sh.full[s]);
          } else {
            mbar_arrive(&sh.full[s]);
          }
          ++it;
        }
      }
      item = next;
    }
    if (ok) {  // end marker
      const int s = (int)(it % NSTAGE);
      const long long use = it / NSTAGE;
      if (use == 0 || mbar_wait_bounded(&sh.empty[s], (uint32_t)((use - 1) & 1), abort)) {
        sh.m0[s] = make_int4(-1, 0, 0, 0);
        mbar_arrive(&sh.full[s]);
        return;
      }
    }
    // gave up: record it, then wait (bounded) for this CTA's copies in flight
    set_status(a.hdr, SPEC_ERR_TIMEOUT, -2);
    *abort = 1;
    for (int s = 0; s < NSTAGE; ++s) {
      const long long issued = (it - s + NSTAGE - 1) / NSTAGE;  // uses of stage s
      if (issued > 0) {
        volatile int never = 0;
        mbar_wait_bounded(&sh.full[s], (uint32_t)((issued - 1) & 1), &never);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1;
  const int ctid = threadIdx.x - 32;
  RunState st{NO_MAX, pk2(0.f, 0.f), 0x7fffffff, 0, 0u};
  PairState ps{NO_MAX, 0.f, 0.f, 0x7fffffff, 0, NO_MAX, 0.f};
  int res_job = -1;
  ResLaw res_law{0.f, 0.f, 0.f, 0.f, 0.f};
  for (long long it = 0;; ++it) {
    const int s = (int)(it % NSTAGE);
    if (!mbar_wait_bounded(&sh.full[s], (uint32_t)((it / NSTAGE) & 1), abort)) {
      set_status(a.hdr, SPEC_ERR_TIMEOUT, -3);
      *abort = 1;
      return;
    }
    const int4 m0 = sh.m0[s];
    if (m0.x < 0) return;
    const int4 m1 = sh.m1[s];
    if (m0.w & (1 << 14)) {   // residual tile pair
      const int ja = m0.x, j = m0.y, ne = m0.w & 0x3fff;
      if (ja != res_job) {
        const Job job = a.jobs[ja];
        res_law = ResLaw{job.mt, 1.f / job.St, job.md, job.Sd > 0.f ? 1.f / job.Sd : 0.f,
                         __int_as_float(m1.x)};
        res_job = ja;
      }
      const unsigned char *rbuf = stage_buf + (size_t)s * TILE_BYTES;
      float rs = ne == SAMPLE_TILE ? consume_res_full(rbuf, ctid, res_law)
                                   : consume_res_partial(rbuf, ctid, ne, res_law);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[s]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
      if (lane == 0) a.tsum4[((long long)ja * a.ntiles + j) * RS_CONS_WARPS + cw] = rs;
      continue;
    }
    if (PAIR && (m0.w & (1 << 15))) {   // target row + draft row
      const int nvp = m0.w & 0xfff;
      const float c = __int_as_float(m1.x);
      const float thr = RANK ? sh.thr[s] : INFINITY;
      const unsigned char *buf = stage_buf + (size_t)s * TILE_BYTES;
      if (a.dtype[0] == SPEC_BF16) {
        for (int v = ctid; v < nvp; v += NCT)
          consume_pair_vec<true, RANK>(lds128(buf + 16 * v), lds128(buf + TILE_BYTES / 2 + 16 * v),
                                       m0.z + 8 * v, c, ps, thr);
      } else {
        for (int v = ctid; v < nvp; v += NCT)
          consume_pair_vec<false, RANK>(lds128(buf + 16 * v), lds128(buf + TILE_BYTES / 2 + 16 * v),
                                        m0.z + 4 * v, c, ps, thr);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.empty[s]);
      if ((m0.w >> 12) & 1) {   // end of the chunk: merge the warp, write both rows
        float m = ps.mt, S = ps.St, A = ps.A, md = ps.md, Sd = ps.Sd;
        int idx = ps.idx, cnt = ps.cnt, nid = 0x7fffffff;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
          const float S2 = __shfl_xor_sync(0xffffffffu, S, o);
          const float A2 = __shfl_xor_sync(0xffffffffu, A, o);
          const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
          merge_stat_a(m, S, idx, A, m2, S2, i2, A2, c);
          const float md2 = __shfl_xor_sync(0xffffffffu, md, o);
          const float Sd2 = __shfl_xor_sync(0xffffffffu, Sd, o);
          merge_stat(md, Sd, nid, md2, Sd2, 0x7fffffff, c);
          cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        }
        if (lane == 0) {
          const long long k = ((long long)m0.x * a.nch_max + m0.y) * RS_CONS_WARPS + cw;
          a.part[k] = Part{m, S, idx, cnt};
          a.part[((long long)m1.z * a.nch_max + m0.y) * RS_CONS_WARPS + cw] =
              Part{md, Sd, 0x7fffffff, 0};
          a.kl_part[k] = A;
        }
        ps = PairState{NO_MAX, 0.f, 0.f, 0x7fffffff, 0, NO_MAX, 0.f};
      }
      continue;
    }
    const int nvec = m0.w & 0xfff;
    const bool last = (m0.w >> 12) & 1;
    const int which = (m0.w >> 13) & 1;
    const int e_first = m0.z;
    const float c = __int_as_float(m1.x);
    const int dt = which ? a.dtype[1] : a.dtype[0];
    const bool bf16 = dt == SPEC_BF16;
    const unsigned char *buf = stage_buf + (size_t)s * TILE_BYTES;
    // rank threshold; +inf counts nothing (logits are finite or -inf)
    const float thr = RANK ? sh.thr[s] : INFINITY;
    if (bf16 && nvec == FULL_NVEC) {
      if (RANK && thr != INFINITY) {
        const uint32_t h = __float_as_uint(thr) >> 16;   // exact: a bf16 logit
        const uint32_t thr2 = h | (h << 16);
        if (c != 0.f) consume_full_bf16<true, true>(buf, ctid, e_first, c, st, thr2);
        else consume_full_bf16<false, true>(buf, ctid, e_first, c, st, thr2);
      } else {
        if (c != 0.f) consume_full_bf16<true, false>(buf, ctid, e_first, c, st, 0u);
        else consume_full_bf16<false, false>(buf, ctid, e_first, c, st, 0u);
      }
    } else if (bf16) {
      for (int v = ctid; v < nvec; v += NCT) {
        if (c != 0.f) consume_vec<true, true>(lds128(buf + 16 * v), e_first + 8 * v, c, st, thr);
        else consume_vec<false, true>(lds128(buf + 16 * v), e_first + 8 * v, c, st, thr);
      }
    } else {
      for (int v = ctid; v < nvec; v += NCT) {
        if (c != 0.f) consume_vec<true, false>(lds128(buf + 16 * v), e_first + 4 * v, c, st, thr);
        else consume_vec<false, false>(lds128(buf + 16 * v), e_first + 4 * v, c, st, thr);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
    if (last) {
      if (cw == 0) {  // unaligned head / tail elements of the chunk
        const int head_n = (m0.w >> 16) & 0xf, tail_n = (m0.w >> 20) & 0xf;
        const char *row = (which ? a.base[1] : a.base[0]) +
                          (long long)m1.y * (which ? a.row_bytes[1] : a.row_bytes[0]);
        if (lane < head_n)
          scalar_update(load_elem(row, dt, m1.z + lane), m1.z + lane, c, st, thr);
        if (lane >= 16 && lane - 16 < tail_n)
          scalar_update(load_elem(row, dt, m1.w + lane - 16), m1.w + lane - 16, c, st, thr);
      }
      float m = st.m, S = lo2(st.S2) + hi2(st.S2);
      int idx = st.idx;
      int cnt = RANK ? st.cnt + (int)(st.cnt2 & 0xffffu) + (int)(st.cnt2 >> 16) : 0;
      if (RANK) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float S2 = __shfl_xor_sync(0xffffffffu, S, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
        merge_stat(m, S, idx, m2, S2, i2, c);
      }
      if (lane == 0) {
        Part p;
        p.m = m;
        p.S = S;
        p.idx = idx;
        p.cnt = cnt;
        a.part[((long long)m0.x * a.nch_max + m0.y) * RS_CONS_WARPS + cw] = p;
      }
      st = RunState{NO_MAX, pk2(0.f, 0.f), 0x7fffffff, 0, 0u};
    }
  }
}

int nchunks(int V, int dtype, int chunk_bytes) {
  const long long bytes = (long long)V * (dtype == SPEC_BF16 ? 2 : 4);
  return (int)((bytes + chunk_bytes - 1) / chunk_bytes);
}

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev < 0 || dev >= 64) return -1;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    cached[dev] = n;
  }
  return cached[dev];
}

static thread_local cudaEvent_t prof_before = nullptr, prof_after = nullptr;

void set_row_pass_events(cudaEvent_t before, cudaEvent_t after) {
  prof_before = before;
  prof_after = after;
}

void take_row_pass_events(cudaEvent_t *before, cudaEvent_t *after) {
  *before = prof_before;
  *after = prof_after;
  prof_before = prof_after = nullptr;
}

int launch_row_pass(const RowPassArgs &a, cudaStream_t stream) {
  const int sms = num_sms();
  if (sms <= 0) return SPEC_ERR_CUDA;
  const size_t smem = (size_t)NSTAGE * TILE_BYTES;
  const bool rank = a.rank_thr != nullptr && !a.residual;
  const bool pair = a.kl_part != nullptr && !a.residual;
  auto kern = rank ? (pair ? k_row_pass<true, true> : k_row_pass<true, false>)
                   : (pair ? k_row_pass<false, true> : k_row_pass<false, false>);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return SPEC_ERR_CUDA;
  cudaEvent_t before = prof_before, after = prof_after;
  prof_before = prof_after = nullptr;
  if (before && cudaEventRecord(before, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  kern<<<(rank || pair ? RS_RANK_CTAS_PER_SM : RS_CTAS_PER_SM) * sms, RS_THREADS, smem,
         stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (after && cudaEventRecord(after, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

bool aligned(const void *p, size_t al) { return ((uintptr_t)p % al) == 0; }

}  // namespace sv
