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
// Design: a persistent grid of RS_CTAS_PER_SM CTAs per SM. Warp 0 lane 0 is
// the producer: it takes work items (row, CHUNK_BYTES chunk) from a global
// counter and streams each chunk into a ring of NSTAGE 16 KB shared-memory
// stages with 1-D TMA bulk copies, completion tracked by mbarriers. The
// RS_CONS_WARPS consumer warps read the stages with 128-bit shared loads; one
// 2^x (MUFU) per element for softmax rows, none for argmax-only rows. No
// cross-warp barrier: each consumer warp writes its own partial. Every wait is
// bounded; on expiry the status word gets SPEC_ERR_TIMEOUT and the CTA drains
// its own copies and returns.
#include "common.cuh"
#include "internal.h"
#include "rowpass.cuh"

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
      const Job job = GLD(a.jobs + (ja));
      const ReqInfo r = GLD(a.req + (job.b));
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
      const RowTask t = GLD(a.list + (entry));
      const int w = t.which;
      const float thr = RANK && w != 1 && t.slot >= 0 ? GLD(a.rank_thr + (t.row)) : INFINITY;
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
        const Job job = GLD(a.jobs + (ja));
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
      if (lane == 0) GST(a.tsum4 + (((long long)ja * a.ntiles + j) * RS_CONS_WARPS + cw), rs);
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
          GST(a.part + (k), Part{m, S, idx, cnt});
          GST(a.part + (((long long)m1.z * a.nch_max + m0.y) * RS_CONS_WARPS + cw), Part{md, Sd, 0x7fffffff, 0});
          GST(a.kl_part + (k), A);
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
    consume_row_stage<RANK>(buf, nvec, e_first, c, bf16, thr, ctid, st);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
    if (last) {
      if (cw == 0) {  // unaligned head / tail elements of the chunk
        const char *row = (which ? a.base[1] : a.base[0]) +
                          (long long)m1.y * (which ? a.row_bytes[1] : a.row_bytes[0]);
        consume_head_tail(row, dt, m0.w, m1.z, m1.w, c, thr, lane, st);
      }
      const Part p = finish_row_chunk<RANK>(st, c);
      if (lane == 0) GST(a.part + (((long long)m0.x * a.nch_max + m0.y) * RS_CONS_WARPS + cw), p);
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

bool row_pass_events_pending() { return prof_before != nullptr || prof_after != nullptr; }

int launch_row_pass(const RowPassArgs &a, cudaStream_t stream) {
  if (check_upload(stream) != SPEC_OK) return SPEC_ERR_CUDA;
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
