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

struct StageMeta {
  int slot;     // -1: no more work
  int chunk;
  int last;     // last stage of the chunk
  int which;    // 0 target, 1 draft
  int row;
  int e_first;  // element index of the first vector element in the stage
  int nvec;     // 16-byte vectors in the stage
  float c;
  int head_e, head_n, tail_e, tail_n;  // scalar elements (last stage only)
  int pad;
};

struct RowPassSmem {
  uint64_t full[NSTAGE];
  uint64_t empty[NSTAGE];
  StageMeta meta[NSTAGE];
  int abort;
};

__device__ __forceinline__ void scalar_update(float x, int e, float c, float &m, float &S,
                                              int &idx) {
  if (x > m) {
    if (c != 0.f) S *= ex2((m - x) * c);
    m = x;
    idx = e;
  } else if (x == m && e < idx) {
    idx = e;
  }
  if (c != 0.f && m != -INFINITY) S += ex2((x - m) * c);
}

template <bool SOFTMAX>
__device__ __forceinline__ void consume_bf16(const uint4 w, int e, float c, float &m, float &S,
                                             int &idx) {
  float x[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
  const float vm = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])),
                         fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
  if (vm > m) {  // rare after the first few vectors
    int j = 7;
#pragma unroll
    for (int k = 6; k >= 0; --k)
      if (x[k] == vm) j = k;
    if (SOFTMAX) S *= ex2((m - vm) * c);
    m = vm;
    idx = e + j;
  }
  if (SOFTMAX && m != -INFINITY) {
    float t[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = ex2((x[k] - m) * c);
    S += ((t[0] + t[1]) + (t[2] + t[3])) + ((t[4] + t[5]) + (t[6] + t[7]));
  }
}

template <bool SOFTMAX>
__device__ __forceinline__ void consume_f32(const uint4 w, int e, float c, float &m, float &S,
                                            int &idx) {
  float x[4] = {__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                __uint_as_float(w.w)};
  const float vm = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  if (vm > m) {
    int j = 3;
#pragma unroll
    for (int k = 2; k >= 0; --k)
      if (x[k] == vm) j = k;
    if (SOFTMAX) S *= ex2((m - vm) * c);
    m = vm;
    idx = e + j;
  }
  if (SOFTMAX && m != -INFINITY) {
    float t[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) t[k] = ex2((x[k] - m) * c);
    S += (t[0] + t[1]) + (t[2] + t[3]);
  }
}

__global__ void __launch_bounds__(RS_THREADS, 2) k_row_pass(const RowPassArgs a) {
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
    const long long n_items = (long long)a.hdr->n_list * a.nch_max;
    long long it = 0;  // stages issued so far
    bool ok = true;
    long long item = atomicAdd(&a.hdr->work, 1u);
    while (ok && item < n_items) {
      const long long next = atomicAdd(&a.hdr->work, 1u);  // one item ahead
      const int entry = (int)(item / a.nch_max);
      const int chunk = (int)(item % a.nch_max);
      const RowTask t = a.list[entry];
      const int w = t.which;
      if (chunk < a.nch[w]) {
        const int esz = dtype_size(a.dtype[w]);
        const uint64_t row0 = (uint64_t)(a.base[w] + (long long)t.row * a.row_bytes[w]);
        const uint64_t cb0 = row0 + (uint64_t)chunk * CHUNK_BYTES;
        const uint64_t cb1 = min(row0 + (uint64_t)a.row_bytes[w], cb0 + CHUNK_BYTES);
        uint64_t A0 = (cb0 + 15) & ~15ull, A1 = cb1 & ~15ull;
        if (A1 <= A0) A0 = A1 = cb1;  // no aligned interior: all scalar
        const int ntile = A1 > A0 ? (int)((A1 - A0 + TILE_BYTES - 1) / TILE_BYTES) : 1;
        for (int tl = 0; tl < ntile; ++tl) {
          const int s = (int)(it % NSTAGE);
          const long long use = it / NSTAGE;
          if (use > 0 && !mbar_wait_bounded(&sh.empty[s], (uint32_t)((use - 1) & 1), abort)) {
            ok = false;
            break;
          }
          const uint64_t off = A0 + (uint64_t)tl * TILE_BYTES;
          const uint32_t nb = (uint32_t)min((uint64_t)TILE_BYTES, A1 - off);
          StageMeta &md = sh.meta[s];
          md.slot = t.slot;
          md.chunk = chunk;
          md.last = tl == ntile - 1;
          md.which = w;
          md.row = t.row;
          md.e_first = (int)((off - row0) / esz);
          md.nvec = (int)(nb / 16);
          md.c = t.c;
          md.head_e = (int)((cb0 - row0) / esz);
          md.head_n = (int)((A0 - cb0) / esz);
          md.tail_e = (int)((A1 - row0) / esz);
          md.tail_n = (int)((cb1 - A1) / esz);
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
        sh.meta[s].slot = -1;
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
  constexpr int NCT = RS_CONS_WARPS * 32;
  float m = -INFINITY, S = 0.f;
  int idx = 0x7fffffff;
  for (long long it = 0;; ++it) {
    const int s = (int)(it % NSTAGE);
    if (!mbar_wait_bounded(&sh.full[s], (uint32_t)((it / NSTAGE) & 1), abort)) {
      set_status(a.hdr, SPEC_ERR_TIMEOUT, -3);
      *abort = 1;
      return;
    }
    const StageMeta md = sh.meta[s];
    if (md.slot < 0) return;
    const unsigned char *buf = stage_buf + (size_t)s * TILE_BYTES;
    const float c = md.c;
    if (a.dtype[md.which] == SPEC_BF16) {
      if (c != 0.f) {
        for (int v = ctid; v < md.nvec; v += NCT)
          consume_bf16<true>(lds128(buf + 16 * v), md.e_first + 8 * v, c, m, S, idx);
      } else {
        for (int v = ctid; v < md.nvec; v += NCT)
          consume_bf16<false>(lds128(buf + 16 * v), md.e_first + 8 * v, c, m, S, idx);
      }
    } else {
      if (c != 0.f) {
        for (int v = ctid; v < md.nvec; v += NCT)
          consume_f32<true>(lds128(buf + 16 * v), md.e_first + 4 * v, c, m, S, idx);
      } else {
        for (int v = ctid; v < md.nvec; v += NCT)
          consume_f32<false>(lds128(buf + 16 * v), md.e_first + 4 * v, c, m, S, idx);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);
    if (md.last) {
      if (cw == 0) {  // unaligned head / tail elements of the chunk
        const char *row = a.base[md.which] + (long long)md.row * a.row_bytes[md.which];
        const int dt = a.dtype[md.which];
        if (lane < md.head_n)
          scalar_update(load_elem(row, dt, md.head_e + lane), md.head_e + lane, c, m, S, idx);
        if (lane >= 16 && lane - 16 < md.tail_n)
          scalar_update(load_elem(row, dt, md.tail_e + lane - 16), md.tail_e + lane - 16, c, m,
                        S, idx);
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
        p.pad = 0;
        a.part[((long long)md.slot * a.nch_max + md.chunk) * RS_CONS_WARPS + cw] = p;
      }
      m = -INFINITY;
      S = 0.f;
      idx = 0x7fffffff;
    }
  }
}

int nchunks(int V, int dtype) {
  const long long bytes = (long long)V * (dtype == SPEC_BF16 ? 2 : 4);
  return (int)((bytes + CHUNK_BYTES - 1) / CHUNK_BYTES);
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

int launch_row_pass(const RowPassArgs &a, cudaStream_t stream) {
  const int sms = num_sms();
  if (sms <= 0) return SPEC_ERR_CUDA;
  const size_t smem = (size_t)NSTAGE * TILE_BYTES;
  if (cudaFuncSetAttribute(k_row_pass, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return SPEC_ERR_CUDA;
  cudaEvent_t before = prof_before, after = prof_after;
  prof_before = prof_after = nullptr;
  if (before && cudaEventRecord(before, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  k_row_pass<<<2 * sms, RS_THREADS, smem, stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (after && cudaEventRecord(after, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

bool aligned(const void *p, size_t al) { return ((uintptr_t)p % al) == 0; }

}  // namespace sv
