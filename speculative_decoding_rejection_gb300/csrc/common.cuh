// Shared device helpers of the verifier kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "specverify.h"

namespace sv {

// ---------------------------------------------------------------- tiling
constexpr int TILE_BYTES = 16384;   // one TMA bulk copy = one pipeline stage
// Position-lazy rounds stream few rows each: finer chunks spread them over
// more CTAs.
constexpr int LAZY_CHUNK_BYTES = 32768;
constexpr int CHUNK_BYTES = 131072; // one unit of dynamic work in the row pass
// The streaming verifier's unit of work: one completion count per chunk.
constexpr int STREAM_CHUNK_BYTES = 131072;
// Row pass shape, chosen by measurement on GB300: six CTAs per SM, each one
// producer lane and four consumer warps over a two-stage ring of 16 KB TMA
// copies (192 KB of copies in flight per SM); a consumer thread takes eight
// 16-byte vectors (64 bf16) per stage, enough independent work to keep the
// exponent pipe fed.
constexpr int NSTAGE = 2;           // pipeline depth per CTA
constexpr int RS_CONS_WARPS = 4;    // consumer warps of the row pass
constexpr int RS_CTAS_PER_SM = 6;   // resident row-pass CTAs per SM
constexpr int RS_THREADS = 32 * (1 + RS_CONS_WARPS);
constexpr int SAMPLE_THREADS = 256;
constexpr int SAMPLE_EPT = 16;      // contiguous elements per thread per tile
constexpr int SAMPLE_TILE = SAMPLE_THREADS * SAMPLE_EPT;
constexpr int MAX_SAMPLE_TILES = (SPEC_MAX_V + SAMPLE_TILE - 1) / SAMPLE_TILE;
constexpr int RES_TILES_PER_ITEM = 4;   // residual tiles per row-pass work item

constexpr float LOG2E = 1.4426950408889634f;
constexpr unsigned long long WAIT_NS = 2000000000ull;  // bounded waits: 2 s

enum ReqMode : int { MODE_SKIP = 0, MODE_GREEDY = 1, MODE_SAMPLE = 2 };

// ------------------------------------------------------ workspace records
struct WsHeader {        // first 256 bytes of every workspace
  int status;            // device-side spec_status (0 = OK)
  int detail;            // first offending request / row, -1 if none
  unsigned int work;     // dynamic work counter of the row pass
  int n_list;            // rows in the row-pass list
  int n_jobs_a;          // final draws over full residual rows (dense drafts)
  int n_jobs_b;          // final draws located from chunk statistics
  unsigned int work2;    // dynamic work counter of the residual tile sums
  int n_done;            // streaming verifier: requests whose final token is written
  unsigned long long work_s;   // streaming verifier: tickets of the static entries
  unsigned long long work_d;   // streaming verifier: tickets of the dynamic entries
  int n_alloc_d;         // streaming verifier: dynamic entries allocated
  int setup_bad;         // streaming verifier: the setup rejected a request
  int pad[50];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// ------------------------------------------------------- checked build
// Built with SPEC_CHECKED (libspecverify_checked.so), every global access
// of the kernels goes through the accessors below, which check it against
// the byte ranges of the buffers of the call being run (its inputs,
// outputs and workspace). An access outside them is skipped (a load gives
// zero, a store or a copy is dropped, a skipped bulk copy still completes
// its barrier's transaction) and reported in the status word as
// SPEC_ERR_BOUNDS with the source line of the access as detail; nothing
// traps. The entry point lists the call's ranges (check_begin, check_add)
// and every launcher copies the list to its translation unit's device copy
// before its kernels (check_upload). Without SPEC_CHECKED the accessors are
// the plain accesses.
constexpr int CHECK_RANGES = 24;
struct CheckTable {
  int n;
  WsHeader *hdr;                           // the call's status word
  unsigned long long lo[CHECK_RANGES];     // byte ranges [lo, hi)
  unsigned long long hi[CHECK_RANGES];
};
#ifdef SPEC_CHECKED
static __device__ CheckTable g_check;   // this translation unit's copy
static __device__ __noinline__ bool gchk_slow(unsigned long long lo, unsigned long long hi, int line) {
  for (int i = 0; i < g_check.n; ++i)
    if (lo >= g_check.lo[i] && hi <= g_check.hi[i]) return true;
  WsHeader *h = g_check.hdr;
  if (h != nullptr && atomicCAS(&h->status, 0, SPEC_ERR_BOUNDS) == 0) atomicExch(&h->detail, line);
  return false;
}
__device__ __forceinline__ bool gchk(const void *p, unsigned long long bytes, int line) {
  const unsigned long long lo = (unsigned long long)p;
  return gchk_slow(lo, lo + bytes, line);
}
#else
__device__ __forceinline__ bool gchk(const void *, unsigned long long, int) { return true; }
#endif
// Checked global accesses: plain load, non-coherent load, L2-only load,
// store, and a range test for atomics and copies.
template <class T>
__device__ __forceinline__ T gld(const T *p, int line) {
  return gchk(p, sizeof(T), line) ? *p : T{};
}
template <class T>
__device__ __forceinline__ T gldg(const T *p, int line) {
  return gchk(p, sizeof(T), line) ? __ldg(p) : T{};
}
template <class T>
__device__ __forceinline__ T gldcg(const T *p, int line) {
  return gchk(p, sizeof(T), line) ? __ldcg(p) : T{};
}
template <class T, class U>
__device__ __forceinline__ void gst(T *p, const U &v, int line) {
  if (gchk(p, sizeof(T), line)) *p = v;
}
#ifdef SPEC_CHECKED
CheckTable &host_check_table();   // the list of the call being set up (this host thread)
void check_begin(WsHeader *hdr);
void check_add(const void *p, unsigned long long bytes);
// This translation unit's device copy of the list, before its kernels.
static inline int check_upload(cudaStream_t st) {
  return cudaMemcpyToSymbolAsync(g_check, &host_check_table(), sizeof(CheckTable), 0,
                                 cudaMemcpyHostToDevice, st) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}
// A device int (the row count cu[B] that sizes a call's buffers), read
// synchronously: the checked build is a test build.
int check_read_int(const int32_t *dev, cudaStream_t st, int *out);
#else
static inline int check_upload(cudaStream_t) { return SPEC_OK; }
static inline void check_begin(WsHeader *) {}
static inline void check_add(const void *, unsigned long long) {}
#endif
#define GLD(p) ::sv::gld((p), __LINE__)
#define GLDG(p) ::sv::gldg((p), __LINE__)
#define GLDCG(p) ::sv::gldcg((p), __LINE__)
#define GST(p, ...) ::sv::gst((p), (__VA_ARGS__), __LINE__)
#define GCHK(p, n) ::sv::gchk((p), (n), __LINE__)

struct RowTask {         // one row (or row pair) streamed by the row pass
  int slot;              // index into the partial-statistics array
  int row;               // row index within its tensor
  int which;             // 0 = target tensor, 1 = draft tensor, 2 = target
                         // row paired with draft row `drow`
  float c;               // log2(e)/T, 0 for argmax-only rows
  int dslot, drow;       // pairs: the draft row's slot and index
  int pad[2];
};
constexpr int ROW_PAIR = 2;

struct Part {            // statistics of one chunk of one row
  float m;               // max logit
  float S;               // sum of 2^((z - m) c)
  int idx;               // lowest index attaining m
  int cnt;               // logits above the rank threshold (rank count only)
};

struct ReqInfo {         // per request, written by the setup kernel
  int t0;                // first target row
  int d0;                // first draft row
  int K;                 // number of drafts
  int mode;              // ReqMode
  float c;               // log2(e)/T
  int n;                 // accepted drafts (written by the accept kernel)
  int pad[2];
};

struct Job {         // one final draw of a sampling request (accept kernel)
  int b;             // request
  int n;             // accepted drafts
  int kind;          // 1: residual after a rejection, 2: bonus
  int pad;
  float mt, St;      // statistics of target row n+1
  float md, Sd;      // statistics of draft row n+1 (dense logits only)
};

struct RowStat { float m, S; int idx; };

// A chunk partial read through L2 only: in the streaming verifier it was
// written by another CTA of the same running kernel.
__device__ __forceinline__ Part ldcg_part(const Part *p) {
  const int4 v = GLDCG(reinterpret_cast<const int4 *>(p));
  return Part{__int_as_float(v.x), __int_as_float(v.y), v.z, v.w};
}

// Running maximum before any element: finite, so (x - m) never forms inf - inf.
// A row whose statistics keep this value holds no finite logit.
constexpr float NO_MAX = -3.402823466e38f;
__device__ __forceinline__ bool row_empty(float m) { return !(m > NO_MAX); }

// --------------------------------------------------------------- status
__device__ __forceinline__ void set_status(WsHeader *h, int code, int detail) {
  if (atomicCAS(&h->status, 0, code) == 0) atomicExch(&h->detail, detail);
}


// ------------------------------------------------------ counter uniforms
// SplitMix64 output function (Steele, Lea & Flood 2014) of x + gamma.
__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// u = top 24 bits of splitmix64(seed ^ splitmix64(key)) * 2^-24, exact in f32.
__device__ __forceinline__ float uniform24(uint64_t seed, uint32_t b,
                                           uint32_t pos, uint32_t stream) {
  const uint64_t key = ((uint64_t)b << 32) | ((uint64_t)pos << 8) | stream;
  const uint64_t h = splitmix64(seed ^ splitmix64(key));
  return (float)(uint32_t)(h >> 40) * 5.9604644775390625e-8f;
}

// --------------------------------------------------------------- math
__device__ __forceinline__ float ex2(float x) {   // MUFU 2^x
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Packed fp32 pairs (Blackwell f32x2 arithmetic) and packed bf16 helpers.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk2(float lo, float hi) {
  return ((f32x2)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float lo2(f32x2 v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi2(f32x2 v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// (lo(w) - m, hi(w) - m) for a packed bf16 pair w, exact for bf16 inputs
// (mixed-precision subtract: the bf16 operand is widened by the instruction).
__device__ __forceinline__ f32x2 bsub2(uint32_t w, float m) {
  float lo, hi;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "sub.rn.f32.bf16 %0, l, %3;\n\tsub.rn.f32.bf16 %1, h, %3;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(w), "f"(m));
  return pk2(lo, hi);
}
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// Packed a > b on two bf16 lanes: each 16-bit half is 0xffff where true.
__device__ __forceinline__ uint32_t bgt2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("set.gt.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ float load_elem(const void *row, int dtype, long long i) {
  if (dtype == SPEC_BF16) {
    const uint16_t v = GLDG(reinterpret_cast<const unsigned short *>(row) + i);
    return __uint_as_float((uint32_t)v << 16);
  }
  return GLDG(reinterpret_cast<const float *>(row) + i);
}

__device__ __forceinline__ int dtype_size(int dtype) { return dtype == SPEC_BF16 ? 2 : 4; }

// Merge (m, S, idx) statistics: m the max, S sum of 2^((z-m)c), idx the
// lowest index attaining the max.
__device__ __forceinline__ void merge_stat(float &m, float &S, int &idx, float m2,
                                           float S2, int i2, float c) {
  const float M = fmaxf(m, m2);
  float s = 0.f;
  if (m != -INFINITY) s += S * ex2((m - M) * c);
  if (m2 != -INFINITY) s += S2 * ex2((m2 - M) * c);
  if (m2 > m || (m2 == m && i2 < idx)) idx = i2;
  m = M;
  S = s;
}

// merge_stat that also carries A = sum 2^((z - m) c) * w, rescaled with S
// (an infinite A stays infinite).
__device__ __forceinline__ void merge_stat_a(float &m, float &S, int &idx, float &A, float m2,
                                             float S2, int i2, float A2, float c) {
  const float M = fmaxf(m, m2);
  const float f1 = ex2((m - M) * c), f2 = ex2((m2 - M) * c);
  const float a1 = isinf(A) ? A : A * f1, a2 = isinf(A2) ? A2 : A2 * f2;
  S = S * f1 + S2 * f2;
  A = a1 + a2;
  if (m2 > m || (m2 == m && i2 < idx)) idx = i2;
  m = M;
}

__device__ __forceinline__ RowStat combine_parts(const Part *p, int n, float c) {
  RowStat r{NO_MAX, 0.f, 0x7fffffff};
  for (int i = 0; i < n; ++i) merge_stat(r.m, r.S, r.idx, p[i].m, p[i].S, p[i].idx, c);
  return r;
}

// Row statistics combined by the whole warp: lane l merges partials
// l, l+32, ..., then a butterfly merges the lanes (every lane gets the row's
// statistics; the merge order is fixed, so the result is deterministic).
__device__ __forceinline__ RowStat warp_row_stat(const Part *p, int n, float c, int lane) {
  float m = NO_MAX, S = 0.f;
  int idx = 0x7fffffff;
  for (int i = lane; i < n; i += 32) {
    const Part q = ldcg_part(p + i);
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

// Load SAMPLE_EPT consecutive elements [x0, x0+EPT) of a row; `fill` beyond V.
__device__ __forceinline__ void load_ept(const char *row, int dt, bool vec_ok, int x0, int V,
                                         float fill, float *z) {
  if (vec_ok && x0 + SAMPLE_EPT <= V) {
    if (dt == SPEC_BF16) {
      const uint4 *p = reinterpret_cast<const uint4 *>(row + 2LL * x0);
#pragma unroll
      for (int q = 0; q < SAMPLE_EPT / 8; ++q) {
        const uint4 w = GLDG(p + q);
        z[8 * q + 0] = bf16lo(w.x); z[8 * q + 1] = bf16hi(w.x);
        z[8 * q + 2] = bf16lo(w.y); z[8 * q + 3] = bf16hi(w.y);
        z[8 * q + 4] = bf16lo(w.z); z[8 * q + 5] = bf16hi(w.z);
        z[8 * q + 6] = bf16lo(w.w); z[8 * q + 7] = bf16hi(w.w);
      }
    } else {
      const uint4 *p = reinterpret_cast<const uint4 *>(row + 4LL * x0);
#pragma unroll
      for (int q = 0; q < SAMPLE_EPT / 4; ++q) {
        const uint4 w = GLDG(p + q);
        z[4 * q + 0] = __uint_as_float(w.x); z[4 * q + 1] = __uint_as_float(w.y);
        z[4 * q + 2] = __uint_as_float(w.z); z[4 * q + 3] = __uint_as_float(w.w);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k)
      z[k] = x0 + k < V ? load_elem(row, dt, x0 + k) : fill;
  }
}

// ----------------------------------------------------- block primitives
// Exclusive prefix sum of one float per thread over the block; returns the
// exclusive value, *total gets the block total (= excl of the last thread +
// its value). `scratch` holds 33 floats. Ends with the block synchronised.
__device__ __forceinline__ float block_excl_scan(float v, float *scratch, float *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  float x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    float w = lane < nw ? scratch[lane] : 0.f;
    float s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    scratch[lane] = s - w;   // exclusive offset of each warp
  }
  __syncthreads();
  float xe = __shfl_up_sync(0xffffffffu, x, 1);   // exact in-warp exclusive
  if (lane == 0) xe = 0.f;
  const float excl = scratch[warp] + xe;
  if (threadIdx.x == blockDim.x - 1) scratch[32] = excl + v;
  __syncthreads();
  *total = scratch[32];
  __syncthreads();
  return excl;
}

__device__ __forceinline__ int block_excl_scan_int(int v, int *scratch, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? scratch[lane] : 0;
    int s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    scratch[lane] = s - w;
    if (lane == 31) scratch[32] = s;
  }
  __syncthreads();
  const int excl = scratch[warp] + (x - v);
  *total = scratch[32];
  __syncthreads();
  return excl;
}

// ------------------------------------------------- mbarrier / bulk copies
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for the phase of `bar` with `parity` to complete, giving up after
// limit_ns of %globaltimer or once *abort is set. Returns false when it gave
// up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  volatile int *abort,
                                                  unsigned long long limit_ns = WAIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// Polls check() until it reports an outcome (nonzero) and returns it, or
// returns `timeout` once limit_ns of %globaltimer have passed; sleeps 256 ns
// between polls. The streaming verifier's producers wait for work this way.
template <class Check>
__device__ __forceinline__ int poll_bounded(Check check, int timeout, unsigned long long limit_ns) {
  const unsigned long long t0 = global_ns();
  while (true) {
    const int o = check();
    if (o) return o;
    if (global_ns() - t0 > limit_ns) return timeout;
    __nanosleep(256);
  }
}
// 1-D TMA bulk copy global -> shared, completion counted on `bar`.
// Asks L2 to fetch [p, p + bytes) ahead of use (a hint: the range is
// trimmed to 16-byte boundaries inside it; nothing is copied anywhere).
__device__ __forceinline__ void prefetch_l2(const void *p, long long bytes) {
  const uintptr_t a0 = ((uintptr_t)p + 15) & ~(uintptr_t)15;
  const uintptr_t a1 = ((uintptr_t)p + (uintptr_t)bytes) & ~(uintptr_t)15;
  if (a1 > a0 && GCHK((const void *)a0, a1 - a0))
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a0), "r"((uint32_t)(a1 - a0))
                 : "memory");
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                        uint64_t *bar) {
  if (!GCHK(src, bytes)) {   // checked build: the copy is dropped, its bytes still count
    asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
    return;
  }
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ uint4 lds128(const void *p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

}  // namespace sv
