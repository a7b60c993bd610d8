// Sparse top-128 draft law ("RheoSampling 2026", §3 "Optimasi Sparse
// Top-128": the draft logits keep their 128 largest entries, the rest is set
// to -inf, and the softmax runs over the survivors).
//
// bf16 rows with V a multiple of 8 and V >= 4096, outside the RheoSampling
// epilogue, take two launches: k_topk128_scan streams the rows and leaves a
// candidate list per row, and k_topk128_finish selects, orders and softmaxes
// (see the two-launch section below). Everything else takes one launch,
// k_topk128:
//
// One 512-thread CTA per row at a time, two CTAs per SM, rows taken in grid
// strides (measured faster than 4 x 256 or 8 x 128 threads per SM). bf16 rows
// (V a multiple of 8, V >= 4096) take the fast path, each pass keeping eight
// 16-byte loads in flight per thread:
//   - a packed bf16 max pass leaves each thread's maximum. It also gathers the
//     elements at or above a bound predicted from the block's previous row
//     (that row's 128th largest logit minus a margin). When at least 128 reach
//     it, the top 128 are among them and the row needs no second pass;
//   - otherwise each warp sorts its 32 maxima, and the smallest of the warps'
//     (128/16 = 8)-th largest maxima bounds the 128th largest logit from
//     below (16 warps x 8 threads hold an element at least that large). A
//     second pass, served from L2, gathers the few hundred elements at or
//     above that bound;
//   - each candidate's rank under the order (logit descending, id ascending)
//     keeps the top 128.
// Other rows, and rows whose candidates overflow, use an exact radix select on
// order-preserving keys (-0 folded onto +0): the maximum, then 8-bit digits of
// the distance from it, and a collection pass that keeps the lowest ids among
// ties. The survivors are put in id order by counting smaller ids and
// softmaxed at temperature T; T < 0.05 gives a one-hot on the argmax.
//
// With a RheoSampling epilogue (spec_rheo_expand) the block then expands the
// row into its tree children from the survivors still in shared memory, so
// the 128 logits are neither written out nor gathered again.
#include "common.cuh"
#include "internal.h"

#include <climits>

namespace sv {

constexpr int TK_THREADS = 512;
constexpr int TK_CTAS_PER_SM = 2;
constexpr int TK_EPT = 16;
constexpr int TK_TILE = TK_THREADS * TK_EPT;

struct TopkArgs {
  const char *logits;
  int dtype;
  long long row_bytes;
  int rows_bound;
  int V;
  const int32_t *cu;
  const float *temp;
  int B;
  int32_t *out_idx;
  float *out_prob;
  WsHeader *hdr;
  int has_rh;
  RheoEpi rh;
  unsigned long long *cand;   // two-launch select: per row TK_GCAP composite keys
  int *cnt;                   // and their count
};

constexpr int TK_WARPS = TK_THREADS / 32;
constexpr int CAND_CAP = 1024;
static_assert(SPEC_TOPK % TK_WARPS == 0 && SPEC_TOPK / TK_WARPS <= 32, "bound needs k per warp");

struct TopkSmem {
  unsigned long long cand[CAND_CAP];   // (key << 32) | ~id of the candidates
  float tmax[TK_WARPS];                // per-warp (128 / warps)-th largest thread maxima
  int cand_n;
  float pilot;           // the scan's bound for a block's first row, from its first chunk
  unsigned hist[256];
  int scratch[33];
  int sel_idx[SPEC_TOPK];
  float sel_val[SPEC_TOPK];
  float sel_e[SPEC_TOPK];
  unsigned kmax;
  unsigned prefix;
  int need;
  int lt_count;
  int use_fallback;
  float S;
  float T;
  float zmax;            // largest survivor logit
  float prev128;         // the 128th largest logit of this block's previous fast-path row
  float delta;           // margin below it for the next row's predicted bound
  float red[8];          // epilogue: per-warp sums and scan totals
  float Zc, qm;
  int probe_lo, probe_hi;
};
constexpr int TK_PARTS = TK_THREADS / SPEC_TOPK;   // epilogue threads per survivor
static_assert(TK_PARTS * SPEC_TOPK == TK_THREADS && TK_PARTS >= 1, "whole parts per survivor");
static_assert(CAND_CAP * 2 >= (TK_PARTS + 1) * SPEC_TOPK, "the epilogue's counters fit");

__device__ __forceinline__ unsigned key_of(uint32_t bits, bool bf16) {
  if (bf16) {
    bits &= 0xffffu;
    if (bits == 0x8000u) bits = 0;
    return (bits & 0x8000u) ? (~bits & 0xffffu) : (bits | 0x8000u);
  }
  if (bits == 0x80000000u) bits = 0;
  return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

__device__ __forceinline__ float value_of_bits(uint32_t bits, bool bf16) {
  return bf16 ? __uint_as_float((bits & 0xffffu) << 16) : __uint_as_float(bits);
}

__device__ __forceinline__ uint32_t load_bits(const char *row, bool bf16, int i) {
  return bf16 ? (uint32_t)GLDG(reinterpret_cast<const unsigned short *>(row) + i)
              : GLDG(reinterpret_cast<const uint32_t *>(row) + i);
}

// Calls f(bits, index) once for every element of the row, spread over the
// block in no particular order (128-bit loads on the aligned interior).
template <bool BF16, class F>
__device__ __forceinline__ void for_each_elem(const char *row, int V, F &&f) {
  constexpr int ESZ = BF16 ? 2 : 4, PER = 16 / ESZ;
  const int mis = (int)((uintptr_t)row & 15);
  const int head = min(V, mis ? (16 - mis) / ESZ : 0);
  const int nvec = (V - head) / PER;
  const int tail0 = head + nvec * PER;
  for (int i = threadIdx.x; i < head; i += blockDim.x) f(load_bits(row, BF16, i), i);
  const uint4 *vp = reinterpret_cast<const uint4 *>(row + (long long)head * ESZ);
#pragma unroll 4
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    const uint4 w = GLDG(vp + v);
    const int e = head + v * PER;
    if (BF16) {
      f(w.x & 0xffffu, e + 0); f(w.x >> 16, e + 1); f(w.y & 0xffffu, e + 2); f(w.y >> 16, e + 3);
      f(w.z & 0xffffu, e + 4); f(w.z >> 16, e + 5); f(w.w & 0xffffu, e + 6); f(w.w >> 16, e + 7);
    } else {
      f(w.x, e + 0); f(w.y, e + 1); f(w.z, e + 2); f(w.w, e + 3);
    }
  }
  for (int i = tail0 + threadIdx.x; i < V; i += blockDim.x) f(load_bits(row, BF16, i), i);
}

// Chooses the digit containing the need-th smallest element from sh.hist;
// extends sh.prefix by it and lowers sh.need by the count below it.
__device__ __forceinline__ void pick_digit(TopkSmem &sh) {
  if (threadIdx.x == 0) {
    unsigned cum = 0;
    int g = 0;
    for (; g < 255; ++g) {
      if (cum + sh.hist[g] >= (unsigned)sh.need) break;
      cum += sh.hist[g];
    }
    sh.prefix = (sh.prefix << 8) | (unsigned)g;
    sh.need -= (int)cum;
  }
  __syncthreads();
}


// bf16 keys back to values (inverse of key_of for 16-bit keys).
__device__ __forceinline__ float value_of_key16(unsigned key) {
  const unsigned bits = (key & 0x8000u) ? (key & 0x7fffu) : (~key & 0xffffu);
  return __uint_as_float(bits << 16);
}

// Appends the elements of 16-byte group v (eight bf16) at or above `bound`
// to the candidates, as composite keys (order-preserving key << 32 | ~id).
__device__ __forceinline__ void gather_candidates(const uint4 &w, int v, float bound,
                                                  TopkSmem &sh) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t b = (k & 1) ? (ww[k >> 1] >> 16) : (ww[k >> 1] & 0xffffu);
    if (__uint_as_float(b << 16) >= bound) {
      const int slot = atomicAdd(&sh.cand_n, 1);
      if (slot < CAND_CAP)
        sh.cand[slot] = ((unsigned long long)key_of(b, true) << 32) | (~(unsigned)(8 * v + k));
    }
  }
}

// Sorts one value per lane across the warp, descending: lane i ends with
// the (i+1)-th largest (bitonic network).
__device__ __forceinline__ float warp_sort_desc(float m) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, m, j);
      m = (((lane & k) == 0) == ((lane & j) == 0)) ? fmaxf(m, o) : fminf(m, o);
    }
  return m;
}

constexpr uint32_t NINF2 = 0xff80ff80u;   // packed (-inf, -inf)

// One 16-byte group (vector v of the row) of the max pass: the thread's
// packed maximum, and the group's elements at or above a finite `pred`.
__device__ __forceinline__ void max_pass_vec(const uint4 &w, int v, float pred, bool predicted,
                                             uint32_t &pm, TopkSmem &sh) {
  const uint32_t m8 = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
  pm = bmax2(pm, m8);
  if (predicted && fmaxf(bf16lo(m8), bf16hi(m8)) >= pred) gather_candidates(w, v, pred, sh);
}

// The rest of the gathering once the max pass has left each thread's packed
// maximum pm (and, with a prediction, its candidates): the count check and,
// when the prediction did not hold, the bound from the warps' maxima and the
// second pass. Starts and ends with a block barrier.
__device__ int finish_gather_bf16(const char *row, int V, TopkSmem &sh, float pred, uint32_t pm,
                                  int *n1_out, bool *held_out) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const uint4 *vp = reinterpret_cast<const uint4 *>(row);
  const int nvec = V / 8;
  const bool predicted = pred > -INFINITY;
  __syncthreads();
  const int n1 = sh.cand_n;
  const bool held = predicted && n1 >= SPEC_TOPK && n1 <= CAND_CAP;
  float bound = -INFINITY;
  if (!held) {   // the same branch in every thread
    const float m = warp_sort_desc(fmaxf(bf16lo(pm), bf16hi(pm)));   // the warp's maxima
    if (lane == SPEC_TOPK / TK_WARPS - 1) sh.tmax[warp] = m;
    __syncthreads();   // also: every thread has read the count before it is reset
    if (t == 0) sh.cand_n = 0;
    __syncthreads();
    bound = sh.tmax[0];
    for (int w = 1; w < TK_WARPS; ++w) bound = fminf(bound, sh.tmax[w]);
  }
  // the second pass (from L2), eight loads in flight again; a group of 8
  // logits is looked at only when its packed maximum reaches the bound
  for (int v0 = t; v0 < nvec && !held; v0 += 8 * TK_THREADS) {
    uint4 wv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int v = v0 + u * TK_THREADS;
      wv[u] = v < nvec ? GLDG(vp + v) : make_uint4(NINF2, NINF2, NINF2, NINF2);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int v = v0 + u * TK_THREADS;
      const uint4 w = wv[u];
      const uint32_t m8 = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
      if (v >= nvec || fmaxf(bf16lo(m8), bf16hi(m8)) < bound) continue;
      gather_candidates(w, v, bound, sh);
    }
  }
  __syncthreads();
  *n1_out = n1;
  *held_out = held;
  return sh.cand_n;
}

__device__ int gather_bf16(const char *row, int V, TopkSmem &sh, float pred, int *n1_out,
                           bool *held_out) {
  const int t = threadIdx.x;
  const uint4 *vp = reinterpret_cast<const uint4 *>(row);
  const int nvec = V / 8;
  uint32_t pm = NINF2;
  const bool predicted = pred > -INFINITY;
  if (t == 0) sh.cand_n = 0;
  __syncthreads();
  // eight 16-byte loads in flight per thread before any is used
  for (int v0 = t; v0 < nvec; v0 += 8 * TK_THREADS) {
    uint4 w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int v = v0 + u * TK_THREADS;
      w[u] = v < nvec ? GLDG(vp + v) : make_uint4(NINF2, NINF2, NINF2, NINF2);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (v0 + u * TK_THREADS < nvec) max_pass_vec(w[u], v0 + u * TK_THREADS, pred, predicted, pm, sh);
  }
  return finish_gather_bf16(row, V, sh, pred, pm, n1_out, held_out);
}

// Each of the n <= CAND_CAP candidates' rank under (logit descending, id
// ascending), counted by a pair of threads (each half the candidates); the
// top 128 land in sel_idx / sel_val by rank. Every lane runs the same number
// of rounds.
__device__ void rank_candidates(TopkSmem &sh, int n) {
  const int t = threadIdx.x;
  for (int base = 0; base < n; base += TK_THREADS / 2) {
    const int i = base + (t >> 1);
    const unsigned long long ci = i < n ? sh.cand[i] : 0ull;
    int r = 0;
    if (i < n)
      for (int j = t & 1; j < n; j += 2) r += sh.cand[j] > ci;
    r += __shfl_xor_sync(0xffffffffu, r, 1);
    if (i < n && (t & 1) == 0 && r < SPEC_TOPK) {
      sh.sel_idx[r] = (int)~(unsigned)(ci & 0xffffffffull);
      sh.sel_val[r] = value_of_key16((unsigned)(ci >> 32));
    }
  }
  __syncthreads();
}

// The next row's prediction (thread 0): this row's 128th largest logit v128,
// and a margin that widens after a miss and narrows when the candidates were
// many.
__device__ __forceinline__ void predict_next(TopkSmem &sh, float v128, bool predicted, bool held,
                                             int n1) {
  sh.prev128 = v128;
  if (predicted && !held) sh.delta = fminf(sh.delta * 2.f, 64.f);
  else if (held && n1 > 4 * SPEC_TOPK) sh.delta = fmaxf(sh.delta * 0.5f, 1.f / 64.f);
}

// Fast selection for bf16 rows with V % 8 == 0 and V >= 8 * TK_THREADS
// (every row 16-byte aligned, every thread holds elements). A packed max pass
// leaves each thread's maximum; every warp sorts its 32 maxima with a
// shuffle bitonic network, and the smallest of the warps' 8th-largest
// maxima is a lower bound on the 128-th largest element (16 warps x 8
// threads each hold an element at least that large). A second pass, read
// back from L2 (one row per CTA, two CTAs per SM, keeps the rows in flight
// far below L2), gathers the elements at or above the bound — a few hundred
// on logit rows — and the exact top 128 (ties to the lower id) is ranked
// among them in shared memory. Returns false, having written no selection,
// when the candidates overflow CAND_CAP.
//
// With a predicted bound `pred` (finite: the block's previous row's 128th
// largest logit minus a margin), the max pass also gathers the elements at or
// above pred. When at least 128 are found, every element of the top 128 is
// among them (the 128th largest is then >= pred), so the second pass is
// skipped; otherwise (too few, or an overflow) the second pass runs as above.
__device__ bool select_bf16_fast(const char *row, int V, TopkSmem &sh, float pred) {
  int n1;
  bool held;
  const int n = gather_bf16(row, V, sh, pred, &n1, &held);
  if (n > CAND_CAP) return false;
  rank_candidates(sh, n);
  if (threadIdx.x == 0) predict_next(sh, sh.sel_val[SPEC_TOPK - 1], pred > -INFINITY, held, n1);
  return true;
}


// RheoSampling expansion of row r ("RheoSampling 2026": §2 true sampling law
// and proxy, §3 rheostat m, §7 no temperature in construction), run by the
// whole block after the select. sh.sel_idx / sel_val hold the survivors in
// ascending id, sh.sel_e / sh.S their law at the tree's temperature (the
// probe's true sampling law) and sh.zmax their largest logit.
__device__ void rheo_epilogue(const TopkArgs &a, TopkSmem &sh, int r, int ksel) {
  const RheoEpi &h = a.rh;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  int *cnt = reinterpret_cast<int *>(sh.cand);   // free once the select is done
  int *rank_of = cnt + TK_PARTS * SPEC_TOPK;
  {
    // rank best first (logit descending, ties and -inf to the lower id,
    // padding last): TK_PARTS threads per survivor count a share each
    constexpr int SHARE = SPEC_TOPK / TK_PARTS;
    const int e = t & (SPEC_TOPK - 1), part = t / SPEC_TOPK;
    const float ze = e < ksel ? sh.sel_val[e] : -INFINITY;
    const int ke = e < ksel ? sh.sel_idx[e] : INT_MAX;
    int c = 0;
#pragma unroll 8
    for (int j = part * SHARE; j < part * SHARE + SHARE; ++j) {
      const float zj = j < ksel ? sh.sel_val[j] : -INFINITY;
      const int kj = j < ksel ? sh.sel_idx[j] : INT_MAX;
      c += (zj > ze || (zj == ze && kj < ke)) ? 1 : 0;
    }
    cnt[part * SPEC_TOPK + e] = c;
  }
  if (t == 0) {
    sh.probe_lo = SPEC_TOPK;
    sh.probe_hi = -1;
    sh.qm = 0.f;
  }
  __syncthreads();
  // survivors (threads t < 128): rank, unscaled weight, probe-law prefix sum
  const bool surv = t < SPEC_TOPK;
  const bool valid = t < ksel;
  int rk = SPEC_TOPK;
  float eu = 0.f, qt = 0.f, C = 0.f;
  if (surv) {
    rk = 0;
#pragma unroll
    for (int q = 0; q < TK_PARTS; ++q) rk += cnt[q * SPEC_TOPK + t];
    rank_of[t] = rk;
    eu = valid && sh.sel_val[t] > -INFINITY ? expf(sh.sel_val[t] - sh.zmax) : 0.f;
    qt = valid ? sh.sel_e[t] / sh.S : 0.f;
    float su = eu;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) su += __shfl_xor_sync(0xffffffffu, su, o);
    C = qt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, C, o);
      if (lane >= o) C += y;
    }
    if (lane == 31) {
      sh.red[warp] = su;
      sh.red[4 + warp] = C;
    }
  }
  __syncthreads();
  float qu = 0.f;
  if (surv) {
    float off = 0.f;
    for (int k = 0; k < warp; ++k) off += sh.red[4 + k];
    C += off;
    if (t == SPEC_TOPK - 1) sh.Zc = C;
    qu = eu / (sh.red[0] + sh.red[1] + sh.red[2] + sh.red[3]);
    if (valid && rk == h.m) sh.qm = qu;        // q(x_{m+1})
  }
  __syncthreads();
  if (surv) {
    // the probe: the smallest id (ascending slot) with u * Z < C; if rounding
    // leaves none, the last slot with weight
    const float tu = uniform24(h.seed, (uint32_t)r, (uint32_t)h.level, 3u) * sh.Zc;
    if (tu < C) atomicMin(&sh.probe_lo, t);
    if (qt > 0.f) atomicMax(&sh.probe_hi, t);
  }
  __syncthreads();
  if (valid) {
    const int ps = sh.probe_lo < SPEC_TOPK ? sh.probe_lo : max(sh.probe_hi, 0);
    const int prk = rank_of[ps];
    const size_t out0 = (size_t)r * h.K;
    const float fs = GLD(h.fscore + (r));
    int slot = -1;
    float pr = qu;
    if (t == ps) {
      slot = h.m;
      pr = sh.qm + h.eps;
    } else {
      const int rr = rk - (prk < rk ? 1 : 0);
      if (rr < h.K - 1) slot = rr < h.m ? rr : rr + 1;
    }
    if (slot >= 0) {
      GST(h.token + (out0 + slot), sh.sel_idx[t]);
      if (h.qproxy) GST(h.qproxy + (out0 + slot), pr);
      if (h.qtrue) GST(h.qtrue + (out0 + slot), qt);
      GST(h.score + (out0 + slot), fs + logf(pr));
    }
  }
  __syncthreads();
}

// Exact top 128 of a row with V > 128 into sel_idx / sel_val (in no
// particular order), by radix select on order-preserving keys (-0 folded
// onto +0): the maximum, then 8-bit digits of the distance from it, and a
// collection pass that keeps the lowest ids among ties. Uses sh.hist,
// sh.kmax and the digit state; ends with the block synchronised.
template <bool BF16>
__device__ void select_radix(const char *row, int V, TopkSmem &sh) {
  constexpr int BITS = BF16 ? 16 : 32;
  const int t = threadIdx.x;
  // pass 1: the maximum key
  __syncthreads();
  if (t == 0) { sh.kmax = 0; sh.lt_count = 0; sh.prefix = 0; sh.need = SPEC_TOPK; }
  for (int i = t; i < 256; i += blockDim.x) sh.hist[i] = 0;
  __syncthreads();
  unsigned km = 0;
  for_each_elem<BF16>(row, V, [&](uint32_t bits, int) { km = max(km, key_of(bits, BF16)); });
  atomicMax(&sh.kmax, km);
  __syncthreads();
  const unsigned kmax = sh.kmax;
  // pass 2: fine histogram of the second digit over d < 2^(BITS-8)
  for_each_elem<BF16>(row, V, [&](uint32_t bits, int) {
    const unsigned d = kmax - key_of(bits, BF16);
    if ((d >> (BITS - 8)) == 0) atomicAdd(&sh.hist[(d >> (BITS - 16)) & 0xffu], 1u);
  });
  __syncthreads();
  if (t == 0) {
    unsigned tot = 0;
    for (int g = 0; g < 256; ++g) tot += sh.hist[g];
    sh.use_fallback = tot < (unsigned)SPEC_TOPK;
  }
  __syncthreads();
  int shift;
  if (!sh.use_fallback) {
    pick_digit(sh);  // the top digit is 0; this picks the second one
    shift = BITS - 24;
  } else {
    // full top-digit pass (rows whose top 128 spread widely)
    for (int i = t; i < 256; i += blockDim.x) sh.hist[i] = 0;
    __syncthreads();
    for_each_elem<BF16>(row, V, [&](uint32_t bits, int) {
      atomicAdd(&sh.hist[(kmax - key_of(bits, BF16)) >> (BITS - 8)], 1u);
    });
    __syncthreads();
    pick_digit(sh);
    shift = BITS - 16;
  }
  for (; shift >= 0; shift -= 8) {
    for (int i = t; i < 256; i += blockDim.x) sh.hist[i] = 0;
    __syncthreads();
    const unsigned pre = sh.prefix;
    for_each_elem<BF16>(row, V, [&](uint32_t bits, int) {
      const unsigned d = kmax - key_of(bits, BF16);
      if ((d >> (shift + 8)) == pre) atomicAdd(&sh.hist[(d >> shift) & 0xffu], 1u);
    });
    __syncthreads();
    pick_digit(sh);
  }
  // collection: d < thr anywhere; among d == thr the `need` lowest ids
  const unsigned thr = sh.prefix;
  const int need = sh.need;
  const int c_lt = SPEC_TOPK - need;
  int tie_base = 0;
  const bool vec_ok = ((uintptr_t)row & 15) == 0;
  for (int x0t = 0; x0t < V; x0t += TK_TILE) {
    const int x0 = x0t + t * TK_EPT;
    uint32_t bits[TK_EPT];
    if (vec_ok && x0 + TK_EPT <= V) {
      const uint4 *p = reinterpret_cast<const uint4 *>(row + (long long)x0 * (BF16 ? 2 : 4));
      if (BF16) {
#pragma unroll
        for (int q = 0; q < TK_EPT / 8; ++q) {
          const uint4 w = GLDG(p + q);
          bits[8 * q + 0] = w.x & 0xffffu; bits[8 * q + 1] = w.x >> 16;
          bits[8 * q + 2] = w.y & 0xffffu; bits[8 * q + 3] = w.y >> 16;
          bits[8 * q + 4] = w.z & 0xffffu; bits[8 * q + 5] = w.z >> 16;
          bits[8 * q + 6] = w.w & 0xffffu; bits[8 * q + 7] = w.w >> 16;
        }
      } else {
#pragma unroll
        for (int q = 0; q < TK_EPT / 4; ++q) {
          const uint4 w = GLDG(p + q);
          bits[4 * q + 0] = w.x; bits[4 * q + 1] = w.y;
          bits[4 * q + 2] = w.z; bits[4 * q + 3] = w.w;
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < TK_EPT; ++k) bits[k] = x0 + k < V ? load_bits(row, BF16, x0 + k) : 0u;
    }
    int nt = 0;
#pragma unroll
    for (int k = 0; k < TK_EPT; ++k) {
      if (x0 + k >= V) break;
      const unsigned d = kmax - key_of(bits[k], BF16);
      if (d < thr) {
        const int slot = atomicAdd(&sh.lt_count, 1);
        if (slot < SPEC_TOPK) {
          sh.sel_idx[slot] = x0 + k;
          sh.sel_val[slot] = value_of_bits(bits[k], BF16);
        }
      } else if (d == thr) {
        ++nt;
      }
    }
    int tot;
    const int excl = block_excl_scan_int(nt, sh.scratch, &tot);
    if (nt > 0) {
      int rank = tie_base + excl;
#pragma unroll
      for (int k = 0; k < TK_EPT; ++k) {
        if (x0 + k >= V) break;
        if (kmax - key_of(bits[k], BF16) == thr) {
          if (rank < need) {
            sh.sel_idx[c_lt + rank] = x0 + k;
            sh.sel_val[c_lt + rank] = value_of_bits(bits[k], BF16);
          }
          ++rank;
        }
      }
    }
    tie_base += tot;
  }
  __syncthreads();
}

// Row r's request (largest b with cu[b] <= r) -> sh.T: warp 0 narrows the
// range 32-fold per step with one load per lane. Ends with a block barrier.
__device__ void row_temperature(const TopkArgs &a, TopkSmem &sh, int r) {
  const int t = threadIdx.x;
  if (t < 32) {
    int lo = 0, hi = a.B;
    while (hi - lo > 1) {
      const int step = (hi - lo + 31) / 32;
      const int probe = lo + t * step;
      const bool le = probe < hi && GLD(a.cu + (probe)) <= r;
      const unsigned m = __ballot_sync(0xffffffffu, le);
      const int last = 31 - __clz(m);        // lane 0 always qualifies (cu[lo] <= r)
      lo = lo + last * step;
      hi = min(hi, lo + step);
    }
    if (t == 0) sh.T = GLD(a.temp + (lo));
  }
  __syncthreads();
}

__device__ void finish_row(const TopkArgs &a, TopkSmem &sh, int r, int ksel);

template <bool BF16>
__device__ void topk_row(const TopkArgs &a, TopkSmem &sh, int r) {
  const char *row = a.logits + (long long)r * a.row_bytes;
  const int V = a.V;
  const int t = threadIdx.x;
  row_temperature(a, sh, r);
  const int ksel = min(SPEC_TOPK, V);
  if (V <= SPEC_TOPK) {
    if (t < SPEC_TOPK) {
      sh.sel_idx[t] = t < V ? t : 0x7fffffff;
      sh.sel_val[t] = t < V ? value_of_bits(load_bits(row, BF16, t), BF16) : -INFINITY;
    }
    __syncthreads();
  } else if (BF16 && V % 8 == 0 && V >= 8 * TK_THREADS && ((uintptr_t)row & 15) == 0 &&
             select_bf16_fast(row, V, sh, sh.prev128 - sh.delta)) {
    // selected by the fast path
  } else {
    select_radix<BF16>(row, V, sh);
  }
  finish_row(a, sh, r, ksel);
}

// The rest of a row once its ksel survivors are in sel_idx / sel_val (in any
// order) and its temperature in sh.T: id order, softmax, the outputs and the
// construction epilogue.
__device__ void finish_row(const TopkArgs &a, TopkSmem &sh, int r, int ksel) {
  const int t = threadIdx.x;
  const float T = sh.T;
  const bool greedy = !(T >= SPEC_GREEDY_T);
  // order the survivors by id: each finds its place by counting smaller ids
  // (ids are distinct; padding slots carry INT_MAX and stay at the end)
  {
    int id = 0x7fffffff, place = SPEC_TOPK;
    float val = -INFINITY;
    if (t < SPEC_TOPK) {
      id = sh.sel_idx[t];
      val = sh.sel_val[t];
      place = 0;
      for (int j = 0; j < SPEC_TOPK; ++j) place += sh.sel_idx[j] < id || (sh.sel_idx[j] == id && j < t);
    }
    __syncthreads();
    if (t < SPEC_TOPK) {
      sh.sel_idx[place] = id;
      sh.sel_val[place] = val;
    }
    __syncthreads();
  }
  // softmax over the survivors (fixed summation order); greedy: one-hot
  if (t < 32) {
    float m = -INFINITY;
    for (int k = t; k < ksel; k += 32) m = fmaxf(m, sh.sel_val[k]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (t == 0) sh.zmax = m;
    if (greedy) {
      int first = 0x7fffffff;
      for (int k = t; k < ksel; k += 32)
        if (sh.sel_val[k] == m) first = min(first, k);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
      for (int k = t; k < SPEC_TOPK; k += 32) sh.sel_e[k] = k == first ? 1.f : 0.f;
      if (t == 0) sh.S = 1.f;
    } else {
      const float c = (float)(1.4426950408889634 / (double)T);
      float s = 0.f;
      for (int k = t; k < SPEC_TOPK; k += 32) {
        const float e = k < ksel ? ex2((sh.sel_val[k] - m) * c) : 0.f;
        sh.sel_e[k] = e;
        s += e;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (t == 0) sh.S = s;
    }
  }
  __syncthreads();
  if (t < SPEC_TOPK && a.out_idx != nullptr) {
    const bool ok = t < ksel;
    GST(a.out_idx + ((long long)r * SPEC_TOPK + t), ok ? sh.sel_idx[t] : -1);
    GST(a.out_prob + ((long long)r * SPEC_TOPK + t), ok ? sh.sel_e[t] / sh.S : 0.f);
  }
  if (a.has_rh) rheo_epilogue(a, sh, r, ksel);
  __syncthreads();
}

__global__ void __launch_bounds__(TK_THREADS, TK_CTAS_PER_SM) k_topk128(const TopkArgs a) {
  __shared__ TopkSmem sh;
  if (a.hdr->status != SPEC_OK) return;   // inputs already rejected
  if (threadIdx.x == 0) {
    sh.prev128 = -INFINITY;   // no prediction for the first row
    sh.delta = 0.5f;
  }
  __syncthreads();
  const int rows = min(a.rows_bound, GLD(a.cu + (a.B)));
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    if (a.dtype == SPEC_BF16) topk_row<true>(a, sh, r);
    else topk_row<false>(a, sh, r);
  }
}

// ------------------------------------------------------ two-launch select
// For bf16 rows with V % 8 == 0 and V >= 8 * TK_THREADS and no epilogue, the
// select runs as two launches so that the blocks streaming the rows keep
// their loads in flight: in the one-launch kernel every block spends about as
// long on a row's ranking, ordering and softmax as on reading it, and the
// blocks, all in step, leave HBM idle meanwhile.
//   - k_topk128_scan (the blocks of k_topk128) streams each row once with the
//     gathering passes above and leaves a list of at most TK_GCAP composite
//     keys (key << 32 | ~id) that holds the row's top 128: its candidates, or,
//     when those are more than TK_GCAP, the top 128 themselves (ranked in the
//     block, or found by the exact radix select after an overflow). The next
//     row's bound is predicted from a histogram of the list's keys.
//   - k_topk128_finish, a warp per row, takes the exact top 128 of the list
//     by radix select on the composite keys (unique, so exactly 128 reach the
//     threshold), orders them by id and softmaxes them with the arithmetic of
//     the one-launch kernel.
constexpr int TK_GCAP = 512;
static_assert(TK_GCAP >= SPEC_TOPK && TK_GCAP <= CAND_CAP, "a list holds the top 128");

// Called by a whole warp on a histogram of one 8-bit digit: the digit g
// holding the need-th largest of the counted keys (1 <= need <= total), with
// `above` the count of keys in higher digits and `cnt` the count in g, in
// every lane; -1 when the histogram holds fewer than `need`. Lane l reads
// digits 255 - 8l down to 248 - 8l.
__device__ __forceinline__ int warp_digit_from_top(const unsigned *hist, unsigned need,
                                                   unsigned &above, unsigned &cnt) {
  const int lane = threadIdx.x & 31;
  unsigned h[8], s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    h[j] = hist[255 - 8 * lane - j];
    s += h[j];
  }
  unsigned incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int g = -1;
  above = 0;
  cnt = 0;
  if (incl - s < need && incl >= need) {
    unsigned cum = incl - s;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (g < 0 && cum + h[j] >= need) {
        g = 255 - 8 * lane - j;
        above = cum;
        cnt = h[j];
      }
      cum += h[j];
    }
  }
  const int owner = __ffs(__ballot_sync(0xffffffffu, g >= 0)) - 1;
  if (owner < 0) return -1;
  above = __shfl_sync(0xffffffffu, above, owner);
  cnt = __shfl_sync(0xffffffffu, cnt, owner);
  return __shfl_sync(0xffffffffu, g, owner);
}

template <int NS>
struct ScanRing {
  uint64_t full[NS];
  unsigned rel[NS];   // warps done with the stage's current chunk
  int uses[NS];       // chunks issued into the stage
  int abort;
};

// Issues chunk k of the block's sequence (its j-th row's chunk c,
// k = j * nch + c) into stage k % NS.
template <int NS, int ST>
__device__ __forceinline__ void scan_issue(const TopkArgs &a, ScanRing<NS> &rg,
                                           unsigned char *ring, long long k, int nch) {
  const long long j = k / nch;
  const int c = (int)(k - j * nch);
  const long long r = blockIdx.x + j * gridDim.x;
  const long long off = (long long)c * ST;
  const uint32_t bytes = (uint32_t)min((long long)ST, a.row_bytes - off);
  const int s = (int)(k % NS);
  mbar_arrive_tx(&rg.full[s], bytes);
  bulk_g2s(ring + (size_t)s * ST, a.logits + r * a.row_bytes + off, bytes, &rg.full[s]);
  ++rg.uses[s];
}

// One row of the scan: the max pass over the row's chunks as they land in the
// ring (the last warp done with a stage refills it with the chunk NS ahead,
// which runs on into the block's next row), then the rest of the gathering,
// the row's list and the next row's bound. Returns early, in every thread,
// once a wait has given up.
template <int NS, int ST>
__device__ void scan_row(const TopkArgs &a, TopkSmem &sh, ScanRing<NS> &rg, unsigned char *ring,
                         int r, int j, int nch, long long total) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const char *row = a.logits + (long long)r * a.row_bytes;
  // the bound predicted from the block's previous row; the first row takes
  // one from its first chunk instead (below)
  const bool cross = sh.prev128 - sh.delta > -INFINITY;
  float pred = sh.prev128 - sh.delta;
  bool predicted = cross;
  volatile int *abort = &rg.abort;
  if (t == 0) sh.cand_n = 0;
  __syncthreads();
  uint32_t pm = NINF2;
  // every warp reads every chunk, in order: a warp waits for a stage's next
  // use only after its previous one completed, as the parity wait requires
  for (int c = 0; c < nch; ++c) {
    const long long k = (long long)j * nch + c;
    const int s = (int)(k % NS);
    const bool landed = mbar_wait_bounded(&rg.full[s], (uint32_t)((k / NS) & 1), abort);
    const int nv = (int)(min((long long)ST, a.row_bytes - (long long)c * ST) / 16);
    const unsigned char *buf = ring + (size_t)s * ST;
    if (landed) {
#pragma unroll 4
      for (int v = t; v < nv; v += TK_THREADS)
        max_pass_vec(lds128(buf + 16 * v), c * (ST / 16) + v, pred, predicted, pm, sh);
    } else if (!*abort) {
      set_status(a.hdr, SPEC_ERR_TIMEOUT, -4);
      *abort = 1;
    }
    if (c == 0 && !cross) {
      // first row: the 24th largest of the warps' two largest thread maxima
      // over the first chunk. At least 24 of the chunk's logits reach it; on
      // rows whose large logits are spread evenly about 2 in 1000 of the row
      // do, a few hundred candidates. The chunk is gathered again while it
      // is still staged. With fewer than 128 the second pass runs as usual.
      const float m = warp_sort_desc(fmaxf(bf16lo(pm), bf16hi(pm)));
      if (lane < 2) sh.sel_val[2 * warp + lane] = m;
      __syncthreads();
      if (warp == 0) {
        const float v = warp_sort_desc(sh.sel_val[lane]);
        if (lane == 23) sh.pilot = v;
      }
      __syncthreads();
      pred = sh.pilot;
      predicted = pred > -INFINITY;
      if (landed && predicted)
        for (int v = t; v < nv; v += TK_THREADS) {
          const uint4 w = lds128(buf + 16 * v);
          const uint32_t m8 = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
          if (fmaxf(bf16lo(m8), bf16hi(m8)) >= pred) gather_candidates(w, c * (ST / 16) + v, pred, sh);
        }
    }
    __syncwarp();   // the warp's reads of the stage are done
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&rg.rel[s], 1u) == TK_WARPS - 1) {   // the last warp out
        rg.rel[s] = 0;
        if (k + NS < total && !*abort) scan_issue<NS, ST>(a, rg, ring, k + NS, nch);
      }
    }
  }
  __syncthreads();
  if (*abort) return;   // read after the barrier: the same in every thread
  int n1;
  bool held;
  const int n = finish_gather_bf16(row, a.V, sh, pred, pm, &n1, &held);
  int nw = n;
  if (n > TK_GCAP) {
    if (n > CAND_CAP) {
      select_radix<true>(row, a.V, sh);
      // the radix select leaves its histogram behind
      for (int i = t; i < 256; i += TK_THREADS) sh.hist[i] = 0;
    } else {
      rank_candidates(sh, n);
    }
    if (t < SPEC_TOPK) {
      const uint32_t bits = __float_as_uint(sh.sel_val[t]) >> 16;
      sh.cand[t] = ((unsigned long long)key_of(bits, true) << 32) | ~(unsigned)sh.sel_idx[t];
    }
    __syncthreads();
    nw = SPEC_TOPK;
  }
  unsigned long long *dst = a.cand + (long long)r * TK_GCAP;
  for (int i = t; i < nw; i += TK_THREADS) GST(dst + i, sh.cand[i]);
  // the list's 128th largest key, by its two 8-bit digits (the histogram is
  // clear between rows): stored with the list, and the next row's bound
  for (int i = t; i < nw; i += TK_THREADS)
    atomicAdd(&sh.hist[(unsigned)(sh.cand[i] >> 40) & 0xffu], 1u);
  __syncthreads();
  if (warp == 0) {
    unsigned above, cnt;
    const int g1 = warp_digit_from_top(sh.hist, SPEC_TOPK, above, cnt);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j) sh.hist[8 * lane + j] = 0;
    if (lane == 0) {
      sh.prefix = (unsigned)max(g1, 0);
      sh.need = SPEC_TOPK - (int)above;
    }
  }
  __syncthreads();
  const unsigned g1 = sh.prefix;
  for (int i = t; i < nw; i += TK_THREADS) {
    const unsigned k = (unsigned)(sh.cand[i] >> 32);
    if ((k >> 8) == g1) atomicAdd(&sh.hist[k & 0xffu], 1u);
  }
  __syncthreads();
  if (warp == 0) {
    unsigned above, cnt;
    const int g0 = warp_digit_from_top(sh.hist, (unsigned)sh.need, above, cnt);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j) sh.hist[8 * lane + j] = 0;
    if (lane == 0) {
      const unsigned k128 = (g1 << 8) | (unsigned)max(g0, 0);
      GST(a.cnt + r, nw | (int)(k128 << 16));   // the list's size and 128th largest key
      const float v128 = value_of_key16(k128);
      if (cross && n1 > CAND_CAP) {   // the predicted bound was far too low
        sh.prev128 = v128;
        sh.delta = fmaxf(sh.delta * 0.5f, 1.f / 64.f);
      } else {
        predict_next(sh, v128, cross, held && cross, n1);
      }
    }
  }
  __syncthreads();   // the prediction and the cleared histogram before the next row
}

template <int NS, int ST, int CPS>
__global__ void __launch_bounds__(TK_THREADS, CPS) k_topk128_scan(const TopkArgs a) {
  extern __shared__ __align__(128) unsigned char ring[];   // NS * ST bytes
  __shared__ TopkSmem sh;
  __shared__ ScanRing<NS> rg;
  if (a.hdr->status != SPEC_OK) return;   // inputs already rejected
  const int t = threadIdx.x;
  const int rows = min(a.rows_bound, GLD(a.cu + (a.B)));
  const int nrow = rows > (int)blockIdx.x ? (rows - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int nch = (int)((a.row_bytes + ST - 1) / ST);
  const long long total = (long long)nrow * nch;
  for (int r = rows + (int)blockIdx.x * TK_THREADS + t; r < a.rows_bound;
       r += (int)gridDim.x * TK_THREADS)
    GST(a.cnt + r, 0);   // past the call's rows: empty lists
  for (int i = t; i < 256; i += TK_THREADS) sh.hist[i] = 0;
  if (t == 0) {
    sh.prev128 = -INFINITY;   // no prediction for the first row
    sh.delta = 0.5f;
    for (int s = 0; s < NS; ++s) {
      mbar_init(&rg.full[s], 1);
      rg.rel[s] = 0;
      rg.uses[s] = 0;
    }
    fence_mbar_init();
    rg.abort = 0;
  }
  __syncthreads();
  if (t == 0)
    for (long long k = 0; k < min((long long)NS, total); ++k)
      scan_issue<NS, ST>(a, rg, ring, k, nch);
  for (int j = 0; j < nrow; ++j) {
    scan_row<NS, ST>(a, sh, rg, ring, (int)blockIdx.x + j * (int)gridDim.x, j, nch, total);
    if (*(volatile int *)&rg.abort) break;   // set before a barrier every thread passed
  }
  if (t == 0 && *(volatile int *)&rg.abort) {
    // gave up: wait (bounded) for this block's copies in flight
    volatile int never = 0;
    for (int s = 0; s < NS; ++s)
      if (rg.uses[s] > 0) mbar_wait_bounded(&rg.full[s], (uint32_t)((rg.uses[s] - 1) & 1), &never);
  }
}

// The scan's ring and blocks per SM: two blocks of two 32 KB stages each
// (measured on B=256, K=7, V=151936: 4 x 16 KB 0.143 ms, 6 x 16 KB 0.146,
// 8 x 8 KB 0.207, 3 x 32 KB 0.126, 2 x 32 KB 0.124, 2 x 48 KB 0.123; one
// block per SM with 8 or 12 x 16 KB 0.205-0.218). Each stage costs every warp
// a wait and a release, so few large stages do best.
constexpr int TS_NS = 2, TS_STAGE = 32768, TS_CPS = 2;

constexpr int TF_THREADS = 128;   // the finishing launch: one block per row
static_assert(TF_THREADS == SPEC_TOPK, "a thread per survivor");

struct __align__(16) FinishSmem {
  int id[SPEC_TOPK];     // survivors; by id once sorted
  float val[SPEC_TOPK];
  int sid[SPEC_TOPK];    // each warp's 32 survivors sorted by id
  int tie[TK_GCAP];      // ids of the list's keys equal to its 128th largest
  int ngt, nt;
  float T;
};

// Lower bound of x in the ascending ids l[0..31]: how many are below x.
__device__ __forceinline__ int below32(const int *l, int x) {
  int lo = 0;
#pragma unroll
  for (int step = 16; step > 0; step >>= 1)
    if (l[lo + step - 1] < x) lo += step;
  return lo + (l[lo] < x);   // lo <= 31 here
}

__global__ void __launch_bounds__(TF_THREADS) k_topk128_finish(const TopkArgs a) {
  __shared__ FinishSmem f;
  if (a.hdr->status != SPEC_OK) return;   // the lists were not written
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const unsigned FULL = 0xffffffffu;
  // rows past the call's are marked empty by the scan
  for (int r = blockIdx.x; r < a.rows_bound; r += gridDim.x) {
    const int packed = GLD(a.cnt + r);
    const int n = packed & 0xffff;
    const unsigned k128 = (unsigned)packed >> 16;
    if (n == 0) continue;
    if (n < SPEC_TOPK || n > TK_GCAP) {   // not a list the scan leaves
      if (t == 0) set_status(a.hdr, SPEC_ERR_INVALID_ARG, r);
      continue;
    }
    if (t == 0) f.ngt = f.nt = 0;
    __syncthreads();
    if (warp == 0) {
      // request of this row (largest b with cu[b] <= r) -> temperature, the
      // range narrowed 32-fold per step with one load per lane
      int lo = 0, hi = a.B;
      while (hi - lo > 1) {
        const int step = (hi - lo + 31) / 32;
        const int probe = lo + lane * step;
        const bool le = probe < hi && GLD(a.cu + (probe)) <= r;
        const unsigned m = __ballot_sync(FULL, le);
        lo = lo + (31 - __clz(m)) * step;   // lane 0 always qualifies (cu[lo] <= r)
        hi = min(hi, lo + step);
      }
      if (lane == 0) f.T = GLD(a.temp + (lo));
    } else {
      // the other warps sort the list by the 128th largest key: keys above
      // it are in, keys equal to it are ties
      const unsigned long long *src = a.cand + (long long)r * TK_GCAP;
#pragma unroll 2
      for (int i = t - 32; i < n; i += TF_THREADS - 32) {
        const unsigned long long c = GLD(src + i);
        const unsigned key = (unsigned)(c >> 32);
        const int id = (int)~(unsigned)(c & 0xffffffffull);
        if (key > k128) {
          const int p = atomicAdd(&f.ngt, 1);
          if (p < SPEC_TOPK) {
            f.id[p] = id;
            f.val[p] = value_of_key16(key);
          }
        } else if (key == k128) {
          f.tie[atomicAdd(&f.nt, 1)] = id;
        }
      }
    }
    __syncthreads();
    const int ngt = f.ngt, nt = f.nt, need = SPEC_TOPK - ngt;
    if (ngt >= SPEC_TOPK || nt < need) {   // cannot happen: k128 is the 128th largest key
      if (t == 0) set_status(a.hdr, SPEC_ERR_INVALID_ARG, r);
      __syncthreads();
      continue;
    }
    // the `need` lowest ids among the ties
    for (int q = t; q < nt; q += TF_THREADS) {
      const int id = f.tie[q];
      int rank = 0;
      for (int j = 0; j < nt; ++j) rank += f.tie[j] < id;
      if (rank < need) {
        f.id[ngt + rank] = id;
        f.val[ngt + rank] = value_of_key16(k128);
      }
    }
    __syncthreads();
    // id order: a bitonic sort of each warp's 32, then each survivor's place
    // is its rank in its warp plus the count of smaller ids in the others
    int id = f.id[t];
    float val = f.val[t];
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        const int oid = __shfl_xor_sync(FULL, id, j);
        const float oval = __shfl_xor_sync(FULL, val, j);
        const bool keep_min = ((lane & k) == 0) == ((lane & j) == 0);
        if (keep_min ? oid < id : oid > id) {
          id = oid;
          val = oval;
        }
      }
    f.sid[t] = id;
    __syncthreads();
    int place = lane;
#pragma unroll
    for (int w = 0; w < SPEC_TOPK / 32; ++w)
      if (w != warp) place += below32(&f.sid[32 * w], id);
    f.id[place] = id;
    f.val[place] = val;
    __syncthreads();
    if (warp == 0) {
      // softmax over the survivors in id order, summed in the order of the
      // one-launch kernel; greedy: one-hot on the first maximum
      float v[4], m = -INFINITY;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[q] = f.val[lane + 32 * q];
        m = fmaxf(m, v[q]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
      const float T = f.T;
      float e[4], S;
      if (!(T >= SPEC_GREEDY_T)) {
        int first = 0x7fffffff;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (v[q] == m) first = min(first, lane + 32 * q);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(FULL, first, o));
#pragma unroll
        for (int q = 0; q < 4; ++q) e[q] = lane + 32 * q == first ? 1.f : 0.f;
        S = 1.f;
      } else {
        const float cT = (float)(1.4426950408889634 / (double)T);
        S = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          e[q] = ex2((v[q] - m) * cT);
          S += e[q];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(FULL, S, o);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const long long k = (long long)r * SPEC_TOPK + lane + 32 * q;
        GST(a.out_idx + k, f.id[lane + 32 * q]);
        GST(a.out_prob + k, e[q] / S);
      }
    }
    __syncthreads();   // the block's buffers are read before the next row
  }
}

// The finishing launch for rows with the construction epilogue: one
// 512-thread block per row takes the top 128 from the scan's list as
// k_topk128_finish does (keys above the 128th largest, the lowest ids among
// ties at it), then runs the one-launch kernel's id order, softmax and
// epilogue on them.
__global__ void __launch_bounds__(TK_THREADS) k_topk128_finish_rows(const TopkArgs a) {
  __shared__ TopkSmem sh;
  if (a.hdr->status != SPEC_OK) return;   // the lists were not written
  const int t = threadIdx.x;
  int *tie = reinterpret_cast<int *>(sh.cand);   // ids whose key equals the 128th
  static_assert(sizeof(sh.cand) >= TK_GCAP * sizeof(int), "the ties fit");
  // rows past the call's are marked empty by the scan
  for (int r = blockIdx.x; r < a.rows_bound; r += gridDim.x) {
    const int packed = GLD(a.cnt + r);
    const int n = packed & 0xffff;
    const unsigned k128 = (unsigned)packed >> 16;
    if (n == 0) continue;
    if (n < SPEC_TOPK || n > TK_GCAP) {   // not a list the scan leaves
      if (t == 0) set_status(a.hdr, SPEC_ERR_INVALID_ARG, r);
      continue;
    }
    if (t == 0) sh.cand_n = sh.lt_count = 0;
    row_temperature(a, sh, r);   // ends with a barrier
    if (t < n) {
      const unsigned long long c = GLD(a.cand + ((long long)r * TK_GCAP + t));
      const unsigned key = (unsigned)(c >> 32);
      const int id = (int)~(unsigned)(c & 0xffffffffull);
      if (key > k128) {
        const int p = atomicAdd(&sh.cand_n, 1);
        if (p < SPEC_TOPK) {
          sh.sel_idx[p] = id;
          sh.sel_val[p] = value_of_key16(key);
        }
      } else if (key == k128) {
        tie[atomicAdd(&sh.lt_count, 1)] = id;
      }
    }
    __syncthreads();
    const int ngt = sh.cand_n, nt = sh.lt_count, need = SPEC_TOPK - ngt;
    if (ngt >= SPEC_TOPK || nt < need) {   // cannot happen: k128 is the 128th largest key
      if (t == 0) set_status(a.hdr, SPEC_ERR_INVALID_ARG, r);
      __syncthreads();
      continue;
    }
    if (t < nt) {   // the `need` lowest ids among the ties
      const int id = tie[t];
      int rank = 0;
      for (int j = 0; j < nt; ++j) rank += tie[j] < id;
      if (rank < need) {
        sh.sel_idx[ngt + rank] = id;
        sh.sel_val[ngt + rank] = value_of_key16(k128);
      }
    }
    __syncthreads();
    finish_row(a, sh, r, SPEC_TOPK);
  }
}

__global__ void k_topk_validate(const TopkArgs a) {
  // one block: reset the status word, check offsets and temperatures
  if (threadIdx.x == 0) {
    a.hdr->status = SPEC_OK;
    a.hdr->detail = -1;
  }
  __syncthreads();
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
    const int K = GLD(a.cu + (b + 1)) - GLD(a.cu + (b));
    const float T = GLD(a.temp + (b));
    if ((b == 0 && GLD(a.cu + (0)) != 0) || K < 0 || !(T >= 0.f) || !isfinite(T))
      set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);
  }
  if (threadIdx.x == 0 && GLD(a.cu + (a.B)) > a.rows_bound) set_status(a.hdr, SPEC_ERR_INVALID_ARG, a.B);
}

size_t topk_list_bytes_for(long long rows, int V) {
  return V % 8 == 0 && V >= 8 * TK_THREADS ? topk_list_bytes(rows) : 0;
}

size_t topk_list_bytes(long long rows) {
  return align256(sizeof(unsigned long long) * (size_t)rows * TK_GCAP) +
         align256(sizeof(int) * (size_t)rows);
}

bool topk_two_launch(int dtype, int V) {
  return dtype == SPEC_BF16 && V % 8 == 0 && V >= 8 * TK_THREADS;
}

int launch_topk128(const void *logits, int dtype, int rows_bound, int V, const int32_t *cu_rows,
                   const float *temperature, int B, int32_t *out_idx, float *out_prob,
                   WsHeader *hdr, cudaStream_t stream, const RheoEpi *rh, void *lists,
                   cudaEvent_t before, cudaEvent_t after) {
  if (check_upload(stream) != SPEC_OK) return SPEC_ERR_CUDA;
  TopkArgs a{};
  a.has_rh = rh != nullptr;
  if (rh) a.rh = *rh;
  a.logits = static_cast<const char *>(logits);
  a.dtype = dtype;
  a.row_bytes = (long long)V * (dtype == SPEC_BF16 ? 2 : 4);
  a.rows_bound = rows_bound;
  a.V = V;
  a.cu = cu_rows;
  a.temp = temperature;
  a.B = B;
  a.out_idx = out_idx;
  a.out_prob = out_prob;
  a.hdr = hdr;
  if (rows_bound <= 0) return SPEC_OK;
  const int sms = num_sms();
  if (sms <= 0) return SPEC_ERR_CUDA;
  const int grid = min(rows_bound, TK_CTAS_PER_SM * sms);
  if (before && cudaEventRecord(before, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  if (lists != nullptr && topk_two_launch(dtype, V)) {
    const int sgrid = min(rows_bound, TS_CPS * sms);
    a.cand = static_cast<unsigned long long *>(lists);
    a.cnt = reinterpret_cast<int *>(static_cast<char *>(lists) +
                                    align256(sizeof(unsigned long long) * (size_t)rows_bound *
                                             TK_GCAP));
    constexpr int ring_bytes = TS_NS * TS_STAGE;
    if (cudaFuncSetAttribute(k_topk128_scan<TS_NS, TS_STAGE, TS_CPS>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, ring_bytes) != cudaSuccess)
      return SPEC_ERR_CUDA;
    k_topk128_scan<TS_NS, TS_STAGE, TS_CPS><<<sgrid, TK_THREADS, ring_bytes, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
    if (after && cudaEventRecord(after, stream) != cudaSuccess) return SPEC_ERR_CUDA;
    if (rh != nullptr)
      k_topk128_finish_rows<<<min(rows_bound, 4 * sms), TK_THREADS, 0, stream>>>(a);
    else
      k_topk128_finish<<<min(rows_bound, 16 * sms), TF_THREADS, 0, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
  }
  k_topk128<<<grid, TK_THREADS, 0, stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (after && cudaEventRecord(after, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

constexpr size_t TOPK_WS = 256;

}  // namespace sv

using namespace sv;

extern "C" size_t draft_topk_softmax_workspace(int rows, int V) {
  if (rows < 0 || V <= 0 || V > SPEC_MAX_V) return 0;
  // the header, then the candidate lists of the two-launch select
  return TOPK_WS + topk_list_bytes_for(rows, V);
}

extern "C" int draft_topk_softmax(const void *draft_logits, int dt, int rows, int V,
                                  const int32_t *cu_rows, const float *temperature, int B,
                                  int k, int32_t *out_idx, float *out_prob, void *workspace,
                                  size_t ws_bytes, spec_stream_t stream) {
  if (rows < 0 || B < 0 || V <= 0 || V > SPEC_MAX_V) return SPEC_ERR_INVALID_ARG;
  if (k != SPEC_TOPK) return SPEC_ERR_UNSUPPORTED;
  if (dt != SPEC_F32 && dt != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (cu_rows == nullptr || (B > 0 && temperature == nullptr)) return SPEC_ERR_INVALID_ARG;
  if (rows > 0 && (draft_logits == nullptr || out_idx == nullptr || out_prob == nullptr))
    return SPEC_ERR_INVALID_ARG;
  if (!aligned(draft_logits, 16) || !aligned(cu_rows, 4) || !aligned(temperature, 4) ||
      !aligned(out_idx, 4) || !aligned(out_prob, 4))
    return SPEC_ERR_INVALID_ARG;
  const size_t need = draft_topk_softmax_workspace(rows, V);
  if (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < need)
    return SPEC_ERR_WORKSPACE;
  WsHeader *hdr = static_cast<WsHeader *>(workspace);
  TopkArgs a{};
  a.cu = cu_rows;
  a.temp = temperature;
  a.B = B;
  a.rows_bound = rows;
  a.hdr = hdr;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
#ifdef SPEC_CHECKED
  check_begin(hdr);
  check_add(workspace, need);
  check_add(draft_logits, (unsigned long long)rows * V * (dt == SPEC_BF16 ? 2 : 4));
  check_add(cu_rows, (B + 1) * 4ull);
  check_add(temperature, B * 4ull);
  check_add(out_idx, (unsigned long long)rows * SPEC_TOPK * 4);
  check_add(out_prob, (unsigned long long)rows * SPEC_TOPK * 4);
#endif
  if (check_upload(st) != SPEC_OK) return SPEC_ERR_CUDA;
  k_topk_validate<<<1, 256, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  cudaEvent_t before, after;
  take_row_pass_events(&before, &after);
  return launch_topk128(draft_logits, dt, rows, V, cu_rows, temperature, B, out_idx, out_prob,
                        hdr, st, nullptr, need > TOPK_WS ? static_cast<char *>(workspace) + TOPK_WS
                                                         : nullptr,
                        before, after);
}
