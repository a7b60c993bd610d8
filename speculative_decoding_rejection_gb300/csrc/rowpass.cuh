// Consumer-side arithmetic of the TMA row pass: per-thread running softmax
// statistics over 16 KB shared-memory stages (full packed-bf16 stages, generic
// 16-byte vectors, residual tile pairs and target/draft row pairs). Shared by
// the statistics pass and the streaming verifier.
#pragma once

#include "common.cuh"

namespace sv {

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
  // rank count: only a thread holding a logit above the threshold compares
  // its 32 (the draft token is usually among the largest logits)
  if (RANK && vm > __uint_as_float(thr2 << 16)) {
#pragma unroll
    for (int k = 0; k < VEC_PER_THREAD; ++k)
      st.cnt2 += (bgt2(v[k].x, thr2) & 0x00010001u) + (bgt2(v[k].y, thr2) & 0x00010001u) +
                 (bgt2(v[k].z, thr2) & 0x00010001u) + (bgt2(v[k].w, thr2) & 0x00010001u);
  }
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

// One stage of a single row: full packed-bf16 stages take the fast path,
// partial stages and fp32 rows the generic one. thr is the rank threshold
// (+inf counts nothing: logits are finite or -inf).
template <bool RANK>
__device__ __forceinline__ void consume_row_stage(const unsigned char *buf, int nvec, int e_first,
                                                  float c, bool bf16, float thr, int ctid,
                                                  RunState &st) {
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
}

// The unaligned head and tail elements of a chunk (at most 15 each, counts in
// bits 16-19 and 20-23 of `flags`), taken by one warp with scalar loads.
__device__ __forceinline__ void consume_head_tail(const char *row, int dt, int flags, int head_e,
                                                  int tail_e, float c, float thr, int lane,
                                                  RunState &st) {
  const int head_n = (flags >> 16) & 0xf, tail_n = (flags >> 20) & 0xf;
  if (lane < head_n) scalar_update(load_elem(row, dt, head_e + lane), head_e + lane, c, st, thr);
  if (lane >= 16 && lane - 16 < tail_n)
    scalar_update(load_elem(row, dt, tail_e + lane - 16), tail_e + lane - 16, c, st, thr);
}

// End of a chunk: the warp's statistics merged in a fixed butterfly order
// (every lane gets them); the running state is reset for the next chunk.
template <bool RANK>
__device__ __forceinline__ Part finish_row_chunk(RunState &st, float c) {
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
  st = RunState{NO_MAX, pk2(0.f, 0.f), 0x7fffffff, 0, 0u};
  return Part{m, S, idx, cnt};
}

// The rank count and the row-pair sums need more registers than 6 CTAs per SM
// leave; 5 runs faster than 4 on the CACTUS workload.
constexpr int RS_RANK_CTAS_PER_SM = 5;

}  // namespace sv
