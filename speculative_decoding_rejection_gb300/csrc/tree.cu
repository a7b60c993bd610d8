// Tree verification by recursive rejection sampling without replacement
// ("RheoSampling 2026", §4 "RheoVerification"): at node v the children are
// tested in the order they were drawn (node-index order). Child j with token
// x is accepted with probability min(1, p_j(x)/q_j(x)); on acceptance the
// walk descends into it. On rejection the target law becomes the normalised
// residual p_{j+1} = norm(max(0, p_j - q_j)) and the draft law drops x and is
// renormalised by 1 - q(E) (without replacement). If every child is rejected
// the final token is drawn from the last residual; at an accepted leaf it is a
// bonus draw from that leaf's target law. Greedy trees (T < 0.05) accept the
// first child equal to argmax p_v and otherwise emit argmax p_v.
//
// Point-mass children (spec_verify_tree_ext): a child flagged fixed was not
// drawn from the draft law (a deterministic lead of a RheoSampling tree,
// §3), so its draft law is the point mass on its token. It is accepted with
// probability p_j(x); on rejection p_{j+1} is p_j without x, renormalised by
// 1 - p_j(x) (a scalar: no pass over the rows), and the draft law of the
// drawn children is unchanged.
//
// Uniforms: coin of child c at u(seed, b, c, 0); the final draw at node v at
// u(seed, b, v + 1, 1) (residual) or u(seed, b, v + 1, 2) (bonus), so a chain
// tree reproduces the linear verifier draw for draw.
//
// Pipeline: a one-block-per-tree setup kernel validates every tree and
// writes its child lists (per node: the children in node-index order, each
// with its token, the parent's two logits at that token and its own list);
// then a cluster of CTAs per tree walks it. The walk reads only the rows of
// the nodes it visits (the others never enter the decision): at each visited
// node the cluster first reduces the node's target row (and, for a sampling
// node with children, its draft row) to max / normaliser / argmax, each CTA
// over its vocabulary slice, then tests the children. When the slices fit,
// each CTA copies its slices of the node's rows into shared memory with one
// TMA bulk copy per row as soon as it reaches the node (the node's record
// says whether it has children), loads the children's records meanwhile,
// and every pass over the node (statistics, residuals, the final draw) reads
// shared memory, bf16 slices with packed arithmetic. The residual laws are
// never stored: every pass recomputes
// p_j(y) from p(y) and q(y) through the chain of normalisers, which are
// scalars. A token rejected at step k has q_k > p_k, so p_{k+1} is exactly 0
// there and stays 0; the chain can therefore use q(y) s_j for every y without
// testing membership of the excluded set.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace sv {

// The walk of one tree runs on a cluster of WALK_CLUSTER CTAs. Every CTA
// repeats the walk's scalar decisions (children, node statistics, coins) on
// identical data; each full-row pass is split into contiguous vocabulary
// slices, one per CTA, whose totals are exchanged through distributed shared
// memory. Only the CTA whose slice holds the drawn mass searches it.
constexpr int WALK_THREADS = 256;
constexpr int WALK_CLUSTER = 8;
constexpr int WALK_TILE = WALK_THREADS * SAMPLE_EPT;   // elements per tile of a walk pass
constexpr int MAX_WALK_TILES = (SPEC_MAX_V + WALK_TILE - 1) / WALK_TILE;
constexpr int MAX_SLICE_TILES = (MAX_WALK_TILES + WALK_CLUSTER - 1) / WALK_CLUSTER;
// Largest staged slices (target + draft) per CTA: two walk CTAs per SM keep
// room for their static shared memory.
constexpr size_t WALK_STAGE_MAX = 96 * 1024;

struct TreeInfo {
  int base;        // first node row
  int N;           // nodes
  int mode;        // ReqMode
  float c;         // log2(e)/T
  int root_kids;   // children of the root (its list starts at 0)
  int pad[3];
};

// One child in its parent's list (the setup writes every tree's lists, each
// parent's children contiguous in node-index order): x packs the child's local
// id (bits 0-11), its own number of children (bits 12-18), its point-mass flag
// (bit 19) and the start of its own list (bits 20-31); y is its token; z, w
// the bits of the parent's target and draft logits (or probability) at that
// token, which the child's coin needs (0 in greedy trees).
struct KidRec {
  int x, y;
  float z, w;
};
__device__ __forceinline__ int kid_id(int x) { return x & 0xfff; }
__device__ __forceinline__ int kid_count(int x) { return (x >> 12) & 0x7f; }
__device__ __forceinline__ int kid_fixed(int x) { return (x >> 19) & 1; }
__device__ __forceinline__ int kid_start(int x) { return (int)((unsigned)x >> 20); }
static_assert(SPEC_MAX_TREE_NODES <= 4096 && SPEC_MAX_TREE_BRANCH <= 127,
              "child records pack ids and counts in 12 and 7 bits");

struct TreeArgs {
  const char *target;
  const char *draft;
  int tdt, ddt, dk;
  const int32_t *node_token;
  const int32_t *parent;
  const int32_t *node_fixed;   // optional point-mass flags
  const int32_t *cu;
  const float *temp;
  int B, n_nodes, V, max_depth, max_branch;
  uint64_t seed;
  const uint64_t *seed_dev;   // optional: the seed read on the device at run time
  int32_t *out_tokens, *out_accepted, *out_path;
  WsHeader *hdr;
  TreeInfo *tree;
  KidRec *kids;   // [n_nodes]: every tree's child lists at its node rows
  long long t_row_bytes, d_row_bytes;
  int staged;    // row slices are copied to shared memory
  int dsm_off;   // byte offset of the draft slice in the dynamic shared memory
};

// The call's seed: from device memory when the caller gave a pointer.
__device__ __forceinline__ uint64_t tree_seed(const TreeArgs &a) {
  return a.seed_dev != nullptr ? GLDG(a.seed_dev) : a.seed;
}

struct TreeLayout {
  size_t hdr, tree, kids, total;
};

static TreeLayout tree_layout(int B, int n_nodes) {
  TreeLayout L;
  size_t o = 0;
  L.hdr = o;  o += align256(sizeof(WsHeader));
  L.tree = o; o += align256(sizeof(TreeInfo) * (size_t)B);
  L.kids = o; o += align256(sizeof(KidRec) * (size_t)n_nodes);
  L.total = o;
  return L;
}

// ------------------------------------------------------------------ setup
// One block per tree. The tree's parent ids are staged in shared memory; one
// thread derives depths in topological order, the block counts children and
// checks tokens (in the vocabulary, distinct among drawn siblings). The header
// was cleared before the launch; an invalid tree sets the status word and the
// walk of every tree is skipped. A valid tree's child lists are written for
// the walk: the list starts are an exclusive scan of the child counts, and a
// child's place in its list is the number of its earlier siblings.
constexpr int SETUP_THREADS = 256;

__global__ void __launch_bounds__(SETUP_THREADS) k_setup_tree(const TreeArgs a) {
  __shared__ int s_par[SPEC_MAX_TREE_NODES];
  __shared__ unsigned short s_depth[SPEC_MAX_TREE_NODES];   // depths <= 4095
  __shared__ int s_kids[SPEC_MAX_TREE_NODES];
  __shared__ int s_bad;
  const int b = blockIdx.x, t = threadIdx.x;
  TreeInfo ti;
  ti.base = GLD(a.cu + (b));
  ti.N = GLD(a.cu + (b + 1)) - GLD(a.cu + (b));
  ti.root_kids = 0;
  ti.pad[0] = ti.pad[1] = ti.pad[2] = 0;
  const float T = GLD(a.temp + (b));
  const bool greedy = T < SPEC_GREEDY_T;
  bool ok = (b > 0 || GLD(a.cu + (0)) == 0) && ti.base >= 0 && ti.N >= 1 &&
            ti.N <= SPEC_MAX_TREE_NODES && GLD(a.cu + (b + 1)) <= a.n_nodes && T >= 0.f && isfinite(T);
  if (ok && !greedy && a.draft == nullptr) ok = false;
  if (t == 0) s_bad = !ok;
  __syncthreads();
  if (ok) {
    for (int c = t; c < ti.N; c += SETUP_THREADS) {
      const int p = GLD(a.parent + (ti.base + c));
      s_par[c] = p;
      s_kids[c] = 0;
      const bool good = c == 0 ? p == -1
                               : (p >= 0 && p < c && (unsigned)GLD(a.node_token + (ti.base + c)) <
                                                          (unsigned)a.V);
      if (!good) s_bad = 1;
    }
  }
  __syncthreads();
  if (ok && !s_bad) {
    for (int c = t + 1; c < ti.N; c += SETUP_THREADS) atomicAdd(&s_kids[s_par[c]], 1);
    if (t == 0) {   // depths in topological order (parent[c] < c)
      s_depth[0] = 0;
      int worst = 0;
      for (int c = 1; c < ti.N; ++c) {
        s_depth[c] = (unsigned short)(s_depth[s_par[c]] + 1);
        worst = max(worst, (int)s_depth[c]);
      }
      if (worst > a.max_depth) s_bad = 1;
    }
  }
  __syncthreads();
  if (ok && !s_bad)
    for (int c = t; c < ti.N; c += SETUP_THREADS)
      if (s_kids[c] > a.max_branch) s_bad = 1;
  __syncthreads();
  // the depths are checked: their array now holds each node's list start
  if (ok && !s_bad && t == 0) {
    int start = 0;
    for (int c = 0; c < ti.N; ++c) {
      s_depth[c] = (unsigned short)start;
      start += s_kids[c];
    }
    ti.root_kids = s_kids[0];
  }
  __syncthreads();
  // drawn siblings carry distinct tokens (drawn without replacement); a
  // point-mass child may repeat one. The child counts are no longer needed,
  // so their array holds each node's token, -1 where the node is exempt.
  if (ok && !s_bad)
    for (int c = t; c < ti.N; c += SETUP_THREADS)
      s_kids[c] = (c == 0 || (a.node_fixed != nullptr && GLD(a.node_fixed + (ti.base + c)) != 0))
                      ? -1
                      : GLD(a.node_token + (ti.base + c));
  __syncthreads();
  if (ok && !s_bad)
    for (int c = t + 1; c < ti.N; c += SETUP_THREADS) {
      const int x = s_kids[c], p = s_par[c];
      int rank = 0;   // earlier siblings lie between the parent and c
      for (int o = c - 1; o > p; --o)
        if (s_par[o] == p) {
          ++rank;
          if (x >= 0 && s_kids[o] == x) s_bad = 1;
        }
      // c's record in its parent's list
      const int own = (int)s_depth[c];
      const int n_own = (c + 1 < ti.N ? (int)s_depth[c + 1] : ti.N - 1) - own;
      const int fixed = a.node_fixed != nullptr && GLD(a.node_fixed + (ti.base + c)) != 0;
      const int tok = GLD(a.node_token + (ti.base + c));
      KidRec r;
      r.x = c | (n_own << 12) | (fixed << 19) | (own << 20);
      r.y = tok;
      r.z = 0.f;
      r.w = 0.f;
      if (!greedy) {
        const long long rp = (long long)ti.base + p;
        r.z = load_elem(a.target + rp * a.t_row_bytes, a.tdt, tok);
        r.w = load_elem(a.draft + rp * a.d_row_bytes, a.ddt, tok);
      }
      GST(a.kids + (ti.base + (int)s_depth[p] + rank), r);
    }
  __syncthreads();
  ok = ok && !s_bad;
  ti.mode = ok ? (greedy ? MODE_GREEDY : MODE_SAMPLE) : MODE_SKIP;
  ti.c = (ok && !greedy) ? (float)(1.4426950408889634 / (double)T) : 0.f;
  if (t == 0) {
    GST(a.tree + (b), ti);
    if (!ok) set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);
  }
}

// ------------------------------------------------------------------- walk
struct WalkSmem {
  float tsum[MAX_SLICE_TILES];           // tile totals of this CTA's slice
  float wsum[64 * (WALK_THREADS / 32)];  // per-warp tile sums of one batch
  float zx[2][WALK_CLUSTER];             // every slice's total, pushed by its CTA, by pass parity
  float zall[WALK_CLUSTER];              // every slice's total of the last pass
  float scratch[33];
  // the children of the node being walked, by node parity (the threads decide
  // its coins without a barrier, so a fast one may load the next node's while
  // a slow one still reads these)
  int kids[2][SPEC_MAX_TREE_BRANCH];
  int knext[2][SPEC_MAX_TREE_BRANCH];    // each child's packed record (its own list)
  int kx[2][SPEC_MAX_TREE_BRANCH];       // children's tokens
  int kfix[2][SPEC_MAX_TREE_BRANCH + 1]; // point-mass child (its level of the chain)
  float kzt[2][SPEC_MAX_TREE_BRANCH];    // target logit at each child's token
  float kzd[2][SPEC_MAX_TREE_BRANCH];    // draft logit (or probability) there
  float ucoin[2][SPEC_MAX_TREE_BRANCH];  // the uniform of each child's coin
  float s[SPEC_MAX_TREE_BRANCH + 1];     // 1 / (1 - q(E_j))
  float rinv[SPEC_MAX_TREE_BRANCH + 1];  // 1 / Z_j
  int skip[SPEC_MAX_TREE_BRANCH + 1];    // Z_j == 0: p_{j+1} = p_j
  RowStat wst[WALK_THREADS / 32][2];     // per-warp statistics of a node pass (target, draft)
  RowStat xst[2][WALK_CLUSTER][2];       // every slice's statistics, pushed by its CTA, by pass
                                         // parity (target, draft)
  RowStat node[2];                       // the node's statistics (target, draft)
  uint64_t bar_t, bar_d;                 // completion of the staged target / draft slice
  int jstar, xmin, xlast, rstar, par, ok, go, never;
  float carry, target, Z;
};

struct NodeLaw {        // p(y) = 2^((zt - mt) c) / St, q(y) likewise or given
  const int *kx, *kfix;             // the node's children: tokens, point-mass flags
  const char *trow, *drow;
  const unsigned char *tsm, *dsm;   // this CTA's staged slices, or null
  long long e0;                     // first element of the slice
  bool tvec, dvec;
  float mt, invSt, md, invSd;
};

// SAMPLE_EPT elements x0.. of a row (fill beyond V): from this CTA's staged
// slice, starting at element e0, when `sm` is set, else from global memory.
__device__ __forceinline__ void load_row_ept(const char *row, const unsigned char *sm,
                                             long long e0, int dt, bool vec_ok, int x0, int V,
                                             float fill, float *z) {
  if (sm == nullptr) {
    load_ept(row, dt, vec_ok, x0, V, fill, z);
    return;
  }
  const int esz = dt == SPEC_BF16 ? 2 : 4;
  const unsigned char *p = sm + ((long long)x0 - e0) * esz;
  if (x0 + SAMPLE_EPT <= V) {
    if (dt == SPEC_BF16) {
#pragma unroll
      for (int q = 0; q < SAMPLE_EPT / 8; ++q) {
        const uint4 w = lds128(p + 16 * q);
        z[8 * q + 0] = bf16lo(w.x); z[8 * q + 1] = bf16hi(w.x);
        z[8 * q + 2] = bf16lo(w.y); z[8 * q + 3] = bf16hi(w.y);
        z[8 * q + 4] = bf16lo(w.z); z[8 * q + 5] = bf16hi(w.z);
        z[8 * q + 6] = bf16lo(w.w); z[8 * q + 7] = bf16hi(w.w);
      }
    } else {
#pragma unroll
      for (int q = 0; q < SAMPLE_EPT / 4; ++q) {
        const uint4 w = lds128(p + 16 * q);
        z[4 * q + 0] = __uint_as_float(w.x); z[4 * q + 1] = __uint_as_float(w.y);
        z[4 * q + 2] = __uint_as_float(w.z); z[4 * q + 3] = __uint_as_float(w.w);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k) {
      if (x0 + k >= V) {
        z[k] = fill;
      } else if (dt == SPEC_BF16) {
        z[k] = __uint_as_float((uint32_t)reinterpret_cast<const unsigned short *>(p)[k] << 16);
      } else {
        z[k] = reinterpret_cast<const float *>(p)[k];
      }
    }
  }
}

// Waits for a staged slice; on running out of time records SPEC_ERR_TIMEOUT
// and waits once more (bounded) for the copy in flight before going on.
__device__ __forceinline__ void wait_slice(const TreeArgs &a, WalkSmem &sh, uint64_t *bar,
                                           uint32_t parity) {
  if (!mbar_wait_bounded(bar, parity, &sh.never)) {
    set_status(a.hdr, SPEC_ERR_TIMEOUT, -3);
    mbar_wait_bounded(bar, parity, &sh.never);
  }
}

// Thread 0 copies this CTA's slice [e0, e1) of `row` into `dst`, completion
// on `bar` (one bulk copy: splitting it to reduce pieces as they land
// measured slower).
__device__ __forceinline__ void stage_slice(uint64_t *bar, unsigned char *dst, const char *row,
                                            int esz, long long e0, long long e1) {
  const uint32_t bytes = (uint32_t)((e1 - e0) * esz);
  mbar_arrive_tx(bar, bytes);
  bulk_g2s(dst, row + e0 * esz, bytes, bar);
}

struct Slice { int j0, j1; };   // tiles [j0, j1) of this CTA

__device__ __forceinline__ Slice my_slice(int V, int rank) {
  const int nt = (V + WALK_TILE - 1) / WALK_TILE;
  return Slice{rank * nt / WALK_CLUSTER, (rank + 1) * nt / WALK_CLUSTER};
}

// p_L(y) and the residual max(0, p_L - q_L) (or p_L itself) from the raw
// p(y), q(y) of token y through the chain of normalisers. A point-mass level
// removes its own token and rescales the rest.
__device__ __forceinline__ float chain_weight(float p, float q, int y, int L, bool residual,
                                              const WalkSmem &sh, const NodeLaw &nl) {
  for (int i = 0; i < L; ++i) {
    if (sh.skip[i]) continue;
    p = nl.kfix[i] ? (y == nl.kx[i] ? 0.f : p * sh.rinv[i])
                   : fmaxf(0.f, p - q * sh.s[i]) * sh.rinv[i];
  }
  if (!residual) return p;
  return nl.kfix[L] ? (y == nl.kx[L] ? 0.f : p) : fmaxf(0.f, p - q * sh.s[L]);
}

// p(y) (and q(y)) of the SAMPLE_EPT elements x0.. of a staged bf16 slice,
// two per packed operation: the same roundings per element as the scalar
// form (an exact bf16 widening, then f32 subtract, multiply, 2^x, multiply).
__device__ __forceinline__ void staged_law_bf16(const unsigned char *sm, long long e0, int x0,
                                                float m, float c, float inv, float *out) {
  const unsigned char *p = sm + ((long long)x0 - e0) * 2;
  const f32x2 c2 = pk2(c, c), i2 = pk2(inv, inv);
#pragma unroll
  for (int h = 0; h < SAMPLE_EPT / 8; ++h) {
    const uint4 v = lds128(p + 16 * h);
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const f32x2 t = mul2(bsub2(wv[q], m), c2);
      const f32x2 e = mul2(pk2(ex2(lo2(t)), ex2(hi2(t))), i2);
      out[8 * h + 2 * q] = lo2(e);
      out[8 * h + 2 * q + 1] = hi2(e);
    }
  }
}

template <int DK>
__device__ __forceinline__ void tile_weights_tree(const TreeArgs &a, const WalkSmem &sh,
                                                  const NodeLaw &nl, float c, int L,
                                                  bool residual, int j, float *w) {
  const int x0 = j * WALK_TILE + (int)threadIdx.x * SAMPLE_EPT;
  const bool full = x0 + SAMPLE_EPT <= a.V;
  if (full && nl.tsm != nullptr && a.tdt == SPEC_BF16) {
    staged_law_bf16(nl.tsm, nl.e0, x0, nl.mt, c, nl.invSt, w);
  } else {
    float zt[SAMPLE_EPT];
    load_row_ept(nl.trow, nl.tsm, nl.e0, a.tdt, nl.tvec, x0, a.V, -INFINITY, zt);
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k) w[k] = ex2((zt[k] - nl.mt) * c) * nl.invSt;
  }
  if (L == 0 && !residual) return;
  float q[SAMPLE_EPT];
  if (DK == SPEC_DRAFT_LOGITS && full && nl.dsm != nullptr && a.ddt == SPEC_BF16) {
    staged_law_bf16(nl.dsm, nl.e0, x0, nl.md, c, nl.invSd, q);
  } else {
    float zd[SAMPLE_EPT];
    load_row_ept(nl.drow, nl.dsm, nl.e0, a.ddt, nl.dvec, x0, a.V,
                 DK == SPEC_DRAFT_PROBS ? 0.f : -INFINITY, zd);
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k)
      q[k] = DK == SPEC_DRAFT_PROBS ? zd[k] : ex2((zd[k] - nl.md) * c) * nl.invSd;
  }
  // the chain level by level over all elements (the same operations per
  // element as chain_weight, so the same bits)
  for (int i = 0; i < L; ++i) {
    if (sh.skip[i]) continue;
    const float si = sh.s[i], ri = sh.rinv[i];
    if (nl.kfix[i]) {
      const int xi = nl.kx[i];
#pragma unroll
      for (int k = 0; k < SAMPLE_EPT; ++k) w[k] = x0 + k == xi ? 0.f : w[k] * ri;
    } else {
#pragma unroll
      for (int k = 0; k < SAMPLE_EPT; ++k) w[k] = fmaxf(0.f, w[k] - q[k] * si) * ri;
    }
  }
  if (residual) {
    if (nl.kfix[L]) {
      const int xL = nl.kx[L];
#pragma unroll
      for (int k = 0; k < SAMPLE_EPT; ++k) w[k] = x0 + k == xL ? 0.f : w[k];
    } else {
      const float sL = sh.s[L];
#pragma unroll
      for (int k = 0; k < SAMPLE_EPT; ++k) w[k] = fmaxf(0.f, w[k] - q[k] * sL);
    }
  }
}

// One pass over the node's rows: this CTA's tile totals of the level-L
// weights into sh.tsum, the slice totals of the whole cluster into sh.zall
// and their sum (ascending slice order, the same in every CTA) into sh.Z.
template <int DK>
__device__ void weight_pass(const TreeArgs &a, WalkSmem &sh, const NodeLaw &nl, float c, int L,
                            bool residual, const Slice sl, cg::cluster_group &cluster) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float w[SAMPLE_EPT];
  for (int j0 = sl.j0; j0 < sl.j1; j0 += 64) {
    const int j1 = min(sl.j1, j0 + 64);
#pragma unroll 2
    for (int j = j0; j < j1; ++j) {
      tile_weights_tree<DK>(a, sh, nl, c, L, residual, j, w);
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < SAMPLE_EPT; ++k) s += w[k];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) sh.wsum[(j - j0) * (WALK_THREADS / 32) + warp] = s;
    }
    __syncthreads();
    if (threadIdx.x < j1 - j0) {
      float t = 0.f;
      for (int q = 0; q < WALK_THREADS / 32; ++q)
        t += sh.wsum[threadIdx.x * (WALK_THREADS / 32) + q];
      sh.tsum[j0 + threadIdx.x - sl.j0] = t;
    }
    __syncthreads();
  }
  const int par = sh.par;
  if (threadIdx.x < WALK_CLUSTER) {   // this slice's total into every CTA's slot for it
    float Zr = 0.f;
    for (int j = sl.j0; j < sl.j1; ++j) Zr += sh.tsum[j - sl.j0];
    *cluster.map_shared_rank(&sh.zx[par][cluster.block_rank()], (int)threadIdx.x) = Zr;
  }
  cluster.sync();   // every slice total pushed (slots alternate by parity)
  if (threadIdx.x == 0) {
    float Z = 0.f;
    for (int r = 0; r < WALK_CLUSTER; ++r) {
      sh.zall[r] = sh.zx[par][r];
      Z += sh.zall[r];
    }
    sh.Z = Z;
    sh.par = par ^ 1;
  }
  __syncthreads();
}

// Inverse-CDF draw at u from the level-L weights of the last pass: the slice
// holding u*Z is found from the slice totals, then its tile, then the element
// (smallest y with u*Z < C_y; the last positive weight if rounding leaves
// none). Returns the token in the CTA that owns it, -1 in the others.
template <int DK>
__device__ int weight_draw(const TreeArgs &a, WalkSmem &sh, const NodeLaw &nl, float c, int L,
                           bool residual, float u, const Slice sl, int rank) {
  if (threadIdx.x == 0) {
    sh.target = u * sh.Z;
    float carry = 0.f;
    int rs = -1;
    for (int r = 0; r < WALK_CLUSTER; ++r) {
      const float nc = carry + sh.zall[r];
      if (nc > sh.target) { rs = r; break; }
      carry = nc;
    }
    if (rs < 0) {
      carry = 0.f;
      for (int r = 0; r < WALK_CLUSTER; ++r)
        if (sh.zall[r] > 0.f) rs = r;
      for (int r = 0; r < rs; ++r) carry += sh.zall[r];
    }
    sh.rstar = rs;
    sh.carry = carry;
  }
  __syncthreads();
  // with no mass anywhere, rank 0 reports it
  if (sh.rstar != rank && !(sh.rstar < 0 && rank == 0)) return -1;
  if (threadIdx.x == 0) {
    float carry = sh.carry;
    int js = -1;
    for (int j = sl.j0; j < sl.j1; ++j) {
      const float nc = carry + sh.tsum[j - sl.j0];
      if (nc > sh.target) { js = j; break; }
      carry = nc;
    }
    if (js < 0) {
      carry = sh.carry;
      for (int j = sl.j0; j < sl.j1; ++j)
        if (sh.tsum[j - sl.j0] > 0.f) js = j;
      for (int j = sl.j0; j < js; ++j) carry += sh.tsum[j - sl.j0];
    }
    sh.jstar = js;
    sh.carry = carry;
    sh.xmin = 0x7fffffff;
    sh.xlast = -1;
  }
  __syncthreads();
  const int js = sh.jstar;
  if (js >= 0) {
    float w[SAMPLE_EPT];
    tile_weights_tree<DK>(a, sh, nl, c, L, residual, js, w);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k) s += w[k];
    float tot;
    const float excl = block_excl_scan(s, sh.scratch, &tot);
    const int x0 = js * WALK_TILE + (int)threadIdx.x * SAMPLE_EPT;
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
  int x = sh.xmin != 0x7fffffff ? sh.xmin : sh.xlast;
  if (x < 0) x = 0x7fffffff;   // owner found no mass: reported as invalid below
  __syncthreads();
  return x;
}

// Running statistics of SAMPLE_EPT consecutive logits into (m, S, idx):
// max, sum of 2^((z - m) c) (none when c is 0), lowest index of the max.
__device__ __forceinline__ void stat_update(const float *z, int x0, float c, float &m, float &S,
                                            int &idx) {
  float vm = z[0];
  int j = 0;
#pragma unroll
  for (int k = 1; k < SAMPLE_EPT; ++k)
    if (z[k] > vm) { vm = z[k]; j = k; }
  if (vm > m) {
    if (c != 0.f) S *= ex2((m - vm) * c);
    m = vm;
    idx = x0 + j;
  }
  if (c != 0.f) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < SAMPLE_EPT; ++k) t += ex2((z[k] - m) * c);
    S += t;
  }
}

// Running max of one thread's vectors of a staged bf16 slice (vectors t,
// t + WALK_THREADS, ... < nv) through packed bf16 maxima, and the first
// vector holding it (-1: nothing finite).
__device__ __forceinline__ void slice_max_bf16(const unsigned char *sm, int v, int nv, float &vm,
                                               int &vb) {
  for (; v < nv; v += WALK_THREADS) {
    const uint4 w = lds128(sm + 16 * (size_t)v);
    const uint32_t a2 = bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w));
    const float x = fmaxf(bf16lo(a2), bf16hi(a2));
    if (x > vm) {
      vm = x;
      vb = v;
    }
  }
}

// Lowest element index holding vm in vector vb.
__device__ __forceinline__ int first_in_vec(const unsigned char *sm, int vb, float vm,
                                            long long e0) {
  const uint4 w = lds128(sm + 16 * (size_t)vb);
  const uint32_t q[4] = {w.x, w.y, w.z, w.w};
  int jb = 7;
#pragma unroll
  for (int k = 7; k >= 0; --k)
    if (((k & 1) ? bf16hi(q[k >> 1]) : bf16lo(q[k >> 1])) == vm) jb = k;
  return (int)(e0 + 8LL * vb + jb);
}

// Sum of 2^((z - m) c) over the 8 elements of one vector, as packed pairs.
__device__ __forceinline__ f32x2 vec_exp_sum(const uint4 w, float m, f32x2 c2) {
  const f32x2 t0 = mul2(bsub2(w.x, m), c2), t1 = mul2(bsub2(w.y, m), c2);
  const f32x2 t2 = mul2(bsub2(w.z, m), c2), t3 = mul2(bsub2(w.w, m), c2);
  const f32x2 s01 = add2(pk2(ex2(lo2(t0)), ex2(hi2(t0))), pk2(ex2(lo2(t1)), ex2(hi2(t1))));
  const f32x2 s23 = add2(pk2(ex2(lo2(t2)), ex2(hi2(t2))), pk2(ex2(lo2(t3)), ex2(hi2(t3))));
  return add2(s01, s23);
}

// One thread's statistics of the staged bf16 slices of a node's target row
// and, when `dsm` is set, its draft row (nv 16-byte vectors each, element e0
// first; vectors t, t + WALK_THREADS, ...): per row the max through packed
// bf16 maxima and its lowest index, then the sum of 2^((z - max) c) (none
// when c is 0), the two rows' vectors taken in the same loop so their
// loads and 2^x overlap.
__device__ __forceinline__ void slice_stats_bf16(const unsigned char *tsm,
                                                 const unsigned char *dsm, int nv, long long e0,
                                                 float c, RowStat &t, RowStat &d) {
  const int v0 = (int)threadIdx.x;
  float tm = NO_MAX, dm = NO_MAX;
  int tb = -1, db = -1;
  slice_max_bf16(tsm, v0, nv, tm, tb);
  if (dsm != nullptr) slice_max_bf16(dsm, v0, nv, dm, db);
  t = RowStat{NO_MAX, 0.f, 0x7fffffff};
  d = RowStat{NO_MAX, 0.f, 0x7fffffff};
  if (tb >= 0) t = RowStat{tm, 0.f, first_in_vec(tsm, tb, tm, e0)};
  if (db >= 0) d = RowStat{dm, 0.f, first_in_vec(dsm, db, dm, e0)};
  if (c == 0.f) return;
  const f32x2 c2 = pk2(c, c);
  f32x2 at = pk2(0.f, 0.f), ad = pk2(0.f, 0.f);
  if (dsm != nullptr && tb >= 0 && db >= 0) {
    for (int v = v0; v < nv; v += WALK_THREADS) {
      const uint4 wt = lds128(tsm + 16 * (size_t)v);
      const uint4 wd = lds128(dsm + 16 * (size_t)v);
      at = add2(at, vec_exp_sum(wt, tm, c2));
      ad = add2(ad, vec_exp_sum(wd, dm, c2));
    }
  } else {
    if (tb >= 0)
      for (int v = v0; v < nv; v += WALK_THREADS)
        at = add2(at, vec_exp_sum(lds128(tsm + 16 * (size_t)v), tm, c2));
    if (dsm != nullptr && db >= 0)
      for (int v = v0; v < nv; v += WALK_THREADS)
        ad = add2(ad, vec_exp_sum(lds128(dsm + 16 * (size_t)v), dm, c2));
  }
  t.S = lo2(at) + hi2(at);
  d.S = lo2(ad) + hi2(ad);
}

// Statistics of node rows computed by the cluster: every CTA reduces its
// vocabulary slice of the target row (and, when `drow` is set, of the draft
// row), the slices are exchanged through distributed shared memory and merged
// in rank order, so every CTA gets the same bits. Only the rows of nodes the
// walk visits are read.
__device__ void node_stats(const TreeArgs &a, WalkSmem &sh, const char *trow, const char *drow,
                           const unsigned char *tsm, const unsigned char *dsm, uint32_t pt,
                           uint32_t pd, float c, const Slice sl, cg::cluster_group &cluster,
                           RowStat &ts, RowStat &ds) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool tvec = ((uintptr_t)trow & 15) == 0, dvec = drow && ((uintptr_t)drow & 15) == 0;
  const long long e0 = (long long)sl.j0 * WALK_TILE;
  float m = NO_MAX, S = 0.f, md = NO_MAX, Sd = 0.f;
  int idx = 0x7fffffff, idd = 0x7fffffff;
  if (tsm != nullptr) wait_slice(a, sh, &sh.bar_t, pt);
  if (drow && dsm != nullptr) wait_slice(a, sh, &sh.bar_d, pd);
  if (tsm != nullptr && a.tdt == SPEC_BF16 &&
      (drow == nullptr || (dsm != nullptr && a.ddt == SPEC_BF16))) {
    // staged bf16 slices (whole 16-byte vectors: staging needs V % 8 == 0)
    const int nv = (int)((min((long long)sl.j1 * WALK_TILE, (long long)a.V) - e0) / 8);
    RowStat t, d;
    slice_stats_bf16(tsm, drow ? dsm : nullptr, nv, e0, c, t, d);
    m = t.m;
    S = t.S;
    idx = t.idx;
    md = d.m;
    Sd = d.S;
    idd = d.idx;
  } else {
    float z[SAMPLE_EPT];
#pragma unroll 2
    for (int j = sl.j0; j < sl.j1; ++j) {
      const int x0 = j * WALK_TILE + (int)threadIdx.x * SAMPLE_EPT;
      load_row_ept(trow, tsm, e0, a.tdt, tvec, x0, a.V, -INFINITY, z);
      stat_update(z, x0, c, m, S, idx);
      if (drow) {
        load_row_ept(drow, dsm, e0, a.ddt, dvec, x0, a.V, -INFINITY, z);
        stat_update(z, x0, c, md, Sd, idd);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float S2 = __shfl_xor_sync(0xffffffffu, S, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    merge_stat(m, S, idx, m2, S2, i2, c);
    const float md2 = __shfl_xor_sync(0xffffffffu, md, o);
    const float Sd2 = __shfl_xor_sync(0xffffffffu, Sd, o);
    const int id2 = __shfl_xor_sync(0xffffffffu, idd, o);
    merge_stat(md, Sd, idd, md2, Sd2, id2, c);
  }
  if (lane == 0) {
    sh.wst[warp][0] = RowStat{m, S, idx};
    sh.wst[warp][1] = RowStat{md, Sd, idd};
  }
  __syncthreads();
  const int par = sh.par;
  if (threadIdx.x < 2 * WALK_CLUSTER) {
    // this slice's statistics of row r (0: target, 1: draft) into CTA k's slot
    // for them; the 8 threads of a row merge the warps in the same order
    const int r = threadIdx.x & 1, k = threadIdx.x >> 1;
    RowStat q{NO_MAX, 0.f, 0x7fffffff};
    for (int w = 0; w < WALK_THREADS / 32; ++w)
      merge_stat(q.m, q.S, q.idx, sh.wst[w][r].m, sh.wst[w][r].S, sh.wst[w][r].idx, c);
    *cluster.map_shared_rank(&sh.xst[par][cluster.block_rank()][r], k) = q;
  }
  cluster.sync();   // every slice's statistics pushed (slots alternate by parity)
  if (threadIdx.x < 2) {
    const int r = threadIdx.x;
    RowStat q{NO_MAX, 0.f, 0x7fffffff};
    for (int k = 0; k < WALK_CLUSTER; ++k)
      merge_stat(q.m, q.S, q.idx, sh.xst[par][k][r].m, sh.xst[par][k][r].S, sh.xst[par][k][r].idx,
                 c);
    sh.node[r] = q;
  }
  __syncthreads();
  if (threadIdx.x == 0) sh.par = par ^ 1;
  ts = sh.node[0];
  ds = sh.node[1];
}

__device__ __forceinline__ void write_final(const TreeArgs &a, int b, int depth, int x) {
  if (x == 0x7fffffff) {
    set_status(a.hdr, SPEC_ERR_INVALID_ARG, b);   // a row without mass
    x = -1;
  }
  GST(a.out_tokens + ((long long)b * (a.max_depth + 1) + depth), x);
}

// The walk of tree b on the CTA of cluster rank `rank`. Every exit of this
// function is followed by the kernel's closing cluster barrier, so no CTA
// leaves while another may still read its slice totals.
template <int DK>
__device__ __forceinline__ void walk_tree(const TreeArgs &a, WalkSmem &sh, const TreeInfo &t,
                                          int b, int rank, cg::cluster_group &cluster,
                                          unsigned char *tsm, unsigned char *dsm) {
  const int W = a.max_depth + 1;
  const Slice sl = my_slice(a.V, rank);
  int32_t *out = a.out_tokens + (long long)b * W;
  int32_t *path = a.out_path ? a.out_path + (long long)b * W : nullptr;
  const float c = t.c;
  int v = 0, depth = 0;
  const int esz_t = dtype_size(a.tdt), esz_d = dtype_size(a.ddt);
  const long long se0 = (long long)sl.j0 * WALK_TILE;
  const long long se1 = min((long long)sl.j1 * WALK_TILE, (long long)a.V);
  const bool has_slice = sl.j1 > sl.j0;
  if (!has_slice) tsm = dsm = nullptr;
  uint32_t pt = 0, pd = 0;   // phases of the staged-slice barriers
  int kst = 0, nk = t.root_kids;   // the current node's child list: start, length
  int kb = 0;                      // the node's children buffer (node parity)
  while (true) {
    const long long rv = t.base + v;
    const int row = t.base + v;
    // a sampling node with children tests them against its draft row
    const bool use_d = t.mode != MODE_GREEDY && nk > 0;
    const bool stage_d = dsm != nullptr && use_d;
    // this CTA's slices of node v's rows into shared memory (or L2) first,
    // so the copies overlap the loads of the children
    if (threadIdx.x == 0 && has_slice) {
      if (tsm != nullptr) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        stage_slice(&sh.bar_t, tsm, a.target + rv * a.t_row_bytes, esz_t, se0, se1);
        if (stage_d) stage_slice(&sh.bar_d, dsm, a.draft + rv * a.d_row_bytes, esz_d, se0, se1);
      } else {
        prefetch_l2(a.target + rv * a.t_row_bytes + se0 * esz_t, (se1 - se0) * esz_t);
      }
      if (!stage_d && use_d && a.draft != nullptr)
        prefetch_l2(a.draft + rv * a.d_row_bytes + se0 * esz_d, (se1 - se0) * esz_d);
    }
    // the children in node-index order, with the logits and the uniforms
    // their coins need, one thread each (read after the statistics' barriers)
    if ((int)threadIdx.x < nk) {
      const int j = threadIdx.x;
      const KidRec r = GLD(a.kids + (t.base + kst + j));
      sh.kids[kb][j] = kid_id(r.x);
      sh.knext[kb][j] = r.x;
      sh.kx[kb][j] = r.y;
      sh.kfix[kb][j] = kid_fixed(r.x);
      sh.kzt[kb][j] = r.z;
      sh.kzd[kb][j] = r.w;
      sh.ucoin[kb][j] = uniform24(tree_seed(a), (uint32_t)b, (uint32_t)kid_id(r.x), 0);
    }
    // the node's statistics: its target row, and its draft row when a
    // sampling node has children to test
    const char *trow = a.target + (long long)row * a.t_row_bytes;
    const bool want_d = use_d && DK == SPEC_DRAFT_LOGITS;
    RowStat ts, dstat;
    node_stats(a, sh, trow, want_d ? a.draft + (long long)row * a.d_row_bytes : nullptr, tsm,
               want_d ? dsm : nullptr, pt, pd, c, sl, cluster, ts, dstat);
    if (tsm != nullptr) pt ^= 1;
    if (stage_d && !want_d) wait_slice(a, sh, &sh.bar_d, pd);   // draft probabilities
    if (stage_d) pd ^= 1;
    if (t.mode == MODE_GREEDY) {   // every thread finds the same child
      int ac = -1, anext = 0;
      for (int j = 0; j < nk; ++j)
        if (sh.kx[kb][j] == ts.idx) {
          ac = sh.kids[kb][j];
          anext = sh.knext[kb][j];
          break;
        }
      if (ac >= 0 && depth < a.max_depth) {
        if (rank == 0 && threadIdx.x == 0) {
          GST(out + depth, ts.idx);   // the accepted child's token is the argmax
          if (path) GST(path + depth, ac);
        }
        v = ac;
        ++depth;
        kst = kid_start(anext);
        nk = kid_count(anext);
        kb ^= 1;
        continue;
      }
      if (rank == 0 && threadIdx.x == 0) {
        GST(out + depth, ts.idx);
        GST(a.out_accepted + (b), depth);
      }
      return;
    }
    NodeLaw nl;
    nl.kx = sh.kx[kb];
    nl.kfix = sh.kfix[kb];
    nl.trow = trow;
    nl.tsm = tsm;
    nl.dsm = stage_d ? dsm : nullptr;
    nl.e0 = se0;
    nl.tvec = ((uintptr_t)nl.trow & 15) == 0;
    nl.mt = ts.m;
    nl.invSt = 1.f / ts.S;
    nl.drow = nullptr;
    nl.dvec = false;
    nl.md = 0.f;
    nl.invSd = 0.f;
    if (nk == 0) {  // accepted leaf (or a bare root): bonus draw from p_v
      weight_pass<DK>(a, sh, nl, c, 0, false, sl, cluster);
      const int x = weight_draw<DK>(a, sh, nl, c, 0, false,
                                    uniform24(tree_seed(a), (uint32_t)b, (uint32_t)(v + 1), 2), sl,
                                    rank);
      if (x != -1 && threadIdx.x == 0) write_final(a, b, depth, x);
      if (rank == 0 && threadIdx.x == 0) GST(a.out_accepted + (b), depth);
      return;
    }
    nl.drow = a.draft + (long long)row * a.d_row_bytes;
    nl.dvec = ((uintptr_t)nl.drow & 15) == 0;
    if (DK == SPEC_DRAFT_LOGITS) {
      nl.md = dstat.m;
      nl.invSd = 1.f / dstat.S;
    }
    float qE = 0.f;
    int accepted = -1, acc_next = 0, acc_tok = -1, L = 0;
    bool passed = false;   // the tile totals of level L's residual are in sh
    for (int j = 0; j < nk; ++j) {
      // coin of child j at its token x, with p_j(x) and q_j(x) from the chain
      // (a point mass has q_j(x) = 1), taken by every thread on the same
      // shared values
      const float p = ex2((sh.kzt[kb][j] - nl.mt) * c) * nl.invSt;
      const float qx = DK == SPEC_DRAFT_PROBS ? sh.kzd[kb][j]
                                              : ex2((sh.kzd[kb][j] - nl.md) * c) * nl.invSd;
      const float pj = chain_weight(p, qx, sh.kx[kb][j], j, false, sh, nl);
      const float qj = sh.kfix[kb][j] ? 1.f : qx * sh.s[j];
      const float acc = qj <= pj ? 1.f : pj / qj;
      if (sh.ucoin[kb][j] < acc) {
        accepted = sh.kids[kb][j];
        acc_next = sh.knext[kb][j];
        acc_tok = sh.kx[kb][j];
        break;
      }
      if (sh.kfix[kb][j]) {
        // point-mass rejection: p_{j+1} = p_j without x over Z_j = 1 - p_j(x)
        L = j;
        passed = false;
        if (threadIdx.x == 0) {
          const float Zf = 1.f - pj;
          sh.skip[j] = !(Zf > 0.f);
          sh.rinv[j] = Zf > 0.f ? 1.f / Zf : 1.f;
          sh.s[j + 1] = sh.s[j];
        }
        __syncthreads();
        continue;
      }
      // rejection: Z_j of the residual at level j (tile totals kept for a
      // possible final draw), then the next draft normaliser
      weight_pass<DK>(a, sh, nl, c, j, true, sl, cluster);
      L = j;
      passed = true;
      qE += qx;
      const float left = 1.f - qE;
      if (threadIdx.x == 0) {
        sh.skip[j] = !(sh.Z > 0.f);
        sh.rinv[j] = sh.Z > 0.f ? 1.f / sh.Z : 1.f;
        sh.s[j + 1] = left > 0.f ? 1.f / left : 0.f;
      }
      __syncthreads();
      if (!(left > 0.f)) break;   // every draft token used up
    }
    if (accepted >= 0 && depth < a.max_depth) {
      if (rank == 0 && threadIdx.x == 0) {
        GST(out + depth, acc_tok);
        if (path) GST(path + depth, accepted);
      }
      v = accepted;
      ++depth;
      kst = kid_start(acc_next);
      nk = kid_count(acc_next);
      kb ^= 1;
      continue;
    }
    // all tested children rejected: draw from p_{L+1} = norm(residual at L),
    // or from p_L itself when that residual had no mass
    bool residual = true;
    if (sh.skip[L]) {
      residual = false;
      weight_pass<DK>(a, sh, nl, c, L, false, sl, cluster);
    } else if (!passed) {   // the last rejection was a point mass: no pass yet
      weight_pass<DK>(a, sh, nl, c, L, true, sl, cluster);
    }
    const int x = weight_draw<DK>(a, sh, nl, c, L, residual,
                                  uniform24(tree_seed(a), (uint32_t)b, (uint32_t)(v + 1), 1), sl, rank);
    if (x != -1 && threadIdx.x == 0) write_final(a, b, depth, x);
    if (rank == 0 && threadIdx.x == 0) GST(a.out_accepted + (b), depth);
    return;
  }
}

template <int DK>
__global__ void __cluster_dims__(WALK_CLUSTER, 1, 1) __launch_bounds__(WALK_THREADS, 2)
    k_tree_walk(const TreeArgs a) {
  __shared__ WalkSmem sh;
  extern __shared__ __align__(16) unsigned char rows_sm[];
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / WALK_CLUSTER;
  const TreeInfo t = GLD(a.tree + (b));
  const int W = a.max_depth + 1;
  if (rank == 0)
    for (int j = threadIdx.x; j < W; j += blockDim.x) {
      GST(a.out_tokens + ((long long)b * W + j), -1);
      if (a.out_path) GST(a.out_path + ((long long)b * W + j), -1);
    }
  // Whether to walk is decided once for the whole cluster: the status word
  // can change under a running walk (another tree without mass), so each CTA
  // reads it and the CTAs agree on the conjunction.
  if (threadIdx.x == 0) {
    sh.ok = t.mode != MODE_SKIP && *(volatile int *)&a.hdr->status == SPEC_OK;
    sh.par = 0;
    sh.never = 0;
    sh.s[0] = 1.f;   // level 0 of the draft law is q itself
    mbar_init(&sh.bar_t, 1);
    mbar_init(&sh.bar_d, 1);
    fence_mbar_init();
  }
  cluster.sync();   // also orders the -1 fill before every later token write
  if (threadIdx.x == 0) {
    int all = 1;
    for (int r = 0; r < WALK_CLUSTER; ++r) all &= *cluster.map_shared_rank(&sh.ok, r);
    sh.go = all;
  }
  __syncthreads();
  if (sh.go)
    walk_tree<DK>(a, sh, t, b, rank, cluster, a.staged ? rows_sm : nullptr,
                  a.staged ? rows_sm + a.dsm_off : nullptr);
  else if (rank == 0 && threadIdx.x == 0)
    GST(a.out_accepted + (b), -1);
  cluster.sync();
}

}  // namespace sv

using namespace sv;

extern "C" size_t spec_verify_tree_workspace(int B, int n_nodes, int V, int max_depth,
                                             int max_branch) {
  if (B < 0 || n_nodes < B || V <= 0 || V > SPEC_MAX_V) return 0;
  if (max_depth < 0 || max_depth > SPEC_MAX_TREE_DEPTH) return 0;
  if (max_branch < 1 || max_branch > SPEC_MAX_TREE_BRANCH) return 0;
  return tree_layout(B, n_nodes).total;
}

static int verify_tree(const void *target, int tdt, const void *draft, int ddt, int dk,
                       const int32_t *node_token, const int32_t *parent,
                       const int32_t *node_fixed, const int32_t *cu_nodes,
                       const float *temperature, int B, int n_nodes, int V, int max_depth,
                       int max_branch, uint64_t seed, const uint64_t *seed_dev,
                       int32_t *out_tokens, int32_t *out_accepted, int32_t *out_path,
                       void *workspace, size_t ws_bytes, spec_stream_t stream) {
  if (B < 0 || n_nodes < B || V <= 0 || V > SPEC_MAX_V) return SPEC_ERR_INVALID_ARG;
  if (max_depth < 0 || max_branch < 1) return SPEC_ERR_INVALID_ARG;
  if (max_depth > SPEC_MAX_TREE_DEPTH || max_branch > SPEC_MAX_TREE_BRANCH)
    return SPEC_ERR_UNSUPPORTED;
  if ((tdt != SPEC_F32 && tdt != SPEC_BF16) || (ddt != SPEC_F32 && ddt != SPEC_BF16))
    return SPEC_ERR_INVALID_ARG;
  if (dk != SPEC_DRAFT_LOGITS && dk != SPEC_DRAFT_PROBS) return SPEC_ERR_INVALID_ARG;
  if (B > 0 && (target == nullptr || node_token == nullptr || parent == nullptr ||
                cu_nodes == nullptr || temperature == nullptr || out_tokens == nullptr ||
                out_accepted == nullptr))
    return SPEC_ERR_INVALID_ARG;
  if (!aligned(target, 16) || !aligned(draft, 16) || !aligned(node_token, 4) ||
      !aligned(parent, 4) || !aligned(cu_nodes, 4) || !aligned(temperature, 4) ||
      !aligned(out_tokens, 4) || !aligned(out_accepted, 4) || !aligned(out_path, 4) ||
      !aligned(node_fixed, 4) || !aligned(seed_dev, 8))
    return SPEC_ERR_INVALID_ARG;
  const TreeLayout L = tree_layout(B, n_nodes);
  if (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < L.total)
    return SPEC_ERR_WORKSPACE;
  char *ws = static_cast<char *>(workspace);
  TreeArgs a;
  a.target = static_cast<const char *>(target);
  a.draft = static_cast<const char *>(draft);
  a.tdt = tdt;
  a.ddt = ddt;
  a.dk = dk;
  a.node_token = node_token;
  a.parent = parent;
  a.node_fixed = node_fixed;
  a.cu = cu_nodes;
  a.temp = temperature;
  a.B = B;
  a.n_nodes = n_nodes;
  a.V = V;
  a.max_depth = max_depth;
  a.max_branch = max_branch;
  a.seed = seed;
  a.seed_dev = seed_dev;
  a.out_tokens = out_tokens;
  a.out_accepted = out_accepted;
  a.out_path = out_path;
  a.hdr = reinterpret_cast<WsHeader *>(ws + L.hdr);
  a.tree = reinterpret_cast<TreeInfo *>(ws + L.tree);
  a.kids = reinterpret_cast<KidRec *>(ws + L.kids);
  a.t_row_bytes = (long long)V * (tdt == SPEC_BF16 ? 2 : 4);
  a.d_row_bytes = (long long)V * (ddt == SPEC_BF16 ? 2 : 4);
  // stage the row slices in shared memory when they fit and every slice
  // copy starts and ends on 16-byte boundaries
  const long long slice_elems =
      (long long)((V + WALK_TILE - 1) / WALK_TILE + WALK_CLUSTER - 1) / WALK_CLUSTER * WALK_TILE;
  const size_t t_stage = ((size_t)slice_elems * (tdt == SPEC_BF16 ? 2 : 4) + 15) & ~(size_t)15;
  const size_t d_stage = draft ? (size_t)slice_elems * (ddt == SPEC_BF16 ? 2 : 4) : 0;
  a.staged = t_stage + d_stage <= WALK_STAGE_MAX && a.t_row_bytes % 16 == 0 &&
             (draft == nullptr || a.d_row_bytes % 16 == 0);
  a.dsm_off = (int)t_stage;
  const size_t smem = a.staged ? t_stage + d_stage : 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(a.hdr, 0, sizeof(WsHeader), st) != cudaSuccess) return SPEC_ERR_CUDA;
  if (B == 0) return SPEC_OK;
#ifdef SPEC_CHECKED
  check_begin(a.hdr);
  check_add(workspace, L.total);
  check_add(target, (unsigned long long)n_nodes * a.t_row_bytes);
  check_add(draft, (unsigned long long)n_nodes * a.d_row_bytes);
  check_add(node_token, n_nodes * 4ull);
  check_add(parent, n_nodes * 4ull);
  check_add(node_fixed, n_nodes * 4ull);
  check_add(cu_nodes, (B + 1) * 4ull);
  check_add(temperature, B * 4ull);
  check_add(out_tokens, (unsigned long long)B * (max_depth + 1) * 4);
  check_add(out_accepted, B * 4ull);
  check_add(out_path, (unsigned long long)B * (max_depth + 1) * 4);
  check_add(seed_dev, 8);
#endif
  if (check_upload(st) != SPEC_OK) return SPEC_ERR_CUDA;
  k_setup_tree<<<B, SETUP_THREADS, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  // profiling events, if registered, bracket the walk
  cudaEvent_t before, after;
  take_row_pass_events(&before, &after);
  if (before && cudaEventRecord(before, st) != cudaSuccess) return SPEC_ERR_CUDA;
  if (dk == SPEC_DRAFT_PROBS) {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(k_tree_walk<SPEC_DRAFT_PROBS>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return SPEC_ERR_CUDA;
    k_tree_walk<SPEC_DRAFT_PROBS><<<B * WALK_CLUSTER, WALK_THREADS, smem, st>>>(a);
  } else {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(k_tree_walk<SPEC_DRAFT_LOGITS>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return SPEC_ERR_CUDA;
    k_tree_walk<SPEC_DRAFT_LOGITS><<<B * WALK_CLUSTER, WALK_THREADS, smem, st>>>(a);
  }
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  if (after && cudaEventRecord(after, st) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

extern "C" int spec_verify_tree(const void *target, int tdt, const void *draft, int ddt, int dk,
                                const int32_t *node_token, const int32_t *parent,
                                const int32_t *cu_nodes, const float *temperature, int B,
                                int n_nodes, int V, int max_depth, int max_branch, uint64_t seed,
                                int32_t *out_tokens, int32_t *out_accepted, int32_t *out_path,
                                void *workspace, size_t ws_bytes, spec_stream_t stream) {
  return verify_tree(target, tdt, draft, ddt, dk, node_token, parent, nullptr, cu_nodes,
                     temperature, B, n_nodes, V, max_depth, max_branch, seed, nullptr, out_tokens,
                     out_accepted, out_path, workspace, ws_bytes, stream);
}

extern "C" int spec_verify_tree_ext(const void *target, int tdt, const void *draft, int ddt,
                                    int dk, const int32_t *node_token, const int32_t *parent,
                                    const int32_t *node_fixed, const int32_t *cu_nodes,
                                    const float *temperature, int B, int n_nodes, int V,
                                    int max_depth, int max_branch, uint64_t seed,
                                    const uint64_t *seed_dev, int32_t *out_tokens,
                                    int32_t *out_accepted, int32_t *out_path, void *workspace,
                                    size_t ws_bytes, spec_stream_t stream) {
  return verify_tree(target, tdt, draft, ddt, dk, node_token, parent, node_fixed, cu_nodes,
                     temperature, B, n_nodes, V, max_depth, max_branch, seed, seed_dev,
                     out_tokens, out_accepted, out_path, workspace, ws_bytes, stream);
}
