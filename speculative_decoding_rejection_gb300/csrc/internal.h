// Host-side interfaces between the translation units of the library.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "specverify.h"

namespace sv {

struct WsHeader;
struct RowTask;
struct Part;
struct Job;
struct ReqInfo;

// Arguments of the row-statistics pass: every listed row is split into
// CHUNK_BYTES chunks; each consumer warp leaves one Part per chunk at
// part[(slot * nch_max + chunk) * RS_CONS_WARPS + warp].
struct RowPassArgs {
  const char *base[2];      // target / draft tensor
  long long row_bytes[2];   // V * element size
  int dtype[2];
  int nch[2];               // chunks per row of each tensor
  int nch_max;
  int chunk_bytes;          // chunk size, a multiple of TILE_BYTES
  const RowTask *list;      // rows to stream (count in hdr->n_list)
  WsHeader *hdr;
  Part *part;
  // Optional rank count: for a listed target row r, rank_thr[r] is the
  // draft token's logit (+inf: no count) and every Part's `cnt` receives the
  // number of the chunk's logits strictly above it. NULL: no counting.
  const float *rank_thr;
  // Optional row pairs (RowTask::which == ROW_PAIR): a target row and its
  // draft row streamed together; kl_part receives, per target part, A = the
  // sum of 2^((zt - m) c) (zt - zd) over the chunk. NULL: no pairs.
  float *kl_part;
  // Residual mode: instead of the row list, stream for every job of `jobs`
  // (count in hdr->n_jobs_a) target row t0+n and draft row d0+n tile by tile
  // (SAMPLE_TILE elements of each, bf16, 16-byte aligned rows) and leave per
  // consumer warp the tile sum of max(0, p - q) at
  // tsum4[(job * ntiles + tile) * RS_CONS_WARPS + warp].
  int residual;
  const Job *jobs;
  const ReqInfo *req;
  float *tsum4;
  int ntiles;
  int V;
};

int num_sms();
void set_row_pass_events(cudaEvent_t before, cudaEvent_t after);
bool row_pass_events_pending();
// Hands the registered events to a caller that brackets several launches
// itself (and unregisters them).
void take_row_pass_events(cudaEvent_t *before, cudaEvent_t *after);
int launch_row_pass(const RowPassArgs &a, cudaStream_t stream);
int nchunks(int V, int dtype, int chunk_bytes);
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Optional epilogue of the top-128 select for RheoSampling tree expansion:
// for every row f, the K children in rheostat slot order (the m best tokens
// other than the probe, the probe drawn from the row's top-128 law at
// u(seed, f, level, 3), the next best), their proxy probabilities under the
// unscaled top-128 law (the probe's: q(x_{m+1}) + eps), the probe law of
// each child's token, and path scores fscore[f] + ln q_proxy, written to
// [rows, K] arrays (qproxy and qtrue may be NULL).
struct RheoEpi {
  const float *fscore;
  int K, m;
  float eps;
  uint64_t seed;
  int level;
  int32_t *token;
  float *qproxy, *qtrue, *score;
};

// Top-128 select + softmax over draft rows. Row r belongs to the request b
// with cu_rows[b] <= r < cu_rows[b+1]; rows >= cu_rows[B] are skipped.
// out_idx / out_prob may be NULL when `rh` is given: the rows then feed the
// RheoSampling epilogue instead. With `lists` (topk_list_bytes(rows_bound)
// bytes, 256-byte aligned) and rows topk_two_launch() takes, the select runs
// as a scan launch and a finishing launch (which also runs the epilogue);
// otherwise as one launch. The events, if given, are recorded around the
// launch that reads the rows.
int launch_topk128(const void *logits, int dtype, int rows_bound, int V,
                   const int32_t *cu_rows, const float *temperature, int B,
                   int32_t *out_idx, float *out_prob, WsHeader *hdr,
                   cudaStream_t stream, const RheoEpi *rh = nullptr, void *lists = nullptr,
                   cudaEvent_t before = nullptr, cudaEvent_t after = nullptr);
size_t topk_list_bytes(long long rows);
// topk_list_bytes(rows) when V suits the two-launch select (any dtype), else 0
size_t topk_list_bytes_for(long long rows, int V);
bool topk_two_launch(int dtype, int V);

bool aligned(const void *p, size_t a);

}  // namespace sv
