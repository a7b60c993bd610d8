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
// Hands the registered events to a caller that brackets several launches
// itself (and unregisters them).
void take_row_pass_events(cudaEvent_t *before, cudaEvent_t *after);
int launch_row_pass(const RowPassArgs &a, cudaStream_t stream);
int nchunks(int V, int dtype, int chunk_bytes);
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Top-128 select + softmax over draft rows. Row r belongs to the request b
// with cu_rows[b] <= r < cu_rows[b+1]; rows >= cu_rows[B] are skipped.
// When `req_mode` is non-NULL, rows of requests whose mode is not
// sampling are skipped.
int launch_topk128(const void *logits, int dtype, int rows_bound, int V,
                   const int32_t *cu_rows, const float *temperature, int B,
                   int32_t *out_idx, float *out_prob, WsHeader *hdr,
                   cudaStream_t stream);

bool aligned(const void *p, size_t a);

}  // namespace sv
