// Tree verification (RRSw). Placeholder until the walker lands.
#include "common.cuh"
#include "internal.h"

extern "C" size_t spec_verify_tree_workspace(int, int, int, int, int) { return 0; }

extern "C" int spec_verify_tree(const void *, int, const void *, int, int, const int32_t *,
                                const int32_t *, const int32_t *, const float *, int, int, int,
                                int, int, uint64_t, int32_t *, int32_t *, int32_t *, void *,
                                size_t, spec_stream_t) {
  return SPEC_ERR_UNSUPPORTED;
}
