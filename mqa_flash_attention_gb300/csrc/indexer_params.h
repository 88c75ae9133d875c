// Parameters of the indexer kernels (scoring of compressed rows and top-k
// selection).  Shared by the host code that fills them and by the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace ds4a {

// Candidates of the token at position p: compressed rows c with
// (c+1)*ratio <= p+1 (the pooled span has ended), capped by the rows stored.
struct IndexerGeom {
  int T, q_pos0, n_comp, ratio;
};

struct TopkParams {
  IndexerGeom g;
  const float *scores;
  long long score_stride;  // elements
  int32_t *idx;
  long long idx_stride;    // elements
  int top_k;
  int cached_keys;         // rows whose keys fit in the shared-memory cache
};

struct ScoreParams {
  IndexerGeom g;
  CUtensorMap tm_q;        // 3-D {head_dim, n_heads, T}, box {64, n_heads, tokens per group}
  CUtensorMap tm_k;        // 2-D {head_dim, n_comp}, box {64, 128}
  const float *w;          // [T][n_heads]
  float *scores;
  long long score_stride;  // elements
  float scale;
  int relu;
  int head_dim;            // 64, 128 or 256
  int n_groups;            // token groups of (256 / n_heads) tokens
  int n_row_tiles;         // ceil(n_comp / 128)
  int tiles_per_item;      // row tiles of one work item (a group's tiles are cut into items)
  int items_per_group;
  unsigned long long timeout_ns;
  unsigned int *err;
};

}  // namespace ds4a
