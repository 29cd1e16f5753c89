// Split-KV block attention: work items, merge pairs and launch arguments.
#pragma once

#include <cuda.h>

#include "internal.h"

namespace dfl {

// One CTA of work: keys [k0, k1) of sequence s, kv head g. Key index space:
// [0, n_ctx) are the window's ctx rows (positions ws..pos-1), then the gamma
// block rows. An item never mixes ctx and block keys. slot < 0: the pair has
// this one item and writes its output directly.
struct AttnItem {
  int32_t s, g, k0, k1, slot;
};

// A (sequence, kv head) cut into nc items whose partials sit in slots
// slot0..slot0+nc-1.
struct AttnPair {
  int32_t s, g, slot0, nc;
};

struct AttnArgs {
  Geo g;
  const bf16 *q, *kb, *vb;    // [R, nq*d], [R, kv], [R, kv]
  bf16 *o;                    // [R, nq*d]
  const SeqMeta *seq;
  const int32_t *page_ids;
  const void *pool;
  const float *kv_scale;
  int layer;
  float scale;                // 1/sqrt(d)
  const AttnItem *items;
  int n_items;                // grid size: at least the call's item count
  const AttnPair *pairs;
  int n_pairs;                // grid size: at least the call's pair count
  const int *counts;          // device: [0] items, [1] pairs of this call
  float *ws;                  // partial slots
  int64_t slot_floats;        // n_q*d + 2*n_q, rounded up to a multiple of 4
  int *status;
  // tensor-core kernel: CTA b runs items [cta_off[b], cta_off[b + 1])
  const int32_t *cta_off;
  int grid_tc;
};

// TMA maps of the tensor-core kernel's operands (ok = false: not supported).
struct AttnMaps {
  CUtensorMap q, pool, kb, vb;
  bool ok = false;
};

// Query vectors of one (sequence, kv head): gamma * (nq / nkv), at most 128.
int attn_query_rows(const Geo &g);
// mma.sync kernel (any supported geometry, bf16 or FP8 cache) + merge.
cudaError_t attention_split(const AttnArgs &a, cudaStream_t s);
// Merge of the split items' partials (pairs cut into several items).
cudaError_t attention_merge(const AttnArgs &a, cudaStream_t s);

// tcgen05 kernel (attention_tc.cu): bf16 cache, head dim 128, <= 128 query
// vectors per (sequence, kv head). The caller runs attention_merge after it.
bool attention_tc_supported(const Geo &g);
// Builds the maps (m->ok stays false when the geometry is not supported);
// false on an encoding failure.
bool attention_tc_maps(const Geo &g, int R_max, const void *q, const void *pool, const void *kb,
                       const void *vb, AttnMaps *m);
cudaError_t attention_tc(const AttnArgs &a, const AttnMaps &m, cudaStream_t s);
// Key tiles the tensor-core kernel runs for an item (its scheduling cost).
int attention_tc_tiles(const Geo &g, const SeqMeta &sm, const AttnItem &it);

}  // namespace dfl
