// Split-KV block attention: work items, merge pairs and launch arguments.
#pragma once

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
  int64_t slot_floats;        // n_q*d + 2*n_q
  int *status;
};

// Query vectors of one (sequence, kv head): gamma * (nq / nkv), at most 128.
int attn_query_rows(const Geo &g);
cudaError_t attention_split(const AttnArgs &a, cudaStream_t s);

}  // namespace dfl
