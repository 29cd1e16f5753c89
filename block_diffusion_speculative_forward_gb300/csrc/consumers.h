// Kernels that consume a projection's output (dense or split-K partials).
#pragma once

#include "gemm_tc.h"
#include "internal.h"

namespace dfl {

struct AddNormArgs {
  float *x;             // [rows, n] residual (updated when has_y), or NULL: start from 0
  bool has_y;
  Partials y;           // added to x
  const bf16 *g;        // [n] gain
  float eps;
  int n;
  bf16 *out;            // [rows, n] normed (or NULL)
  float *x_tap;         // [rows, n] copy of the updated residual (or NULL)
  bf16 *z_tap;          // [rows, n] copy of the normed rows (or NULL)
  bf16 *z;              // draft rows only: [n_seq * nd, n] (or NULL)
  int nd, gamma;
  int first;            // block row of a sequence's first draft row
  uint16_t *z16;        // draft rows again as f16 bits (or NULL)
};

struct QkvPostArgs {
  Geo g;
  Partials y;           // [R, qkv_w]
  const SeqMeta *seq;
  const bf16 *q_norm, *k_norm;
  const float *cos_t, *sin_t;
  bf16 *q, *kb, *vb;
};


cudaError_t add_norm(const AddNormArgs &p, int rows, cudaStream_t s);
cudaError_t qkv_post(const QkvPostArgs &p, int R, cudaStream_t s);

}  // namespace dfl
