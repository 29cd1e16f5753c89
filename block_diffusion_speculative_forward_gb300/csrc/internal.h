// Internal declarations shared by libdflash's translation units: geometry,
// per-call device metadata, and the kernel launchers. Nothing here is part of
// the public ABI (include/dflash.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

namespace dfl {

using bf16 = __nv_bfloat16;

// Geometry of one head, copied into kernels by value.
struct Geo {
  int L, H, I, nq, nkv, d, V, gamma, B, S;
  int kv;        // nkv * d
  int qkv_w;     // nq*d + 2*kv: width of the stitched QKV output
  int pages;     // pages in the KV pool
  int kv_fp8;    // cache dtype
  int draft0;    // block row of the first draft: 1, or 0 with shifted rows
  float eps;
};

// One sequence of a propose call.
struct SeqMeta {
  int32_t pos;        // block position p (row 0 of the block)
  int32_t ws;         // window start: ctx positions ws..pos-1 are attended
  int32_t page_base;  // index in page_ids of logical page ws / B
  int32_t token;      // last verified token
};

// One ctx row to compute and store.
struct RowMeta {
  int32_t pos;        // target position of the row
  int32_t page;       // physical page that receives it
  int32_t slot;       // pos % B
  int32_t seq;        // sequence index within the call
  const bf16 *src;    // the row in the caller's stack
};

// Per-layer weights as kernels see them.
struct LayerW {
  const bf16 *in_norm, *q_norm, *k_norm, *post_norm;
  const bf16 *w_qkv;   // [qkv_w, H] stitched q;k;v
  const bf16 *w_o;     // [H, nq*d]
  const bf16 *w_gu;    // [2I, H] gate/up rows alternating
  const bf16 *w_down;  // [H, I]
};

// Bits of the device status word.
enum : int {
  ST_TOKEN = 1,   // a token id >= vocab reached the embed gather
  ST_PAGE = 2,    // a page id outside the pool reached a KV access
  ST_TIMEOUT = 4, // a bounded wait inside a kernel ran out; that kernel's output is invalid
};

// Element offset of (page, layer, kind, kv head, slot, 0) in the KV pool,
// laid out [page][L][K|V][nkv][B][d].
__host__ __device__ inline int64_t kv_offset(const Geo &g, int64_t page, int l, int kind, int h,
                                              int slot) {
  return ((((page * g.L + l) * 2 + kind) * g.nkv + h) * (int64_t)g.B + slot) * g.d;
}

// ------------------------------------------- programmatic dependent launch --
// Every kernel of the forward is launched with programmatic stream
// serialisation: it may start while its predecessor drains, lets its own
// successor launch at once (pdl_trigger), and touches data produced upstream
// only after pdl_wait, which returns once the predecessor grid has completed
// and its writes are visible. Every kernel executes pdl_wait, so completion
// is transitive along the stream.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same with a thread-block cluster of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t s, int cluster_x, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------------- launchers --
cudaError_t embed_block(const bf16 *E, const SeqMeta *seq, int n_seq, const Geo &g,
                        uint32_t mask_token, float *x, int *status, cudaStream_t s);

cudaError_t pack_rows(const RowMeta *rows, int m, int S, bf16 *out, cudaStream_t s);

struct Partials;
cudaError_t ctx_kv_write(const Partials &kv, int m, const RowMeta *rows, const Geo &g,
                         const bf16 *const *k_norm_dev, const float *cos_t, const float *sin_t,
                         void *pool, const float *kv_scale, int *status, cudaStream_t s);

// Per sequence: drafts, n_out, conf (and the status word) into out.
cudaError_t finalize(const int32_t *row_id, const float *row_p1, int n_seq, int nd,
                     const int *status, uint32_t *drafts, int32_t *n_out, float *conf,
                     int32_t *status_out, cudaStream_t s);

cudaError_t widen_lm_table(int fmt, const uint8_t *codes, const uint8_t *scales, int64_t rows,
                           int64_t k, bf16 *dst, cudaStream_t s);

cudaError_t rope_table(const float *inv_freq, int max_pos, int half, float scale, float *cos_t,
                       float *sin_t, cudaStream_t s);

cudaError_t gather_kv(const void *pool, const Geo &g, int layer, const RowMeta *rows, int n,
                      const float *kv_scale, float *k_out, float *v_out, cudaStream_t s);

}  // namespace dfl
