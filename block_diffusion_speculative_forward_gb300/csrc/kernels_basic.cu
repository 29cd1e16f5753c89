// Elementwise, normalisation, RoPE, paged-KV, attention and reduction kernels
// of the draft-head propose forward, plus a plain tiled GEMM used for the
// debug logits tap and for shapes the tensor-core GEMM does not take.
//
// Each kernel cites the passage of the head's API pages it implements:
//   [P1] "Struct BlockDiffusionDraftHead" (spark_model docs)
//   [P2] "BlockDiffusionDraftHead" (metrale docs)
//   [P3] "Trait DraftProposer" (spark_model docs)
#include "gemm_tc.h"
#include "internal.h"

#include <cuda_fp16.h>
#include <cuda_fp4.h>

#include <cfloat>
#include <cmath>

namespace dfl {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float fp8_to_float(uint8_t c) {
  __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(hr));
}

__device__ __forceinline__ uint8_t float_to_fp8(float v) {
  return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// ----------------------------------------------------------- block embed --
// [P1] fields gamma, mask_token_id, embed_tokens_shared: row 0 of each
// sequence's block embeds the last verified token, rows 1..gamma-1 the mask.
// Nothing earlier in the step touches x (the new ctx rows' kernels read and
// write their own buffers) and the previous step has completed, so the rows
// are written while the kernel before runs; the wait at the end keeps the
// next kernel behind both.
__global__ void k_embed_block(const bf16 *__restrict__ E, const SeqMeta *__restrict__ seq,
                              int gamma, int H, int V, uint32_t mask_token, float *__restrict__ x,
                              int *status) {
  pdl_trigger();
  int r = blockIdx.x;
  int i = r % gamma;
  uint32_t tok = i == 0 ? (uint32_t)seq[r / gamma].token : mask_token;
  if (tok >= (uint32_t)V) {
    if (threadIdx.x == 0) atomicOr(status, ST_TOKEN);
    tok = 0;
  }
  const bf16 *er = E + (int64_t)tok * H;
  for (int e = threadIdx.x; e < H; e += blockDim.x) x[(int64_t)r * H + e] = __bfloat162float(er[e]);
  pdl_wait();
}

cudaError_t embed_block(const bf16 *E, const SeqMeta *seq, int n_seq, const Geo &g,
                        uint32_t mask_token, float *x, int *status, cudaStream_t s) {
  launch_pdl(k_embed_block, dim3(n_seq * g.gamma), dim3(256), 0, s, E, seq, g.gamma, g.H, g.V, mask_token, x, status);
  return cudaGetLastError();
}

// ------------------------------------------------------------- row pack --
// Gathers the ctx rows to compute from the callers' stacks into one
// contiguous [m, S] buffer (16-byte vectors; S*2 is a multiple of 16).
// Padding rows (seq < 0) become zero rows.
__global__ void k_pack_rows(const RowMeta *__restrict__ rows, int S, bf16 *__restrict__ out) {
  pdl_trigger();
  pdl_wait();
  int r = blockIdx.x;
  const RowMeta rm = rows[r];
  const uint4 *src = (const uint4 *)rm.src;
  uint4 *dst = (uint4 *)(out + (int64_t)r * S);
  int nv = S / 8;
  if (rm.seq < 0 || !src) {
    for (int e = threadIdx.x; e < nv; e += blockDim.x) dst[e] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  for (int e = threadIdx.x; e < nv; e += blockDim.x) dst[e] = src[e];
}

cudaError_t pack_rows(const RowMeta *rows, int m, int S, bf16 *out, cudaStream_t s) {
  if (m <= 0) return cudaSuccess;
  launch_pdl(k_pack_rows, dim3(m), dim3(256), 0, s, rows, S, out);
  return cudaGetLastError();
}

// ------------------------------------------- per-head RMSNorm + RoPE --
// Normalises one head vector held by a warp (lane owns the pairs i = lane +
// 32t, i < d/2, elements i and i + d/2), applies gain g, then rotates each
// pair by the position's angle (rotate-half pairing over the full head,
// [P1] field rotary_dim). v[2*t] is element i, v[2*t+1] element i + d/2.
// gk[2t], gk[2t+1]: the gains of elements i and i + d/2; cs[t], sn[t] the
// rotation of pair i.
template <int NP>
__device__ __forceinline__ void norm_rope_warp(float (&v)[2 * NP], const float (&gk)[2 * NP],
                                               float eps, int d, const float (&cs)[NP],
                                               const float (&sn)[NP]) {
  float ss = 0.f;
#pragma unroll
  for (int t = 0; t < 2 * NP; ++t) ss += v[t] * v[t];
  ss = warp_sum(ss);
  float inv = rsqrtf(ss / (float)d + eps);
#pragma unroll
  for (int t = 0; t < NP; ++t) {
    float a = gk[2 * t] * (v[2 * t] * inv);
    float b = gk[2 * t + 1] * (v[2 * t + 1] * inv);
    v[2 * t] = a * cs[t] - b * sn[t];
    v[2 * t + 1] = b * cs[t] + a * sn[t];
  }
}

// ------------------------------------------------ ctx K/V paged write --
// [P1] fields fused_kv_weight, kv_cache, yarn_inv_freq: each ctx row's fused
// K/V GEMM output [L*2*kv] (per layer K then V) becomes, per layer and kv
// head, k = RoPE(k_norm(k), pos) and v, written to (page, slot) of the pool.
template <int NP>
__global__ void k_ctx_kv_write(const Partials kv, const RowMeta *__restrict__ rows,
                               Geo g, const bf16 *const *__restrict__ k_norm,
                               const float *__restrict__ cos_t, const float *__restrict__ sin_t,
                               void *pool, const float *__restrict__ kv_scale, int *status) {
  pdl_trigger();
  const int r = blockIdx.x, l = blockIdx.y;
  const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = g.d, half = d / 2;
  // the row record, contributor ranges, gains and rotation depend on no
  // earlier kernel: read before the wait
  const RowMeta rm = rows[r];
  if (rm.seq < 0) {   // padding row: computed, never stored
    pdl_wait();
    return;
  }
  if (rm.page < 0 || rm.page >= g.pages) {
    if (threadIdx.x == 0) atomicOr(status, ST_PAGE);
    pdl_wait();
    return;
  }
  const int kcol = l * 2 * g.kv + h * d, vcol = kcol + g.kv;
  // a head's K (and V) columns lie in one 128-column tile: one contributor
  // range each for the warp, all of its features' loads issued together
  TileRange trk{}, trv{};
  if (kv.ws) {
    trk = part_range(kv, part_tile(kv, r, kcol));
    trv = part_range(kv, part_tile(kv, r, vcol));
  }
  const bf16 *kg = k_norm[l];
  float gk[2 * NP], cs[NP], sn[NP];
#pragma unroll
  for (int t = 0; t < NP; ++t) {
    const int i = lane + 32 * t;
    gk[2 * t] = __bfloat162float(kg[i]);
    gk[2 * t + 1] = __bfloat162float(kg[i + half]);
    cs[t] = cos_t[(int64_t)rm.pos * half + i];
    sn[t] = sin_t[(int64_t)rm.pos * half + i];
  }
  int fk[2 * NP], fv[2 * NP];
#pragma unroll
  for (int t = 0; t < NP; ++t) {
    fk[2 * t] = kcol + lane + 32 * t;
    fk[2 * t + 1] = kcol + lane + 32 * t + half;
    fv[2 * t] = vcol + lane + 32 * t;
    fv[2 * t + 1] = vcol + lane + 32 * t + half;
  }
  pdl_wait();
  float v[2 * NP], vv[2 * NP];
  if (kv.ws) {
    part_sum_multi<2 * NP>(kv, trk, r, fk, v);
    part_sum_multi<2 * NP>(kv, trv, r, fv, vv);
  } else {
#pragma unroll
    for (int t = 0; t < 2 * NP; ++t) {
      v[t] = kv.dense[(int64_t)r * kv.ld + fk[t]];
      vv[t] = kv.dense[(int64_t)r * kv.ld + fv[t]];
    }
  }
  norm_rope_warp<NP>(v, gk, g.eps, d, cs, sn);
  int64_t ko = kv_offset(g, rm.page, l, 0, h, rm.slot);
  int64_t vo = kv_offset(g, rm.page, l, 1, h, rm.slot);
  if (g.kv_fp8) {
    float sk = kv_scale[(l * g.nkv + h) * 2 + 0], sv = kv_scale[(l * g.nkv + h) * 2 + 1];
    uint8_t *P = (uint8_t *)pool;
#pragma unroll
    for (int t = 0; t < NP; ++t) {
      int i = lane + 32 * t;
      P[ko + i] = float_to_fp8(v[2 * t] / sk);
      P[ko + i + half] = float_to_fp8(v[2 * t + 1] / sk);
    }
#pragma unroll
    for (int t = 0; t < NP; ++t) {
      const int i = lane + 32 * t;
      P[vo + i] = float_to_fp8(vv[2 * t] / sv);
      P[vo + i + half] = float_to_fp8(vv[2 * t + 1] / sv);
    }
  } else {
    bf16 *P = (bf16 *)pool;
#pragma unroll
    for (int t = 0; t < NP; ++t) {
      int i = lane + 32 * t;
      P[ko + i] = __float2bfloat16_rn(v[2 * t]);
      P[ko + i + half] = __float2bfloat16_rn(v[2 * t + 1]);
    }
#pragma unroll
    for (int t = 0; t < NP; ++t) {
      const int i = lane + 32 * t;
      P[vo + i] = __float2bfloat16_rn(vv[2 * t]);
      P[vo + i + half] = __float2bfloat16_rn(vv[2 * t + 1]);
    }
  }
}

cudaError_t ctx_kv_write(const Partials &kv, int m, const RowMeta *rows, const Geo &g,
                         const bf16 *const *k_norm_dev, const float *cos_t, const float *sin_t,
                         void *pool, const float *kv_scale, int *status, cudaStream_t s) {
  if (m <= 0) return cudaSuccess;
  dim3 grid(m, g.L);
  if (g.d == 128)
    launch_pdl(k_ctx_kv_write<2>, dim3(grid), dim3(32 * g.nkv), 0, s, kv, rows, g, k_norm_dev, cos_t, sin_t, pool,
                                                  kv_scale, status);
  else if (g.d == 64)
    launch_pdl(k_ctx_kv_write<1>, dim3(grid), dim3(32 * g.nkv), 0, s, kv, rows, g, k_norm_dev, cos_t, sin_t, pool,
                                                  kv_scale, status);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

// Chain: drafts stop before the first row with nothing allowed; conf is the
// minimum top-1 probability over the produced drafts (0 when none).
__global__ void k_finalize(const int32_t *__restrict__ row_id, const float *__restrict__ row_p1,
                           int n_seq, int nd, const int *status, uint32_t *drafts, int32_t *n_out,
                           float *conf, int32_t *status_out) {
  pdl_trigger();
  pdl_wait();
  int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s == 0) *status_out = *status;
  if (s >= n_seq) return;
  int n = 0;
  float c = INFINITY;
  for (int i = 0; i < nd; ++i) {
    int id = row_id[s * nd + i];
    if (id < 0) break;
    drafts[s * nd + i] = (uint32_t)id;
    c = fminf(c, row_p1[s * nd + i]);
    ++n;
  }
  for (int i = n; i < nd; ++i) drafts[s * nd + i] = 0;
  n_out[s] = n;
  conf[s] = n ? c : 0.f;
}

cudaError_t finalize(const int32_t *row_id, const float *row_p1, int n_seq, int nd,
                     const int *status, uint32_t *drafts, int32_t *n_out, float *conf,
                     int32_t *status_out, cudaStream_t s) {
  launch_pdl(k_finalize, dim3((n_seq + 127) / 128), dim3(128), 0, s, row_id, row_p1, n_seq, nd, status, drafts, n_out,
                                                  conf, status_out);
  return cudaGetLastError();
}

// --------------------------------------------- lm_head table widening --
// A low-precision lm_head table as bf16 values, exactly (every E4M3 value and
// every E2M1 x E4M3 product is a bf16 value), for the many-row tensor-core
// kernels; the row scale (FP8) or global scale (NVFP4) stays in their
// epilogues. fmt 1: codes [rows, k] E4M3; fmt 2: codes [rows, k/2] E2M1
// pairs (element 2j in the low nibble) and scales [rows, k/16] E4M3.
__global__ void k_widen_lm(int fmt, const uint8_t *__restrict__ codes,
                           const uint8_t *__restrict__ scales, int64_t rows, int64_t k,
                           bf16 *__restrict__ dst) {
  const int64_t n = rows * k;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v;
    if (fmt == 1) {
      v = fp8_to_float(codes[i]);
    } else {
      const int64_t r = i / k, c = i % k;
      const uint8_t b = codes[r * (k / 2) + c / 2];
      const __half_raw e = __nv_cvt_fp4_to_halfraw((__nv_fp4_storage_t)((c & 1) ? b >> 4 : b & 15),
                                                   __NV_E2M1);
      v = __half2float(*reinterpret_cast<const __half *>(&e)) * fp8_to_float(scales[r * (k / 16) + c / 16]);
    }
    dst[i] = __float2bfloat16_rn(v);
  }
}

cudaError_t widen_lm_table(int fmt, const uint8_t *codes, const uint8_t *scales, int64_t rows,
                           int64_t k, bf16 *dst, cudaStream_t s) {
  k_widen_lm<<<4096, 256, 0, s>>>(fmt, codes, scales, rows, k, dst);
  return cudaGetLastError();
}

// ------------------------------------------------------------ RoPE table --
// cos/sin of pos * inv_freq[i] for every position the head can reach, times
// the attention temperature scale (1 without YaRN), evaluated in double and
// stored f32 ([P1] field yarn_inv_freq).
__global__ void k_rope_table(const float *__restrict__ inv_freq, int max_pos, int half,
                             float scale, float *__restrict__ cos_t, float *__restrict__ sin_t) {
  pdl_trigger();
  pdl_wait();
  int64_t n = (int64_t)max_pos * half;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n;
       t += (int64_t)gridDim.x * blockDim.x) {
    int pos = (int)(t / half), i = (int)(t % half);
    double a = (double)pos * (double)inv_freq[i];
    double sv, cv;
    sincos(a, &sv, &cv);
    cos_t[t] = (float)(cv * (double)scale);
    sin_t[t] = (float)(sv * (double)scale);
  }
}

cudaError_t rope_table(const float *inv_freq, int max_pos, int half, float scale, float *cos_t,
                       float *sin_t, cudaStream_t s) {
  launch_pdl(k_rope_table, dim3(1024), dim3(256), 0, s, inv_freq, max_pos, half, scale, cos_t,
             sin_t);
  return cudaGetLastError();
}

// ------------------------------------------------------- debug KV gather --
__global__ void k_gather_kv(const void *__restrict__ pool, Geo g, int layer,
                            const RowMeta *__restrict__ rows, const float *__restrict__ kv_scale,
                            float *k_out, float *v_out) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const int page = rows[r].page, slot = rows[r].slot;
  for (int e = threadIdx.x; e < g.kv; e += blockDim.x) {
    int h = e / g.d, i = e % g.d;
    int64_t ko = kv_offset(g, page, layer, 0, h, slot) + i;
    int64_t vo = kv_offset(g, page, layer, 1, h, slot) + i;
    float kx, vx;
    if (g.kv_fp8) {
      kx = fp8_to_float(((const uint8_t *)pool)[ko]) * kv_scale[(layer * g.nkv + h) * 2];
      vx = fp8_to_float(((const uint8_t *)pool)[vo]) * kv_scale[(layer * g.nkv + h) * 2 + 1];
    } else {
      kx = __bfloat162float(((const bf16 *)pool)[ko]);
      vx = __bfloat162float(((const bf16 *)pool)[vo]);
    }
    k_out[(int64_t)r * g.kv + e] = kx;
    v_out[(int64_t)r * g.kv + e] = vx;
  }
}

cudaError_t gather_kv(const void *pool, const Geo &g, int layer, const RowMeta *rows, int n,
                      const float *kv_scale, float *k_out, float *v_out, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  launch_pdl(k_gather_kv, dim3(n), dim3(256), 0, s, pool, g, layer, rows, kv_scale, k_out, v_out);
  return cudaGetLastError();
}

}  // namespace dfl
