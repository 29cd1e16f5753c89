// Elementwise, normalisation, RoPE, paged-KV, attention and reduction kernels
// of the draft-head propose forward, plus a plain tiled GEMM used for the
// debug logits tap and for shapes the tensor-core GEMM does not take.
//
// Each kernel cites the passage of the head's API pages it implements:
//   [P1] "Struct BlockDiffusionDraftHead" (spark_model docs)
//   [P2] "BlockDiffusionDraftHead" (metrale docs)
//   [P3] "Trait DraftProposer" (spark_model docs)
#include "internal.h"

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

// Block-wide sum over blockDim.x threads (a multiple of 32, <= 1024).
__device__ float block_sum(float v, float *sh) {
  v = warp_sum(v);
  int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) sh[w] = v;
  __syncthreads();
  float t = 0.f;
  int nw = blockDim.x >> 5;
  for (int i = 0; i < nw; ++i) t += sh[i];
  return t;
}

// ------------------------------------------------------------ plain GEMM --
// 64x64 output tile, K step 32, 256 threads with a 4x4 micro tile each.
template <int EPI, bool FP8>
__global__ void __launch_bounds__(256) k_gemm_simple(const bf16 *__restrict__ A, int lda,
                                                     const void *__restrict__ W,
                                                     const float *__restrict__ wscale, void *C,
                                                     int ldc, int m, int n, int K) {
  __shared__ float As[32][65];
  __shared__ float Ws[32][65];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 32) {
    for (int i = threadIdx.x; i < 64 * 32; i += 256) {
      int r = i >> 5, kk = i & 31;
      int gr = m0 + r, gc = n0 + r;
      As[kk][r] = gr < m ? __bfloat162float(A[(int64_t)gr * lda + k0 + kk]) : 0.f;
      float wv = 0.f;
      if (gc < n) {
        if (FP8)
          wv = fp8_to_float(((const uint8_t *)W)[(int64_t)gc * K + k0 + kk]);
        else
          wv = __bfloat162float(((const bf16 *)W)[(int64_t)gc * K + k0 + kk]);
      }
      Ws[kk][r] = wv;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int r = m0 + ty * 4 + i;
    if (r >= m) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int c = n0 + tx * 4 + j;
      if (c >= n) continue;
      float v = acc[i][j];
      if (wscale) v *= wscale[c];
      int64_t off = (int64_t)r * ldc + c;
      if (EPI == EPI_STORE_F32) ((float *)C)[off] = v;
      else if (EPI == EPI_ADD_F32) ((float *)C)[off] += v;
      else ((bf16 *)C)[off] = __float2bfloat16_rn(v);
    }
  }
}

cudaError_t gemm_simple(const bf16 *A, int lda, const void *W, bool w_fp8, const float *wscale,
                        void *C, int ldc, int m, int n, int K, GemmEpi epi, cudaStream_t s) {
  if (m <= 0 || n <= 0) return cudaSuccess;
  if (K % 32) return cudaErrorInvalidValue;
  dim3 grid((n + 63) / 64, (m + 63) / 64);
#define DFL_GEMM_CASE(E)                                                                       \
  if (epi == E) {                                                                              \
    if (w_fp8)                                                                                 \
      k_gemm_simple<E, true><<<grid, 256, 0, s>>>(A, lda, W, wscale, C, ldc, m, n, K);         \
    else                                                                                       \
      k_gemm_simple<E, false><<<grid, 256, 0, s>>>(A, lda, W, wscale, C, ldc, m, n, K);        \
  }
  DFL_GEMM_CASE(EPI_STORE_F32)
  DFL_GEMM_CASE(EPI_ADD_F32)
  DFL_GEMM_CASE(EPI_STORE_BF16)
#undef DFL_GEMM_CASE
  return cudaGetLastError();
}

// --------------------------------------------------------------- RMSNorm --
// [P1] fields rms_norm_eps, hidden_norm, norm; the Qwen3 layer norms.
__global__ void k_rmsnorm_rows(const float *__restrict__ x, int n, const bf16 *__restrict__ g,
                               float eps, int nd, int gamma, bf16 *__restrict__ out) {
  __shared__ float sh[32];
  int i = blockIdx.x;
  int r = nd > 0 ? (i / nd) * gamma + 1 + (i % nd) : i;
  const float *xr = x + (int64_t)r * n;
  float ss = 0.f;
  for (int e = threadIdx.x; e < n; e += blockDim.x) ss += xr[e] * xr[e];
  ss = block_sum(ss, sh);
  float inv = rsqrtf(ss / (float)n + eps);
  for (int e = threadIdx.x; e < n; e += blockDim.x)
    out[(int64_t)i * n + e] = __float2bfloat16_rn(__bfloat162float(g[e]) * (xr[e] * inv));
}

cudaError_t rmsnorm_rows(const float *x, int rows, int n, const bf16 *g, float eps, int nd,
                         int gamma, bf16 *out, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  k_rmsnorm_rows<<<rows, 256, 0, s>>>(x, n, g, eps, nd, gamma, out);
  return cudaGetLastError();
}

// ----------------------------------------------------------- block embed --
// [P1] fields gamma, mask_token_id, embed_tokens_shared: row 0 of each
// sequence's block embeds the last verified token, rows 1..gamma-1 the mask.
__global__ void k_embed_block(const bf16 *__restrict__ E, const SeqMeta *__restrict__ seq,
                              int gamma, int H, int V, uint32_t mask_token, float *__restrict__ x,
                              int *status) {
  int r = blockIdx.x;
  int i = r % gamma;
  uint32_t tok = i == 0 ? (uint32_t)seq[r / gamma].token : mask_token;
  if (tok >= (uint32_t)V) {
    if (threadIdx.x == 0) atomicOr(status, ST_TOKEN);
    tok = 0;
  }
  const bf16 *er = E + (int64_t)tok * H;
  for (int e = threadIdx.x; e < H; e += blockDim.x) x[(int64_t)r * H + e] = __bfloat162float(er[e]);
}

cudaError_t embed_block(const bf16 *E, const SeqMeta *seq, int n_seq, const Geo &g,
                        uint32_t mask_token, float *x, int *status, cudaStream_t s) {
  k_embed_block<<<n_seq * g.gamma, 256, 0, s>>>(E, seq, g.gamma, g.H, g.V, mask_token, x, status);
  return cudaGetLastError();
}

// ------------------------------------------------------------- row pack --
// Gathers the ctx rows to compute from the callers' stacks into one
// contiguous [m, S] buffer (16-byte vectors; S*2 is a multiple of 16).
__global__ void k_pack_rows(const RowMeta *__restrict__ rows, int S, bf16 *__restrict__ out) {
  int r = blockIdx.x;
  const uint4 *src = (const uint4 *)rows[r].src;
  uint4 *dst = (uint4 *)(out + (int64_t)r * S);
  int nv = S / 8;
  for (int e = threadIdx.x; e < nv; e += blockDim.x) dst[e] = src[e];
}

cudaError_t pack_rows(const RowMeta *rows, int m, int S, bf16 *out, cudaStream_t s) {
  if (m <= 0) return cudaSuccess;
  k_pack_rows<<<m, 256, 0, s>>>(rows, S, out);
  return cudaGetLastError();
}

// ------------------------------------------- per-head RMSNorm + RoPE --
// Normalises one head vector held by a warp (lane owns the pairs i = lane +
// 32t, i < d/2, elements i and i + d/2), applies gain g, then rotates each
// pair by the position's angle (rotate-half pairing over the full head,
// [P1] field rotary_dim). v[2*t] is element i, v[2*t+1] element i + d/2.
template <int NP>
__device__ __forceinline__ void norm_rope_warp(float (&v)[2 * NP], const bf16 *g, float eps,
                                               int d, const float *cos_row,
                                               const float *sin_row) {
  const int lane = threadIdx.x & 31;
  float ss = 0.f;
#pragma unroll
  for (int t = 0; t < 2 * NP; ++t) ss += v[t] * v[t];
  ss = warp_sum(ss);
  float inv = rsqrtf(ss / (float)d + eps);
#pragma unroll
  for (int t = 0; t < NP; ++t) {
    int i = lane + 32 * t;
    float a = __bfloat162float(g[i]) * (v[2 * t] * inv);
    float b = __bfloat162float(g[i + d / 2]) * (v[2 * t + 1] * inv);
    float c = cos_row[i], s = sin_row[i];
    v[2 * t] = a * c - b * s;
    v[2 * t + 1] = b * c + a * s;
  }
}

// ------------------------------------------------ ctx K/V paged write --
// [P1] fields fused_kv_weight, kv_cache, yarn_inv_freq: each ctx row's fused
// K/V GEMM output [L*2*kv] (per layer K then V) becomes, per layer and kv
// head, k = RoPE(k_norm(k), pos) and v, written to (page, slot) of the pool.
template <int NP>
__global__ void k_ctx_kv_write(const float *__restrict__ kv, const RowMeta *__restrict__ rows,
                               Geo g, const bf16 *const *__restrict__ k_norm,
                               const float *__restrict__ cos_t, const float *__restrict__ sin_t,
                               void *pool, const float *__restrict__ kv_scale, int *status) {
  const int r = blockIdx.x, l = blockIdx.y;
  const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = g.d, half = d / 2;
  const RowMeta rm = rows[r];
  if (rm.page < 0 || rm.page >= g.pages) {
    if (threadIdx.x == 0) atomicOr(status, ST_PAGE);
    return;
  }
  const float *kr = kv + (int64_t)r * (g.L * 2 * g.kv) + (int64_t)l * 2 * g.kv + h * d;
  const float *vr = kr + g.kv;
  float v[2 * NP];
#pragma unroll
  for (int t = 0; t < NP; ++t) {
    v[2 * t] = kr[lane + 32 * t];
    v[2 * t + 1] = kr[lane + 32 * t + half];
  }
  norm_rope_warp<NP>(v, k_norm[l], g.eps, d, cos_t + (int64_t)rm.pos * half,
                     sin_t + (int64_t)rm.pos * half);
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
    for (int e = lane; e < d; e += 32) P[vo + e] = float_to_fp8(vr[e] / sv);
  } else {
    bf16 *P = (bf16 *)pool;
#pragma unroll
    for (int t = 0; t < NP; ++t) {
      int i = lane + 32 * t;
      P[ko + i] = __float2bfloat16_rn(v[2 * t]);
      P[ko + i + half] = __float2bfloat16_rn(v[2 * t + 1]);
    }
    for (int e = lane; e < d; e += 32) P[vo + e] = __float2bfloat16_rn(vr[e]);
  }
}

cudaError_t ctx_kv_write(const float *kv, int m, const RowMeta *rows, const Geo &g,
                         const bf16 *const *k_norm_dev, const float *cos_t, const float *sin_t,
                         void *pool, const float *kv_scale, int *status, cudaStream_t s) {
  if (m <= 0) return cudaSuccess;
  dim3 grid(m, g.L);
  if (g.d == 128)
    k_ctx_kv_write<2><<<grid, 32 * g.nkv, 0, s>>>(kv, rows, g, k_norm_dev, cos_t, sin_t, pool,
                                                  kv_scale, status);
  else if (g.d == 64)
    k_ctx_kv_write<1><<<grid, 32 * g.nkv, 0, s>>>(kv, rows, g, k_norm_dev, cos_t, sin_t, pool,
                                                  kv_scale, status);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

// ----------------------------------------- block q/k norm + RoPE, v copy --
// The Qwen3 per-head q/k RMSNorm, then RoPE at the row's position p + i.
template <int NP>
__global__ void k_block_qkv_post(const float *__restrict__ qkv, const SeqMeta *__restrict__ seq,
                                 Geo g, const bf16 *__restrict__ q_norm,
                                 const bf16 *__restrict__ k_norm, const float *__restrict__ cos_t,
                                 const float *__restrict__ sin_t, bf16 *__restrict__ q,
                                 bf16 *__restrict__ kb, bf16 *__restrict__ vb) {
  const int r = blockIdx.x;
  const int head = blockIdx.y * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int d = g.d, half = d / 2;
  const int pos = seq[r / g.gamma].pos + r % g.gamma;
  const float *row = qkv + (int64_t)r * g.qkv_w;
  if (head < g.nq + g.nkv) {
    const bool is_q = head < g.nq;
    const float *src = is_q ? row + head * d : row + g.nq * d + (head - g.nq) * d;
    float v[2 * NP];
#pragma unroll
    for (int t = 0; t < NP; ++t) {
      v[2 * t] = src[lane + 32 * t];
      v[2 * t + 1] = src[lane + 32 * t + half];
    }
    norm_rope_warp<NP>(v, is_q ? q_norm : k_norm, g.eps, d, cos_t + (int64_t)pos * half,
                       sin_t + (int64_t)pos * half);
    bf16 *dst = is_q ? q + (int64_t)r * g.nq * d + head * d
                     : kb + (int64_t)r * g.kv + (head - g.nq) * d;
#pragma unroll
    for (int t = 0; t < NP; ++t) {
      dst[lane + 32 * t] = __float2bfloat16_rn(v[2 * t]);
      dst[lane + 32 * t + half] = __float2bfloat16_rn(v[2 * t + 1]);
    }
  }
  if (blockIdx.y == 0) {
    const float *vsrc = row + g.nq * d + g.kv;
    for (int e = threadIdx.x; e < g.kv; e += blockDim.x)
      vb[(int64_t)r * g.kv + e] = __float2bfloat16_rn(vsrc[e]);
  }
}

cudaError_t block_qkv_post(const float *qkv, int R, const SeqMeta *seq, const Geo &g,
                           const bf16 *q_norm, const bf16 *k_norm, const float *cos_t,
                           const float *sin_t, bf16 *q, bf16 *kb, bf16 *vb, cudaStream_t s) {
  dim3 grid(R, (g.nq + g.nkv + 7) / 8);
  if (g.d == 128)
    k_block_qkv_post<2><<<grid, 256, 0, s>>>(qkv, seq, g, q_norm, k_norm, cos_t, sin_t, q, kb, vb);
  else if (g.d == 64)
    k_block_qkv_post<1><<<grid, 256, 0, s>>>(qkv, seq, g, q_norm, k_norm, cos_t, sin_t, q, kb, vb);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

// -------------------------------------------------- block attention --
// One warp per (block row, q head): online softmax over the window's ctx keys
// (paged) and the gamma block keys, no mask inside the block. q head j reads
// kv head j * nkv / nq. Lane owns d/32 contiguous elements.
template <int EPL>
__global__ void k_attention_simple(const bf16 *__restrict__ q, const bf16 *__restrict__ kb,
                                   const bf16 *__restrict__ vb, const SeqMeta *__restrict__ seq,
                                   const int32_t *__restrict__ page_ids, Geo g,
                                   const void *__restrict__ pool, int layer,
                                   const float *__restrict__ kv_scale, float scale,
                                   bf16 *__restrict__ o, int *status) {
  const int r = blockIdx.x, j = blockIdx.y, lane = threadIdx.x;
  const int s_idx = r / g.gamma;
  const SeqMeta sm = seq[s_idx];
  const int kvh = (j * g.nkv) / g.nq;
  const int e0 = lane * EPL;
  float qv[EPL], acc[EPL];
  const bf16 *qr = q + (int64_t)r * g.nq * g.d + j * g.d + e0;
#pragma unroll
  for (int t = 0; t < EPL; ++t) {
    qv[t] = __bfloat162float(qr[t]) * scale;
    acc[t] = 0.f;
  }
  float mx = -INFINITY, den = 0.f;
  float sk = 1.f, sv = 1.f;
  if (g.kv_fp8) {
    sk = kv_scale[(layer * g.nkv + kvh) * 2 + 0];
    sv = kv_scale[(layer * g.nkv + kvh) * 2 + 1];
  }
  const int b0 = sm.ws / g.B;
  for (int pos = sm.ws; pos < sm.pos; ++pos) {
    int page = page_ids[sm.page_base + (pos / g.B - b0)];
    if (page < 0 || page >= g.pages) {
      if (lane == 0) atomicOr(status, ST_PAGE);
      break;
    }
    int64_t ko = kv_offset(g, page, layer, 0, kvh, pos % g.B) + e0;
    int64_t vo = kv_offset(g, page, layer, 1, kvh, pos % g.B) + e0;
    float kx[EPL], vx[EPL];
    if (g.kv_fp8) {
      const uint8_t *P = (const uint8_t *)pool;
#pragma unroll
      for (int t = 0; t < EPL; ++t) {
        kx[t] = fp8_to_float(P[ko + t]) * sk;
        vx[t] = fp8_to_float(P[vo + t]) * sv;
      }
    } else {
      const bf16 *P = (const bf16 *)pool;
#pragma unroll
      for (int t = 0; t < EPL; ++t) {
        kx[t] = __bfloat162float(P[ko + t]);
        vx[t] = __bfloat162float(P[vo + t]);
      }
    }
    float dot = 0.f;
#pragma unroll
    for (int t = 0; t < EPL; ++t) dot = fmaf(qv[t], kx[t], dot);
    dot = warp_sum(dot);
    float mn = fmaxf(mx, dot);
    float corr = __expf(mx - mn), p = __expf(dot - mn);
    den = den * corr + p;
#pragma unroll
    for (int t = 0; t < EPL; ++t) acc[t] = acc[t] * corr + p * vx[t];
    mx = mn;
  }
  for (int t2 = 0; t2 < g.gamma; ++t2) {
    const int br = s_idx * g.gamma + t2;
    const bf16 *kr = kb + (int64_t)br * g.kv + kvh * g.d + e0;
    const bf16 *vr = vb + (int64_t)br * g.kv + kvh * g.d + e0;
    float dot = 0.f;
#pragma unroll
    for (int t = 0; t < EPL; ++t) dot = fmaf(qv[t], __bfloat162float(kr[t]), dot);
    dot = warp_sum(dot);
    float mn = fmaxf(mx, dot);
    float corr = __expf(mx - mn), p = __expf(dot - mn);
    den = den * corr + p;
#pragma unroll
    for (int t = 0; t < EPL; ++t) acc[t] = acc[t] * corr + p * __bfloat162float(vr[t]);
    mx = mn;
  }
  bf16 *orow = o + (int64_t)r * g.nq * g.d + j * g.d + e0;
  float inv = 1.f / den;
#pragma unroll
  for (int t = 0; t < EPL; ++t) orow[t] = __float2bfloat16_rn(acc[t] * inv);
}

cudaError_t attention_simple(const bf16 *q, const bf16 *kb, const bf16 *vb, const SeqMeta *seq,
                             const int32_t *page_ids, int n_seq, const Geo &g, const void *pool,
                             int layer, const float *kv_scale, bf16 *o, int *status,
                             cudaStream_t s) {
  dim3 grid(n_seq * g.gamma, g.nq);
  float scale = (float)(1.0 / std::sqrt((double)g.d));
  if (g.d == 128)
    k_attention_simple<4><<<grid, 32, 0, s>>>(q, kb, vb, seq, page_ids, g, pool, layer, kv_scale,
                                              scale, o, status);
  else if (g.d == 64)
    k_attention_simple<2><<<grid, 32, 0, s>>>(q, kb, vb, seq, page_ids, g, pool, layer, kv_scale,
                                              scale, o, status);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

// ------------------------------------------------------------------ SwiGLU --
__global__ void k_swiglu(const float *__restrict__ gu, int I, bf16 *__restrict__ u) {
  const int r = blockIdx.x;
  const float *gr = gu + (int64_t)r * 2 * I;
  for (int e = threadIdx.x; e < I; e += blockDim.x) {
    float a = gr[e], b = gr[I + e];
    u[(int64_t)r * I + e] = __float2bfloat16_rn(a / (1.f + __expf(-a)) * b);
  }
}

cudaError_t swiglu(const float *gu, int R, int I, bf16 *u, cudaStream_t s) {
  k_swiglu<<<R, 256, 0, s>>>(gu, I, u);
  return cudaGetLastError();
}

// ------------------------------------------------- argmax + confidence --
// [P1] field lm_head_shared (per-position argmax), [P3] grammar_bitmask
// (bit tok set => allowed), last_confidence (top-1 softmax probability).
// Ties go to the lowest token id.
__global__ void k_argmax_rows(const float *__restrict__ logits, int V,
                              const int32_t *__restrict__ bitmask, int nd,
                              int32_t *__restrict__ row_id, float *__restrict__ row_p1) {
  __shared__ float smx[32];
  __shared__ int sid[32];
  __shared__ float ssum[32];
  const int r = blockIdx.x;
  const int words = (V + 31) / 32;
  const int32_t *bm = bitmask ? bitmask + (int64_t)(r / nd) * words : nullptr;
  const float *lr = logits + (int64_t)r * V;
  float best = -INFINITY;
  int bid = INT32_MAX;
  for (int t = threadIdx.x; t < V; t += blockDim.x) {
    if (bm && !((((uint32_t)bm[t >> 5]) >> (t & 31)) & 1u)) continue;
    float v = lr[t];
    if (v > best || (v == best && t < bid)) { best = v; bid = t; }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, best, off);
    int oi = __shfl_xor_sync(0xffffffffu, bid, off);
    if (ov > best || (ov == best && oi < bid)) { best = ov; bid = oi; }
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (lane == 0) { smx[w] = best; sid[w] = bid; }
  __syncthreads();
  best = smx[0];
  bid = sid[0];
  for (int i = 1; i < nw; ++i)
    if (smx[i] > best || (smx[i] == best && sid[i] < bid)) { best = smx[i]; bid = sid[i]; }
  if (bid == INT32_MAX) {
    if (threadIdx.x == 0) { row_id[r] = -1; row_p1[r] = 0.f; }
    return;
  }
  float sum = 0.f;
  for (int t = threadIdx.x; t < V; t += blockDim.x) {
    if (bm && !((((uint32_t)bm[t >> 5]) >> (t & 31)) & 1u)) continue;
    sum += __expf(lr[t] - best);
  }
  sum = warp_sum(sum);
  __syncthreads();
  if (lane == 0) ssum[w] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int i = 0; i < nw; ++i) tot += ssum[i];
    row_id[r] = bid;
    row_p1[r] = 1.f / tot;
  }
}

cudaError_t argmax_rows(const float *logits, int rows, int V, const int32_t *bitmask, int nd,
                        int32_t *row_id, float *row_p1, cudaStream_t s) {
  k_argmax_rows<<<rows, 1024, 0, s>>>(logits, V, bitmask, nd, row_id, row_p1);
  return cudaGetLastError();
}

// Chain: drafts stop before the first row with nothing allowed; conf is the
// minimum top-1 probability over the produced drafts (0 when none).
__global__ void k_finalize(const int32_t *__restrict__ row_id, const float *__restrict__ row_p1,
                           int n_seq, int nd, const int *status, uint32_t *drafts, int32_t *n_out,
                           float *conf, int32_t *status_out) {
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
  k_finalize<<<(n_seq + 127) / 128, 128, 0, s>>>(row_id, row_p1, n_seq, nd, status, drafts, n_out,
                                                  conf, status_out);
  return cudaGetLastError();
}

// ------------------------------------------------------------ RoPE table --
// cos/sin of pos * inv_freq[i] for every position the head can reach,
// evaluated in double and stored f32 ([P1] field yarn_inv_freq).
__global__ void k_rope_table(const float *__restrict__ inv_freq, int max_pos, int half,
                             float *__restrict__ cos_t, float *__restrict__ sin_t) {
  int64_t n = (int64_t)max_pos * half;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n;
       t += (int64_t)gridDim.x * blockDim.x) {
    int pos = (int)(t / half), i = (int)(t % half);
    double a = (double)pos * (double)inv_freq[i];
    double sv, cv;
    sincos(a, &sv, &cv);
    cos_t[t] = (float)cv;
    sin_t[t] = (float)sv;
  }
}

cudaError_t rope_table(const float *inv_freq, int max_pos, int half, float *cos_t, float *sin_t,
                       cudaStream_t s) {
  k_rope_table<<<1024, 256, 0, s>>>(inv_freq, max_pos, half, cos_t, sin_t);
  return cudaGetLastError();
}

// ------------------------------------------------------- debug KV gather --
__global__ void k_gather_kv(const void *__restrict__ pool, Geo g, int layer,
                            const RowMeta *__restrict__ rows, const float *__restrict__ kv_scale,
                            float *k_out, float *v_out) {
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
  k_gather_kv<<<n, 256, 0, s>>>(pool, g, layer, rows, kv_scale, k_out, v_out);
  return cudaGetLastError();
}

}  // namespace dfl
