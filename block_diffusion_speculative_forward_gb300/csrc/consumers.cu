// Consumers of the projections: each reads a GEMM's output through a
// Partials view (dense, or the k-segment partials summed in a fixed order)
// and applies the step that follows that projection in the layer:
//   residual add + RMSNorm   (o_proj, down_proj, fc -> hidden_norm, final norm)
//   per-head q/k RMSNorm + RoPE   (after the stitched QKV projection)
// Sources: [P1] "Struct BlockDiffusionDraftHead" fields hidden_norm, norm,
// layers, rms_norm_eps, rotary_dim, yarn_inv_freq.
#include "consumers.h"

#include <cooperative_groups.h>
#include <cuda_fp16.h>

namespace dfl {

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One block of 1024 threads per row: x[a] (+)= y[a]; out = bf16(g * x / rms(x)).
__global__ void __launch_bounds__(1024) k_add_norm(AddNormArgs p) {
  pdl_trigger();
  __shared__ float sh[32];
  __shared__ TileRange tr[32];
  const int a = blockIdx.x;
  const int n = p.n;
  constexpr int MAXE = 4;    // up to 4096 features per row
  // contributor ranges depend on no earlier kernel: before the wait
  if (p.has_y && p.y.ws && threadIdx.x < (n + 127) / 128)
    tr[threadIdx.x] = part_range(p.y, part_tile(p.y, a, threadIdx.x * 128));
  __syncthreads();
  pdl_wait();
  float xv[MAXE];
  float ss = 0.f;
#pragma unroll
  for (int t = 0; t < MAXE; ++t) {
    const int f = threadIdx.x + t * 1024;
    if (f < n) {
      float v = p.x ? p.x[(int64_t)a * n + f] : 0.f;
      if (p.has_y) v += p.y.ws ? part_sum(p.y, tr[f >> 7], a, f) : part_value(p.y, a, f);
      xv[t] = v;
      ss += v * v;
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 32; ++w) tot += sh[w];
  const float inv = rsqrtf(tot / (float)n + p.eps);
  // draft-row index of this row, or -1
  int drow = -1;
  if (p.z) {
    const int i = a % p.gamma - p.first;
    if (i >= 0 && i < p.nd) drow = (a / p.gamma) * p.nd + i;
  }
#pragma unroll
  for (int t = 0; t < MAXE; ++t) {
    const int f = threadIdx.x + t * 1024;
    if (f < n) {
      const float v = xv[t];
      if (p.x && p.has_y) p.x[(int64_t)a * n + f] = v;
      if (p.x_tap) p.x_tap[(int64_t)a * n + f] = v;
      const bf16 h = __float2bfloat16_rn(__bfloat162float(p.g[f]) * (v * inv));
      if (p.out) p.out[(int64_t)a * n + f] = h;
      if (p.z_tap) p.z_tap[(int64_t)a * n + f] = h;
      if (drow >= 0) {
        p.z[(int64_t)drow * n + f] = h;
        if (p.z16) p.z16[(int64_t)drow * n + f] = __half_as_ushort(__float2half_rn(__bfloat162float(h)));
      }
    }
  }
}

// Few rows: a cluster of CL CTAs per row, each CTA holding n / CL features
// (a warp's 32 features lie in one 128-feature tile). Each CTA reduces its
// sum of squares; the row total comes from the peers' shared memory.
constexpr int NORM_CL = 8;
__global__ void __launch_bounds__(256) k_add_norm_cl(AddNormArgs p) {
  namespace cg = cooperative_groups;
  pdl_trigger();
  __shared__ float red[8];
  __shared__ float cta_ss;
  cg::cluster_group cl = cg::this_cluster();
  const int a = blockIdx.x / NORM_CL;
  const int part = (int)cl.block_rank();
  const int n = p.n, per = n / NORM_CL;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int MAXE = 2;   // up to 512 features per CTA
  // contributor ranges and gains depend on no earlier kernel: before the wait
  TileRange tr[MAXE];
  float gv[MAXE];
#pragma unroll
  for (int t = 0; t < MAXE; ++t) {
    const int fl = threadIdx.x + t * 256;
    const int f = part * per + fl;
    tr[t] = TileRange{};
    gv[t] = 0.f;
    if (fl < per) {
      if (p.has_y && p.y.ws) tr[t] = part_range(p.y, part_tile(p.y, a, f & ~31));
      gv[t] = __bfloat162float(p.g[f]);
    }
  }
  pdl_wait();
  float xv[MAXE];
  float ss = 0.f;
#pragma unroll
  for (int t = 0; t < MAXE; ++t) {
    const int fl = threadIdx.x + t * 256;
    const int f = part * per + fl;
    xv[t] = 0.f;
    if (fl < per) {
      float v = p.x ? p.x[(int64_t)a * n + f] : 0.f;
      if (p.has_y) {
        if (p.y.ws) {
          v += part_sum_wide(p.y, tr[t], a, f);
        } else {
          v += p.y.dense[(int64_t)a * p.y.ld + f];
        }
      }
      xv[t] = v;
      ss += v * v;
    }
  }
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += red[w];
    cta_ss = t;
  }
  cl.sync();
  float tot = 0.f;
#pragma unroll
  for (int r = 0; r < NORM_CL; ++r) tot += *cl.map_shared_rank(&cta_ss, r);
  // the peers' sums are read (the release orders those loads): arrive now,
  // wait before exiting, the stores in between
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  const float inv = rsqrtf(tot / (float)n + p.eps);
  int drow = -1;
  if (p.z) {
    const int i = a % p.gamma - p.first;
    if (i >= 0 && i < p.nd) drow = (a / p.gamma) * p.nd + i;
  }
#pragma unroll
  for (int t = 0; t < MAXE; ++t) {
    const int fl = threadIdx.x + t * 256;
    const int f = part * per + fl;
    if (fl < per) {
      const float v = xv[t];
      if (p.x && p.has_y) p.x[(int64_t)a * n + f] = v;
      if (p.x_tap) p.x_tap[(int64_t)a * n + f] = v;
      const bf16 h = __float2bfloat16_rn(gv[t] * (v * inv));
      if (p.out) p.out[(int64_t)a * n + f] = h;
      if (p.z_tap) p.z_tap[(int64_t)a * n + f] = h;
      if (drow >= 0) {
        p.z[(int64_t)drow * n + f] = h;
        if (p.z16) p.z16[(int64_t)drow * n + f] = __half_as_ushort(__float2half_rn(__bfloat162float(h)));
      }
    }
  }
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");   // peers have read cta_ss
}

// Warp per (row, head): q and k heads take RMSNorm with their gain and RoPE at
// the row's position; v is rounded to bf16. From partials (few rows) the v
// features take a y-block of their own, so that no head's CTA runs two
// passes of partial sums; from a dense matrix the first head block copies
// them after its heads.
template <int NP>
__global__ void __launch_bounds__(256) k_qkv_post(QkvPostArgs p) {
  pdl_trigger();
  const Geo &g = p.g;
  const int r = blockIdx.x;
  if (p.y.ws && (int)blockIdx.y == (g.nq + g.nkv + 7) / 8) {
    // v rows: a warp's 32 consecutive features share one tile; the ranges
    // depend on no earlier kernel (before the wait)
    constexpr int MAXV = 4;
    const int vbase = g.nq * g.d + g.kv;
    for (int e0 = 0; e0 < g.kv; e0 += 256 * MAXV) {
      TileRange tv[MAXV];
#pragma unroll
      for (int u = 0; u < MAXV; ++u) {
        const int e = e0 + threadIdx.x + 256 * u;
        tv[u] = TileRange{};
        if (e < g.kv) tv[u] = part_range(p.y, part_tile(p.y, r, (vbase + e) & ~31));
      }
      pdl_wait();
      float y[MAXV];
#pragma unroll
      for (int u = 0; u < MAXV; ++u) {
        const int e = e0 + threadIdx.x + 256 * u;
        y[u] = 0.f;
        if (e < g.kv)
          y[u] = part_sum_wide(p.y, tv[u], r, vbase + e);
      }
#pragma unroll
      for (int u = 0; u < MAXV; ++u) {
        const int e = e0 + threadIdx.x + 256 * u;
        if (e < g.kv) p.vb[(int64_t)r * g.kv + e] = __float2bfloat16_rn(y[u]);
      }
    }
    return;
  }
  const int head = blockIdx.y * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int d = g.d, half = d / 2;
  const int pos = p.seq[r / g.gamma].pos + r % g.gamma;
  if (head < g.nq + g.nkv) {
    const bool is_q = head < g.nq;
    const int base = is_q ? head * d : g.nq * d + (head - g.nq) * d;
    // the head's features lie in one 128-feature tile (d divides 128 or
    // equals it): one contributor range for the warp
    TileRange tr{};
    if (p.y.ws) tr = part_range(p.y, part_tile(p.y, r, base));
    // the range, gains and rotation depend on no earlier kernel: before the wait
    const bf16 *gain = is_q ? p.q_norm : p.k_norm;
    float gn[2 * NP], cs[NP], sn[NP];
#pragma unroll
    for (int t = 0; t < NP; ++t) {
      const int i = lane + 32 * t;
      gn[2 * t] = __bfloat162float(gain[i]);
      gn[2 * t + 1] = __bfloat162float(gain[i + half]);
      cs[t] = p.cos_t[(int64_t)pos * half + i];
      sn[t] = p.sin_t[(int64_t)pos * half + i];
    }
    pdl_wait();
    float v[2 * NP];
    float ss = 0.f;
#pragma unroll
    for (int t = 0; t < NP; ++t) {
      const int f0 = base + lane + 32 * t, f1 = f0 + half;
      v[2 * t] = p.y.ws ? part_sum_wide(p.y, tr, r, f0) : p.y.dense[(int64_t)r * p.y.ld + f0];
      v[2 * t + 1] = p.y.ws ? part_sum_wide(p.y, tr, r, f1) : p.y.dense[(int64_t)r * p.y.ld + f1];
      ss += v[2 * t] * v[2 * t] + v[2 * t + 1] * v[2 * t + 1];
    }
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / (float)d + g.eps);
    bf16 *dst = is_q ? p.q + (int64_t)r * g.nq * d + head * d
                     : p.kb + (int64_t)r * g.kv + (head - g.nq) * d;
#pragma unroll
    for (int t = 0; t < NP; ++t) {
      const int i = lane + 32 * t;
      const float x1 = gn[2 * t] * (v[2 * t] * inv);
      const float x2 = gn[2 * t + 1] * (v[2 * t + 1] * inv);
      dst[i] = __float2bfloat16_rn(x1 * cs[t] - x2 * sn[t]);
      dst[i + half] = __float2bfloat16_rn(x2 * cs[t] + x1 * sn[t]);
    }
  }
  if (!p.y.ws && blockIdx.y == 0) {
    pdl_wait();
    const int vbase = g.nq * d + g.kv;
    for (int e = threadIdx.x; e < g.kv; e += blockDim.x)
      p.vb[(int64_t)r * g.kv + e] = __float2bfloat16_rn(p.y.dense[(int64_t)r * p.y.ld + vbase + e]);
  }
}

}  // namespace

cudaError_t add_norm(const AddNormArgs &p, int rows, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (p.n > 4 * 1024) return cudaErrorInvalidValue;
  // fewer rows than a quarter of the SMs: spread each row over a cluster
  const int per = p.n / NORM_CL;
  if (rows * 4 <= tc::num_sms() && p.n % NORM_CL == 0 && per % 32 == 0 && per <= 512)
    return launch_pdl_cluster(k_add_norm_cl, dim3(rows * NORM_CL), dim3(256), 0, s, NORM_CL, p);
  return launch_pdl(k_add_norm, dim3(rows), dim3(1024), 0, s, p);
}

cudaError_t qkv_post(const QkvPostArgs &p, int R, cudaStream_t s) {
  dim3 grid(R, (p.g.nq + p.g.nkv + 7) / 8 + (p.y.ws ? 1 : 0));   // (+ the v block)
  if (p.g.d == 128) return launch_pdl(k_qkv_post<2>, grid, dim3(256), 0, s, p);
  if (p.g.d == 64) return launch_pdl(k_qkv_post<1>, grid, dim3(256), 0, s, p);
  return cudaErrorInvalidValue;
}


}  // namespace dfl
