// tcgen05/TMA weight-streaming GEMM: parameters and host entry points.
#pragma once

#include <cuda.h>

#include "internal.h"

namespace dfl {

enum TcEpi {
  EPI_TC_STORE_F32 = 0,   // out[a, f] = y
  EPI_TC_ADD_F32 = 1,     // out[a, f] += y        (residual stream)
  EPI_TC_STORE_BF16 = 2,  // out[a, f] = bf16(y)
  EPI_TC_LMHEAD = 3,      // per (row, 128-row vocab tile): max, lowest argmax, sum exp
  EPI_TC_QKV = 4,         // stitched q;k;v rows: per-head RMSNorm + RoPE for q and k, bf16 out
  EPI_TC_SWIGLU = 5,      // gate/up rows alternating: u = silu(gate) * up, bf16 out
  EPI_TC_PARTIAL = 6,     // every k-segment writes its f32 partial; the consumer sums them
};

// The output of a GEMM as its consumer reads it: either a dense f32 matrix,
// or the k-segment partials of an EPI_TC_PARTIAL launch. Element (a, f) of a
// partial view is the sum, in ascending CTA order, of the partials of the
// CTAs whose k-ranges cover tile (f / 128, a / bn): the same value a fused
// epilogue would see, without any inter-CTA synchronisation in the GEMM.
struct Partials {
  const float *ws = nullptr;     // partial slots, or NULL for a dense matrix
  const float *dense = nullptr;  // [rows, ld]
  int ld = 0;
  int tiles_m = 0, kb = 0, G = 0, bn = 0, total = 0;
};

__device__ __forceinline__ int part_begin(int total, int G, int c) {
  return (int)(((unsigned)total * (unsigned)c) / (unsigned)G);
}
__device__ __forceinline__ int part_owner(int total, int G, int i) {
  int c = (int)(((unsigned)i * (unsigned)G) / (unsigned)total);
  while (c + 1 < G && part_begin(total, G, c + 1) <= i) ++c;
  while (c > 0 && part_begin(total, G, c) > i) --c;
  return c;
}

// Contributors of one tile: CTAs c_lo..c_hi; c_lo's segment of the tile is
// its second one when lo_second.
struct TileRange {
  int c_lo, c_hi, lo_second;
};
__device__ __forceinline__ TileRange part_range(const Partials &P, int t) {
  const int i0 = t * P.kb;
  TileRange r;
  r.c_lo = part_owner(P.total, P.G, i0);
  r.c_hi = part_owner(P.total, P.G, i0 + P.kb - 1);
  r.lo_second = part_begin(P.total, P.G, r.c_lo) < i0 ? 1 : 0;
  return r;
}
// Partial slots are laid out [slot][bn rows][128 features]; contributors are
// added in ascending CTA order. part_sum keeps four loads in flight (for the
// many-row consumers, whose threads each sum several features);
// part_sum_wide issues the first PART_BATCH contributors' loads together, so
// one L2 round trip covers every tile of the few-row projections (at most 11
// contributors at batch 1). Both give the same sum.
__device__ __forceinline__ float part_sum(const Partials &P, const TileRange &r, int a, int f) {
  const float *base = P.ws + (a % P.bn) * 128 + (f & 127);
  const long long stride = (long long)P.bn * 128;
  float s = __ldcg(base + (2 * r.c_lo + r.lo_second) * stride);
  for (int c = r.c_lo + 1; c <= r.c_hi; c += 4) {
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = (c + u <= r.c_hi) ? __ldcg(base + 2 * (c + u) * stride) : 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) s += v[u];
  }
  return s;
}
constexpr int PART_BATCH = 12;
__device__ __forceinline__ float part_sum_wide(const Partials &P, const TileRange &r, int a, int f) {
  const float *base = P.ws + (a % P.bn) * 128 + (f & 127);
  const long long stride = (long long)P.bn * 128;
  float b[PART_BATCH];
#pragma unroll
  for (int u = 0; u < PART_BATCH; ++u) {
    const int c = r.c_lo + u;
    b[u] = c <= r.c_hi ? __ldcg(base + (2 * c + (u == 0 ? r.lo_second : 0)) * stride) : 0.f;
  }
  float s = b[0];
#pragma unroll
  for (int u = 1; u < PART_BATCH; ++u) s += b[u];
  for (int c = r.c_lo + PART_BATCH; c <= r.c_hi; c += 4) {
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = (c + u <= r.c_hi) ? __ldcg(base + 2 * (c + u) * stride) : 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) s += v[u];
  }
  return s;
}
// N features f[n] of one row and one tile (one contributor range) at once:
// the first PART_BATCH contributors' loads of every feature are issued
// together. Each sum has part_sum_wide's order.
template <int N>
__device__ __forceinline__ void part_sum_multi(const Partials &P, const TileRange &r, int a,
                                               const int (&f)[N], float (&out)[N]) {
  const float *base = P.ws + (a % P.bn) * 128;
  const long long stride = (long long)P.bn * 128;
  float b[PART_BATCH][N];
#pragma unroll
  for (int u = 0; u < PART_BATCH; ++u) {
    const int c = r.c_lo + u;
    const float *slot = base + (2 * c + (u == 0 ? r.lo_second : 0)) * stride;
#pragma unroll
    for (int n = 0; n < N; ++n) b[u][n] = c <= r.c_hi ? __ldcg(slot + (f[n] & 127)) : 0.f;
  }
#pragma unroll
  for (int n = 0; n < N; ++n) {
    float s = b[0][n];
#pragma unroll
    for (int u = 1; u < PART_BATCH; ++u) s += b[u][n];
    out[n] = s;
  }
  for (int c = r.c_lo + PART_BATCH; c <= r.c_hi; ++c) {
#pragma unroll
    for (int n = 0; n < N; ++n) out[n] += __ldcg(base + 2 * c * stride + (f[n] & 127));
  }
}
__device__ __forceinline__ int part_tile(const Partials &P, int a, int f) {
  return (a / P.bn) * P.tiles_m + (f >> 7);
}
__device__ __forceinline__ float part_value(const Partials &P, int a, int f) {
  if (!P.ws) return P.dense[(long long)a * P.ld + f];
  return part_sum(P, part_range(P, part_tile(P, a, f)), a, f);
}

// One (row, vocab tile) partial of the lm_head reduction.
struct LmPartial {
  float max;
  int32_t id;   // INT32_MAX when nothing in the tile is allowed
  float sum;    // sum over the tile of exp(logit - max)
  int32_t pad;
};

struct GemmParams {
  int m_act;          // activation rows
  int n_w;            // weight rows (output features)
  int k;              // reduction length, multiple of 64
  int epi;
  void *out;          // [m_act, ldo] f32 or bf16 (not LMHEAD)
  int ldo;
  const float *wscale;  // per weight row scale or NULL
  float gscale;         // lm_head: every logit times this (0: none)
  // stream-K
  float *ws;          // partial slots: 2 * grid * BN * 128 floats
  int *counters;      // per tile, zero between launches
  int grid_cap;       // 0 = one CTA per SM
  int dp;             // 1: data-parallel whole tiles (fused epilogues), no stream-K split
  // lm_head
  const int32_t *bitmask;  // [n_seq][mask_words] or NULL
  int mask_words;
  int nd;             // draft rows per sequence (row a belongs to sequence a / nd)
  int lm_gamma;       // 0: activations are draft rows; > 0: blocks of lm_gamma rows whose
  int lm_first;       //   rows lm_first .. lm_first + nd - 1 are the draft rows
  LmPartial *lm_part; // [draft rows][tiles_m]
  int *status;
  // QKV epilogue: rows [0, q_rows) are q heads, [q_rows, q_rows + k_rows) k
  // heads, the rest v; row a of the activations is block row a % gamma of
  // sequence a / gamma, at position seq[a / gamma].pos + a % gamma.
  const SeqMeta *seq;
  int gamma, head_dim, q_rows, k_rows;
  const bf16 *q_norm, *k_norm;
  const float *cos_t, *sin_t;
  float eps;
  bf16 *q_out, *k_out, *v_out;   // [m_act, q_rows], [m_act, k_rows], [m_act, k_rows]
  // SwiGLU epilogue: u[m_act, n_w / 2]
  bf16 *u_out;
  // test hook: > 0 makes every CTA abort after waiting this long (ns) on a
  // barrier that nothing arrives on (the bounded-wait abort path)
  int64_t fault_ns;
  // filled by the launcher
  int tiles_m, tiles_n;
};

// The fused lm_head + row reductions (lmhead_tc.cu).
struct LmArgs {
  int m_act;               // draft rows
  int n_w;                 // vocab
  int k;                   // hidden, multiple of 64
  const int32_t *bitmask;  // [n_seq][mask_words] or NULL
  int mask_words;
  int nd;                  // draft rows per sequence
  const float *wscale;     // per vocab row scale (FP8 head) or NULL
  float gscale;            // every logit times this (NVFP4 head's global scale; 0: none)
  LmPartial *out;          // [m_act][vocab tiles of 256]
  int *status;
};

namespace tc {
int num_sms();
// map_x: draft rows, box 128 rows; map_w: vocab rows, box 256 rows.
cudaError_t lmhead(const CUtensorMap &map_x, const CUtensorMap &map_w, const LmArgs &p,
                   cudaStream_t s);
int lmhead_vocab_tiles(int vocab);
int pick_bn(int m_act);
// Weight-only low-precision lm_head (lm_lowp.cu) over at most 16 draft
// rows: FP8 E4M3 codes with the per-row scale in GemmParams::wscale, or
// NVFP4 codes with block scales and the global factor in GemmParams::gscale.
// map_codes: [V, k] or [V, k/2] bytes (128-byte swizzled boxes of 128 rows x
// 128 bytes); map_scales: [V, k/16] bytes (boxes of 128 rows x 16 bytes,
// NVFP4 only); map_z: the draft rows [m_act, k] as f16 in boxes of 16 rows x
// 64. p.epi is EPI_TC_LMHEAD (per-row partials in lm_part, tiles_m =
// ceil(V/128)) or EPI_TC_STORE_F32 (logits to out). lm_lowp_fits says which
// shapes it takes (m_act <= 16, k a multiple of 256, at most 2048).
enum { LM_LOWP_FP8 = 1, LM_LOWP_NVFP4 = 2 };
bool lm_lowp_fits(int m_act, int k);
cudaError_t lm_lowp(int fmt, const CUtensorMap &map_codes, const CUtensorMap &map_scales,
                    const CUtensorMap &map_z, const GemmParams &p, cudaStream_t s);
// A 2D map of a byte table [rows, cols] (cols a multiple of 4) with boxes of
// box_rows x box_bytes, 128-byte swizzled or not. Its x coordinate counts
// 4-byte words: byte column c is x = c / 4.
bool make_map_u8(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int box_bytes,
                 int box_rows, bool swizzle128);
// Tile width for a data-parallel (whole-tile) launch of this shape.
int pick_bn_dp(int m_act, int n_w, int k);
// 2-D row-major map [rows, cols], box = 128 bytes of a row x box_rows rows, 128B swizzle.
bool make_map_2d(CUtensorMap *map, const void *base, bool fp8, int64_t rows, int64_t cols,
                 int box_rows);
// 3-D bf16 map (dims innermost first, byte strides of dims 1 and 2), 128B
// swizzle; box[0] * 2 bytes must be 128.
bool make_map_3d(CUtensorMap *map, const void *base, const int64_t dims[3],
                 const int64_t strides_bytes[2], const int box[3]);
// Launches the GEMM. For EPI_TC_PARTIAL, *view receives the partials' layout.
cudaError_t gemm(const CUtensorMap &map_w, const CUtensorMap &map_x, int bn, GemmParams p,
                 cudaStream_t s, Partials *view = nullptr);
// Whether EPI_TC_PARTIAL can serve this shape: every CTA's k-range must span
// at most two tiles (two partial slots per CTA).
bool partial_ok(int m_act, int n_w, int k);
// Bytes of stream-K partial workspace for the widest tile and a full grid.
inline size_t ws_floats(int grid) { return (size_t)2 * grid * 256 * 128; }
}  // namespace tc

// Merges the lm_head partials of each draft row: (argmax id or -1, top-1 prob).
cudaError_t lm_reduce(const LmPartial *part, int rows, int tiles, int32_t *row_id, float *row_p1,
                      cudaStream_t s);

}  // namespace dfl
