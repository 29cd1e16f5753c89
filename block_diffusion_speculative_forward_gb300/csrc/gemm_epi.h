// The fused epilogues of the tensor-core GEMMs, shared by the single-GEMM
// kernel (gemm_tc.cu) and the multi-phase batch-1 kernel (chain.cu). Each
// runs on the four epilogue warps (128 threads, named barrier 1), one thread
// per accumulator row (a weight row = an output feature f) holding 16
// accumulator columns (activation rows a0..a0+15).
#pragma once

#include "gemm_tc.h"
#include "internal.h"
#include "tc_ptx.h"

namespace dfl {
namespace tc {

constexpr int BM = 128;                 // weight rows per tile
constexpr int BK = 64;                  // K elements per stage (one 128-byte swizzle span)
constexpr int A_BYTES = BM * BK * 2;    // 16 KB

// Cross-thread scratch of the epilogue warps.
struct EpiScratch {
  float red_v[4][16];
  int red_i[4][16];
  float col_max[16];
  float xch[16][128];   // per-column exchange between the tile's rows (fused epilogues only)
};

// Draft row of activation row a of an lm_head launch (-1: none) and its
// sequence. Activations are either the draft rows themselves (lm_gamma 0;
// row a belongs to sequence a / nd) or whole blocks of lm_gamma rows, whose
// rows lm_first .. lm_first + nd - 1 are the sequence's draft rows.
__device__ __forceinline__ int lm_row(const GemmParams &p, int a, int *seq) {
  if (a >= p.m_act) return -1;
  if (p.lm_gamma == 0) {
    *seq = a / p.nd;
    return a;
  }
  *seq = a / p.lm_gamma;
  const int j = a % p.lm_gamma - p.lm_first;
  return (j >= 0 && j < p.nd) ? *seq * p.nd + j : -1;
}

// Applies the epilogue to 16 accumulator columns held by this thread
// (feature row f of tile tm, activation rows a0..a0+15); et is the thread's
// index among the 128 epilogue threads.
template <int EPI>
__device__ __forceinline__ void finish16(const GemmParams &p, EpiScratch *sm, const float (&v)[16],
                                         int f, int tm, int a0, int q, int lane, int et) {
  const bool f_ok = f < p.n_w;
  if (EPI == EPI_TC_LMHEAD) {
    // Per activation row: max / lowest argmax / sum exp over this tile's 128
    // vocab rows, with the grammar bitmask (bit f of the sequence's mask).
    float val[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      int seq;
      bool ok = f_ok && lm_row(p, a0 + c, &seq) >= 0;
      if (ok && p.bitmask) {
        const uint32_t w = (uint32_t)p.bitmask[(int64_t)seq * p.mask_words + (f >> 5)];
        ok = (w >> (f & 31)) & 1u;
      }
      float x = v[c];
      if (p.wscale && f_ok) x *= p.wscale[f];
      if (p.gscale != 0.f) x *= p.gscale;
      val[c] = ok ? x : -INFINITY;
    }
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      float m = val[c];
      int id = val[c] == -INFINITY ? INT32_MAX : f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float om = __shfl_xor_sync(0xffffffffu, m, o);
        int oi = __shfl_xor_sync(0xffffffffu, id, o);
        if (om > m || (om == m && oi < id)) { m = om; id = oi; }
      }
      if (lane == 0) { sm->red_v[q][c] = m; sm->red_i[q][c] = id; }
    }
    epi_bar();
    if (et < 16) {
      const int c = et;
      float m = sm->red_v[0][c];
      int id = sm->red_i[0][c];
      for (int w = 1; w < 4; ++w) {
        float om = sm->red_v[w][c];
        int oi = sm->red_i[w][c];
        if (om > m || (om == m && oi < id)) { m = om; id = oi; }
      }
      sm->col_max[c] = m;
      sm->red_i[0][c] = id;   // keep the winner for the write below
    }
    epi_bar();
    float s[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float m = sm->col_max[c];
      float e = (m == -INFINITY || val[c] == -INFINITY) ? 0.f : __expf(val[c] - m);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
      s[c] = e;
    }
    epi_bar();   // red_v reuse below: everyone has read col_max/red_i
    if (lane == 0) {
#pragma unroll
      for (int c = 0; c < 16; ++c) sm->red_v[q][c] = s[c];
    }
    epi_bar();
    if (et < 16) {
      const int c = et;
      int seq;
      const int drow = lm_row(p, a0 + c, &seq);
      if (drow >= 0) {
        LmPartial r;
        r.max = sm->col_max[c];
        r.id = sm->red_i[0][c];
        r.sum = sm->red_v[0][c] + sm->red_v[1][c] + sm->red_v[2][c] + sm->red_v[3][c];
        r.pad = 0;
        p.lm_part[(int64_t)drow * p.tiles_m + tm] = r;
      }
    }
    epi_bar();
    return;
  }
  if (EPI == EPI_TC_QKV) {
    // Per-head RMSNorm (gain q_norm / k_norm) then RoPE over the full head for
    // q and k rows; v rows are stored as they are. A 128-row tile lies in one
    // region and holds 128 / head_dim whole heads. The rotation of the 16
    // rows is loaded before the first barrier.
    const int fl = q * 32 + lane;
    const int d = p.head_dim;
    const int tile0 = tm * BM;
    const int nrows = p.m_act - a0 < 16 ? p.m_act - a0 : 16;
    if (tile0 >= p.q_rows + p.k_rows) {
      bf16 *dst = p.v_out + (int64_t)a0 * p.k_rows + (f - p.q_rows - p.k_rows);
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (c < nrows) dst[(int64_t)c * p.k_rows] = __float2bfloat16_rn(v[c]);
      return;
    }
    const bool is_q = tile0 < p.q_rows;
    const bf16 *gain = is_q ? p.q_norm : p.k_norm;
    const int i = fl % d;
    const int half = d / 2;
    float cs[16], sn[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int a = a0 + c;
      const int pos = c < nrows ? p.seq[a / p.gamma].pos + a % p.gamma : 0;
      cs[c] = p.cos_t[(int64_t)pos * half + (i % half)];
      sn[c] = p.sin_t[(int64_t)pos * half + (i % half)];
    }
    const float gi = __bfloat162float(gain[i]);
    float ss[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) ss[c] = v[c] * v[c];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int c = 0; c < 16; ++c) ss[c] += __shfl_xor_sync(0xffffffffu, ss[c], o);
    if (lane == 0) {
#pragma unroll
      for (int c = 0; c < 16; ++c) sm->red_v[q][c] = ss[c];
    }
    epi_bar();
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      float tot;
      if (d == 128) tot = sm->red_v[0][c] + sm->red_v[1][c] + sm->red_v[2][c] + sm->red_v[3][c];
      else tot = sm->red_v[q & 2][c] + sm->red_v[(q & 2) + 1][c];   // d == 64: warps {0,1} / {2,3}
      sm->xch[c][fl] = gi * (v[c] * rsqrtf(tot / (float)d + p.eps));
    }
    epi_bar();
    bf16 *dst = is_q ? p.q_out + (int64_t)a0 * p.q_rows + f
                     : p.k_out + (int64_t)a0 * p.k_rows + (f - p.q_rows);
    const int ld = is_q ? p.q_rows : p.k_rows;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float y = sm->xch[c][fl];
      const float other = sm->xch[c][fl ^ half];
      const float o = (i < half) ? (y * cs[c] - other * sn[c]) : (y * cs[c] + other * sn[c]);
      if (c < nrows) dst[(int64_t)c * ld] = __float2bfloat16_rn(o);
    }
    epi_bar();
    return;
  }
  if (EPI == EPI_TC_SWIGLU) {
    // Weight rows alternate gate / up of one feature (row 2j gate j, 2j+1 up
    // j): the pair sits in lanes (2i, 2i+1) of a warp. The 16 columns run
    // phase by phase (all shuffles, all exponentials, then the stores) so the
    // dependent chains overlap. silu(g) = g / (1 + e^-g), the exponent
    // clamped at 80 so the fast divide stays in range (silu(g) < 1e-33 there).
    const int ldu = p.n_w / 2;
    float up[16], y[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) up[c] = __shfl_xor_sync(0xffffffffu, v[c], 1);
#pragma unroll
    for (int c = 0; c < 16; ++c)
      y[c] = __fdividef(v[c], 1.f + __expf(fminf(-v[c], 80.f))) * up[c];
    if (!(lane & 1) && f_ok) {
      bf16 *dst = p.u_out + (int64_t)a0 * ldu + (f >> 1);
      if (a0 + 16 <= p.m_act) {
#pragma unroll
        for (int c = 0; c < 16; ++c) dst[(int64_t)c * ldu] = __float2bfloat16_rn(y[c]);
      } else {
        const int n = p.m_act - a0;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (c < n) dst[(int64_t)c * ldu] = __float2bfloat16_rn(y[c]);
      }
    }
    return;
  }
  if (!f_ok) return;
  const float sc = (p.wscale ? p.wscale[f] : 1.f) * (p.gscale != 0.f ? p.gscale : 1.f);
  const int nrows = p.m_act - a0 < 16 ? p.m_act - a0 : 16;
  if (EPI == EPI_TC_ADD_F32) {
    // all loads first, then the stores
    float *o = (float *)p.out + (int64_t)a0 * p.ldo + f;
    float r[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) r[c] = c < nrows ? o[(int64_t)c * p.ldo] : 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c)
      if (c < nrows) o[(int64_t)c * p.ldo] = r[c] + v[c] * sc;
  } else {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      if (c >= nrows) break;
      const int64_t off = (int64_t)(a0 + c) * p.ldo + f;
      if (EPI == EPI_TC_STORE_F32) ((float *)p.out)[off] = v[c] * sc;
      else ((bf16 *)p.out)[off] = __float2bfloat16_rn(v[c] * sc);
    }
  }
}


}  // namespace tc
}  // namespace dfl
