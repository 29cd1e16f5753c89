// Block attention of the draft head: for each sequence and kv head, the
// gamma block rows of every query head in the GQA group attend, without a
// mask, to the ctx window (paged K/V, bf16 or FP8 with per-head scales) and to
// the block's own gamma keys ([P1] fields kv_cache, ctx_window, layers;
// [P2] field propose_graphs: attention runs between the layer halves).
//
// Split-KV: the host cuts every (sequence, kv head) key range into chunks;
// each CTA takes one chunk and holds the whole group's gamma x (nq/nkv) query
// vectors (<= 128) as one Q tile of 64 or 128 rows. QK^T and PV run on tensor cores
// (mma.sync m16n8k16, bf16 in, f32 accumulate) with an online softmax in
// registers; K/V tiles of 32 keys stream through a double-buffered cp.async
// ring. A pair cut into several chunks writes unnormalised partials
// (acc, row max, row sum) that k_attn_merge combines; a pair of one chunk
// writes its output directly.
#include "attention.h"

#include <cmath>

#include "gemm_tc.h"

namespace dfl {

namespace {

constexpr int QT = 128;     // query vectors per CTA at most (rows of the Q tile)
constexpr int KT = 32;      // keys per K/V tile
constexpr int THREADS = 128;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  const int n = valid ? 16 : 0;   // zero-fill when invalid
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float fp8_to_float(uint8_t c) {
  __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(hr));
}

template <int D, int QR = QT>
struct Smem {
  static constexpr int LD = D + 8;   // padded row (bf16): conflict-free ldmatrix
  bf16 q[QR * LD];
  bf16 k[2][KT * LD];
  bf16 v[2][KT * LD];
};
// FP8 ctx keys: the raw E4M3 codes land here asynchronously (16 codes per
// copy), RS - 1 tiles ahead of the one being computed, and each tile is
// widened into a bf16 stage after its wait.
template <int MT>
constexpr int raw_stages() {
  return 2;   // (deeper rings measured slower: they cost a resident CTA per SM)
}
template <int D, int RS>
struct SmemRaw {
  uint8_t k[RS][KT * D];
  uint8_t v[RS][KT * D];
};
template <int D, bool FP8, int MT>
constexpr int attn_smem_bytes() {
  return (int)sizeof(Smem<D, 64 * MT>) + (FP8 ? (int)sizeof(SmemRaw<D, raw_stages<MT>()>) : 0);
}

// Loads keys [kt, kt+KT) of the item (key index space: [0, n_ctx) ctx rows at
// positions ws.., then the gamma block rows) into one K/V stage. Keys past
// k1 are zero-filled (and masked by the caller).
template <int D, int RS>
__device__ __forceinline__ void load_kv_tile_fp8(const AttnArgs &a, const AttnItem &it,
                                                 const SeqMeta &sm, SmemRaw<D, RS> *raw,
                                                 int stage, int kt, int *status) {
  constexpr int CH = D / 16;   // 16-byte chunks per row (E4M3 codes)
  const Geo &g = a.g;
  for (int idx = threadIdx.x; idx < KT * CH; idx += THREADS) {
    const int r = idx / CH, c = idx % CH;
    const int kk = kt + r;
    const bool valid = kk < it.k1;   // (a window item: every valid key is a ctx key)
    int64_t ko = 0, vo = 0;
    if (valid) {
      const int pos = sm.ws + kk;
      int page = a.page_ids[sm.page_base + (pos / g.B - sm.ws / g.B)];
      if (page < 0 || page >= g.pages) {
        atomicOr(status, ST_PAGE);
        page = 0;
      }
      ko = kv_offset(g, page, a.layer, 0, it.g, pos % g.B) + c * 16;
      vo = kv_offset(g, page, a.layer, 1, it.g, pos % g.B) + c * 16;
    }
    // a padding key past k1 lands as zero codes (masked out by the caller)
    cp_async16(smem_u32(raw->k[stage] + r * D + c * 16), (const uint8_t *)a.pool + ko, valid);
    cp_async16(smem_u32(raw->v[stage] + r * D + c * 16), (const uint8_t *)a.pool + vo, valid);
  }
}

// The raw codes of raw stage rs (every thread's copies complete and
// visible) widened exactly into the bf16 K/V stage.
template <int D, int RS, int QR>
__device__ __forceinline__ void widen_kv_stage(const SmemRaw<D, RS> *raw, int rs,
                                               Smem<D, QR> *sh, int stage) {
  constexpr int LD = Smem<D, QR>::LD;
  constexpr int CH = D / 16;
  for (int idx = threadIdx.x; idx < 2 * KT * CH; idx += THREADS) {
    const bool is_v = idx >= KT * CH;
    const int i = is_v ? idx - KT * CH : idx;
    const int r = i / CH, c = i % CH;
    const uint4 src = *reinterpret_cast<const uint4 *>((is_v ? raw->v[rs] : raw->k[rs]) +
                                                       r * D + c * 16);
    const uint32_t w[4] = {src.x, src.y, src.z, src.w};
    uint32_t o[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      o[2 * e] = pack_bf16(fp8_to_float(w[e] & 0xFF), fp8_to_float((w[e] >> 8) & 0xFF));
      o[2 * e + 1] = pack_bf16(fp8_to_float((w[e] >> 16) & 0xFF), fp8_to_float(w[e] >> 24));
    }
    bf16 *dst = (is_v ? sh->v[stage] : sh->k[stage]) + r * LD + c * 16;
    *reinterpret_cast<uint4 *>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4 *>(dst + 8) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

template <int D, bool FP8, int QR>
__device__ __forceinline__ void load_kv_tile(const AttnArgs &a, const AttnItem &it,
                                             const SeqMeta &sm, Smem<D, QR> *sh, int stage,
                                             int kt, int *status) {
  constexpr int LD = Smem<D, QR>::LD;
  constexpr int CH = D / 8;   // 16-byte chunks per row (bf16)
  const Geo &g = a.g;
  const int n_ctx = sm.pos - sm.ws;
  for (int idx = threadIdx.x; idx < KT * CH; idx += THREADS) {
    const int r = idx / CH, c = idx % CH;
    const int kk = kt + r;
    const bool valid = kk < it.k1;
    bf16 *dk = sh->k[stage] + r * LD + c * 8;
    bf16 *dv = sh->v[stage] + r * LD + c * 8;
    if (!valid) {
      // padding key past k1: zeros (masked out of the softmax by the caller)
      *reinterpret_cast<uint4 *>(dk) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4 *>(dv) = make_uint4(0, 0, 0, 0);
    } else if (kk < n_ctx) {
      // ctx key: position ws + kk, through the window's page list
      const int pos = sm.ws + kk;
      int page = a.page_ids[sm.page_base + (pos / g.B - sm.ws / g.B)];
      const int slot = pos % g.B;
      if (page < 0 || page >= g.pages) {
        atomicOr(status, ST_PAGE);
        page = 0;
      }
      const int64_t ko = kv_offset(g, page, a.layer, 0, it.g, slot) + c * 8;
      const int64_t vo = kv_offset(g, page, a.layer, 1, it.g, slot) + c * 8;
      if (FP8) {
        const uint2 kr = *reinterpret_cast<const uint2 *>((const uint8_t *)a.pool + ko);
        const uint2 vr = *reinterpret_cast<const uint2 *>((const uint8_t *)a.pool + vo);
        const uint8_t *kb = reinterpret_cast<const uint8_t *>(&kr);
        const uint8_t *vb = reinterpret_cast<const uint8_t *>(&vr);
        uint32_t ko4[4], vo4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          ko4[e] = pack_bf16(fp8_to_float(kb[2 * e]), fp8_to_float(kb[2 * e + 1]));
          vo4[e] = pack_bf16(fp8_to_float(vb[2 * e]), fp8_to_float(vb[2 * e + 1]));
        }
        *reinterpret_cast<uint4 *>(dk) = make_uint4(ko4[0], ko4[1], ko4[2], ko4[3]);
        *reinterpret_cast<uint4 *>(dv) = make_uint4(vo4[0], vo4[1], vo4[2], vo4[3]);
      } else {
        cp_async16(smem_u32(dk), (const bf16 *)a.pool + ko, true);
        cp_async16(smem_u32(dv), (const bf16 *)a.pool + vo, true);
      }
    } else {
      // block key: row (s*gamma + kk - n_ctx) of the block's own K/V
      const int64_t off = (int64_t)(it.s * g.gamma + kk - n_ctx) * g.kv + it.g * D + c * 8;
      if (FP8) {
        *reinterpret_cast<uint4 *>(dk) = *reinterpret_cast<const uint4 *>(a.kb + off);
        *reinterpret_cast<uint4 *>(dv) = *reinterpret_cast<const uint4 *>(a.vb + off);
      } else {
        cp_async16(smem_u32(dk), a.kb + off, true);
        cp_async16(smem_u32(dv), a.vb + off, true);
      }
    }
  }
}

template <int D, bool FP8, int MT>
__global__ void __launch_bounds__(THREADS) k_attn_split(AttnArgs a) {
  if ((int)blockIdx.x >= a.counts[0]) return;   // grid sized for the capacity
  pdl_trigger();
  pdl_wait();
  using SM = Smem<D, 64 * MT>;
  constexpr int LD = SM::LD;
  constexpr int NT = D / 8;          // n8 tiles across the head dim (output)
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SM *sh = reinterpret_cast<SM *>(smem_raw);
  constexpr int RS = raw_stages<MT>();
  SmemRaw<D, RS> *raw = reinterpret_cast<SmemRaw<D, RS> *>(smem_raw + sizeof(SM));
  const AttnItem it = a.items[blockIdx.x];
  const SeqMeta sm = a.seq[it.s];
  const Geo &g = a.g;
  const int grp = g.nq / g.nkv;
  const int n_q = g.gamma * grp;
  const int n_ctx = sm.pos - sm.ws;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;

  // Q tile: query vector qv = i * grp + hh is row i of the block, head g*grp+hh.
  for (int idx = threadIdx.x; idx < 64 * MT * (D / 8); idx += THREADS) {
    const int r = idx / (D / 8), c = idx % (D / 8);
    bf16 *dst = sh->q + r * LD + c * 8;
    const bool valid = r < n_q;
    const int64_t off = valid ? ((int64_t)(it.s * g.gamma + r / grp) * g.nq + it.g * grp + r % grp) * D + c * 8 : 0;
    cp_async16(smem_u32(dst), a.q + off, valid);
  }
  const bool is_ctx = it.k0 < n_ctx;
  float sk = 1.f, sv = 1.f;
  if (FP8 && is_ctx) {
    sk = a.kv_scale[(a.layer * g.nkv + it.g) * 2 + 0];
    sv = a.kv_scale[(a.layer * g.nkv + it.g) * 2 + 1];
  }
  const float qk_scale = a.scale * sk;
  const int n_tiles = (it.k1 - it.k0 + KT - 1) / KT;
  // FP8 ctx keys stream as raw codes (widened per stage below)
  const bool raw_kv = FP8 && is_ctx;
  if (raw_kv) {
    // one copy group per tile, RS - 1 tiles ahead (empty groups past the end)
    for (int i = 0; i < RS - 1; ++i) {
      if (i < n_tiles) load_kv_tile_fp8<D, RS>(a, it, sm, raw, i, it.k0 + i * KT, a.status);
      cp_commit();
    }
  } else {
    load_kv_tile<D, FP8, 64 * MT>(a, it, sm, sh, 0, it.k0, a.status);
    cp_commit();
  }

  float acc[MT][NT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
  float row_m[MT][2], row_l[MT][2];   // [m-tile][row gid / gid+8]
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    row_m[mt][0] = row_m[mt][1] = -INFINITY;
    row_l[mt][0] = row_l[mt][1] = 0.f;
  }
  const int qrow0 = warp * 16 * MT;   // this warp's 16 MT query rows

  for (int t = 0; t < n_tiles; ++t) {
    const int stage = t & 1;
    if (raw_kv) {
      const int ahead = t + RS - 1;
      if (ahead < n_tiles)
        load_kv_tile_fp8<D, RS>(a, it, sm, raw, ahead % RS, it.k0 + ahead * KT, a.status);
      cp_commit();
      cp_wait<RS - 1>();   // tile t's group has landed
      __syncthreads();
      widen_kv_stage<D, RS, 64 * MT>(raw, t % RS, sh, stage);
      __syncthreads();
    } else {
      if (t + 1 < n_tiles) {
        load_kv_tile<D, FP8, 64 * MT>(a, it, sm, sh, stage ^ 1, it.k0 + (t + 1) * KT, a.status);
        cp_commit();
        cp_wait<1>();
      } else {
        cp_wait<0>();
      }
      __syncthreads();
    }
    const int kt = it.k0 + t * KT;
    // S = Q K^T for this warp's 32 rows x 32 keys
    float s[MT][4][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[mt][j][e] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < D; k0 += 16) {
      uint32_t af[MT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int row = qrow0 + mt * 16 + (lane & 15);
        const int col = k0 + (lane >> 4) * 8;
        ldsm_x4(smem_u32(sh->q + row * LD + col), af[mt][0], af[mt][1], af[mt][2], af[mt][3]);
      }
#pragma unroll
      for (int jp = 0; jp < 2; ++jp) {   // pairs of n8 key tiles
        uint32_t b0, b1, b2, b3;
        const int key = jp * 16 + (lane >> 4) * 8 + (lane & 7);
        const int col = k0 + ((lane >> 3) & 1) * 8;
        ldsm_x4(smem_u32(sh->k[stage] + key * LD + col), b0, b1, b2, b3);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          mma16816(s[mt][2 * jp], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b0, b1);
          mma16816(s[mt][2 * jp + 1], af[mt][0], af[mt][1], af[mt][2], af[mt][3], b2, b3);
        }
      }
    }
    // online softmax over the tile's keys (masking keys >= k1)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {   // row gid (h=0) or gid+8 (h=1)
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = kt + j * 8 + 2 * tig + e;
            float v = s[mt][j][2 * h + e] * qk_scale;
            v = key < it.k1 ? v : -INFINITY;
            s[mt][j][2 * h + e] = v;
            mx = fmaxf(mx, v);
          }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(row_m[mt][h], mx);
        const float corr = (row_m[mt][h] == -INFINITY) ? 0.f : __expf(row_m[mt][h] - m_new);
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float v = s[mt][j][2 * h + e];
            const float p = (v == -INFINITY) ? 0.f : __expf(v - m_new);
            s[mt][j][2 * h + e] = p;
            sum += p;
          }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        row_l[mt][h] = row_l[mt][h] * corr + sum;
        row_m[mt][h] = m_new;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          acc[mt][nt][2 * h] *= corr;
          acc[mt][nt][2 * h + 1] *= corr;
        }
      }
    }
    // O += P V  (P from the S registers, values scaled by sv for FP8 ctx)
#pragma unroll
    for (int kc = 0; kc < 2; ++kc) {   // 16-key slices of the tile
      uint32_t pa[MT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        pa[mt][0] = pack_bf16(s[mt][2 * kc][0] * sv, s[mt][2 * kc][1] * sv);
        pa[mt][1] = pack_bf16(s[mt][2 * kc][2] * sv, s[mt][2 * kc][3] * sv);
        pa[mt][2] = pack_bf16(s[mt][2 * kc + 1][0] * sv, s[mt][2 * kc + 1][1] * sv);
        pa[mt][3] = pack_bf16(s[mt][2 * kc + 1][2] * sv, s[mt][2 * kc + 1][3] * sv);
      }
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {   // pairs of n8 dim tiles
        uint32_t b0, b1, b2, b3;
        const int key = kc * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int col = np * 16 + (lane >> 4) * 8;
        ldsm_x4_t(smem_u32(sh->v[stage] + key * LD + col), b0, b1, b2, b3);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          mma16816(acc[mt][2 * np], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], b0, b1);
          mma16816(acc[mt][2 * np + 1], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], b2, b3);
        }
      }
    }
    __syncthreads();   // the stage is reloaded two tiles later
  }

  // epilogue: direct output, or partials for the merge
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int qv = qrow0 + mt * 16 + gid + 8 * h;
      if (qv >= n_q) continue;
      if (it.slot < 0) {
        const float inv = 1.f / row_l[mt][h];
        bf16 *orow = a.o + ((int64_t)(it.s * g.gamma + qv / grp) * g.nq + it.g * grp + qv % grp) * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          *reinterpret_cast<__nv_bfloat162 *>(orow + nt * 8 + 2 * tig) =
              __floats2bfloat162_rn(acc[mt][nt][2 * h] * inv, acc[mt][nt][2 * h + 1] * inv);
      } else {
        float *ws = a.ws + (int64_t)it.slot * a.slot_floats;
        float *arow = ws + (int64_t)qv * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          *reinterpret_cast<float2 *>(arow + nt * 8 + 2 * tig) =
              make_float2(acc[mt][nt][2 * h], acc[mt][nt][2 * h + 1]);
        if (tig == 0) {
          ws[(int64_t)n_q * D + qv] = row_m[mt][h];
          ws[(int64_t)n_q * D + n_q + qv] = row_l[mt][h];
        }
      }
    }
  }
}

// One warp per (pair, query vector), 4 per block: combine the pair's chunks.
// Lane c holds chunk c's (m, l) (32 chunks per round); the weights reach the
// other lanes by shuffle, and every chunk's partial row is loaded before any
// is used.
template <int D>
__global__ void __launch_bounds__(128) k_attn_merge(AttnArgs a) {
  if ((int)blockIdx.x >= a.counts[1]) return;   // grid sized for the capacity
  pdl_trigger();
  const AttnPair pr = a.pairs[blockIdx.x];   // host-written: read before the wait
  pdl_wait();
  constexpr int VPL = D / 32;   // floats per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qv = blockIdx.y * 4 + warp;
  const Geo &g = a.g;
  const int grp = g.nq / g.nkv;
  const int n_q = g.gamma * grp;
  if (qv >= n_q) return;
  const int64_t off_m = (int64_t)n_q * D + qv, off_l = (int64_t)n_q * D + n_q + qv;
  // max over all chunks
  float M = -INFINITY;
  for (int c0 = 0; c0 < pr.nc; c0 += 32) {
    const int c = c0 + lane;
    if (c < pr.nc) M = fmaxf(M, __ldcg(a.ws + (int64_t)(pr.slot0 + c) * a.slot_floats + off_m));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float l = 0.f;
  float acc[VPL];
#pragma unroll
  for (int e = 0; e < VPL; ++e) acc[e] = 0.f;
  for (int c0 = 0; c0 < pr.nc; c0 += 32) {
    const int c = c0 + lane;
    float w = 0.f;
    if (c < pr.nc) {
      const float *ws = a.ws + (int64_t)(pr.slot0 + c) * a.slot_floats;
      const float m = __ldcg(ws + off_m);
      w = (m == -INFINITY) ? 0.f : __expf(m - M);
      l += w * __ldcg(ws + off_l);
    }
    const int nc = pr.nc - c0 < 32 ? pr.nc - c0 : 32;
    // rows of up to 8 chunks in flight, added in chunk order
    for (int b = 0; b < nc; b += 8) {
      float4 r[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (b + u < nc) {
          const float *row = a.ws + (int64_t)(pr.slot0 + c0 + b + u) * a.slot_floats +
                             (int64_t)qv * D + lane * VPL;
          if constexpr (VPL == 4) r[u] = __ldcg(reinterpret_cast<const float4 *>(row));
          else r[u] = make_float4(__ldcg(row), __ldcg(row + 1), 0.f, 0.f);
        } else {
          r[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float wu = __shfl_sync(0xffffffffu, w, (b + u) & 31);
        if (b + u < nc) {
          acc[0] += wu * r[u].x;
          acc[1] += wu * r[u].y;
          if constexpr (VPL == 4) {
            acc[2] += wu * r[u].z;
            acc[3] += wu * r[u].w;
          }
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  const float inv = 1.f / l;
  bf16 *orow = a.o + ((int64_t)(pr.s * g.gamma + qv / grp) * g.nq + pr.g * grp + qv % grp) * D +
               lane * VPL;
#pragma unroll
  for (int e = 0; e < VPL; e += 2)
    *reinterpret_cast<__nv_bfloat162 *>(orow + e) =
        __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
}


// The same merge for a grid of a few blocks per SM (batch 1: one pair per kv
// head, many chunks). The partial rows do not depend on the maximum, so the
// first MERGE_ROWS of them are loaded together with the (m, l) pairs: a pair
// of up to MERGE_ROWS chunks takes one L2 round trip (at ~128 registers, which
// would cost the many-pair grids their resident blocks).
constexpr int MERGE_ROWS = 24;
template <int D>
__global__ void __launch_bounds__(128) k_attn_merge_wide(AttnArgs a) {
  if ((int)blockIdx.x >= a.counts[1]) return;   // grid sized for the capacity
  pdl_trigger();
  const AttnPair pr = a.pairs[blockIdx.x];   // host-written: read before the wait
  pdl_wait();
  constexpr int VPL = D / 32;   // floats per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qv = blockIdx.y * 4 + warp;
  const Geo &g = a.g;
  const int grp = g.nq / g.nkv;
  const int n_q = g.gamma * grp;
  if (qv >= n_q) return;
  const int64_t off_m = (int64_t)n_q * D + qv, off_l = (int64_t)n_q * D + n_q + qv;
  const float *ws0 = a.ws + (int64_t)pr.slot0 * a.slot_floats;
  auto row4 = [&](int c) -> float4 {
    const float *row = ws0 + (int64_t)c * a.slot_floats + (int64_t)qv * D + lane * VPL;
    if constexpr (VPL == 4) return __ldcg(reinterpret_cast<const float4 *>(row));
    else return make_float4(__ldcg(row), __ldcg(row + 1), 0.f, 0.f);
  };
  float4 r[MERGE_ROWS];
#pragma unroll
  for (int u = 0; u < MERGE_ROWS; ++u) r[u] = u < pr.nc ? row4(u) : make_float4(0.f, 0.f, 0.f, 0.f);
  const float m0 = lane < pr.nc ? __ldcg(ws0 + (int64_t)lane * a.slot_floats + off_m) : -INFINITY;
  const float l0 = lane < pr.nc ? __ldcg(ws0 + (int64_t)lane * a.slot_floats + off_l) : 0.f;
  // max over all chunks
  float M = m0;
  for (int c = lane + 32; c < pr.nc; c += 32)
    M = fmaxf(M, __ldcg(ws0 + (int64_t)c * a.slot_floats + off_m));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float l = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int c0 = 0; c0 < pr.nc; c0 += 32) {
    const int c = c0 + lane;
    float w = 0.f;
    if (c < pr.nc) {
      const float *ws = ws0 + (int64_t)c * a.slot_floats;
      const float m = c0 == 0 ? m0 : __ldcg(ws + off_m);
      w = (m == -INFINITY) ? 0.f : __expf(m - M);
      l += w * (c0 == 0 ? l0 : __ldcg(ws + off_l));
    }
    const int nc = pr.nc - c0 < 32 ? pr.nc - c0 : 32;
    // chunk rows added in chunk order; the first batch is already loaded
    for (int b = 0; b < nc; b += MERGE_ROWS) {
      if (c0 > 0 || b > 0) {
#pragma unroll
        for (int u = 0; u < MERGE_ROWS; ++u)
          r[u] = b + u < nc ? row4(c0 + b + u) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < MERGE_ROWS; ++u) {
        const float wu = __shfl_sync(0xffffffffu, w, (b + u) & 31);
        if (b + u < nc) {
          acc[0] += wu * r[u].x;
          acc[1] += wu * r[u].y;
          acc[2] += wu * r[u].z;
          acc[3] += wu * r[u].w;
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  const float inv = 1.f / l;
  bf16 *orow = a.o + ((int64_t)(pr.s * g.gamma + qv / grp) * g.nq + pr.g * grp + qv % grp) * D +
               lane * VPL;
#pragma unroll
  for (int e = 0; e < VPL; e += 2)
    *reinterpret_cast<__nv_bfloat162 *>(orow + e) =
        __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
}

template <int D, bool FP8, int MT>
cudaError_t launch(const AttnArgs &a, cudaStream_t s) {
  const int smem = attn_smem_bytes<D, FP8, MT>();
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_split<D, FP8, MT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  launch_pdl(k_attn_split<D, FP8, MT>, dim3(a.n_items), dim3(THREADS), smem, s, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return attention_merge(a, s);
}

}  // namespace

int attn_query_rows(const Geo &g) { return g.gamma * (g.nq / g.nkv); }

cudaError_t attention_merge(const AttnArgs &a, cudaStream_t s) {
  if (a.n_pairs == 0) return cudaSuccess;   // capacity 0: no ctx window at all
  const int grp = a.g.nq / a.g.nkv;
  const dim3 grid(a.n_pairs, (a.g.gamma * grp + 3) / 4);
  const bool wide = (int64_t)grid.x * grid.y <= 2 * (int64_t)tc::num_sms();
  if (a.g.d == 128) {
    if (wide) launch_pdl(k_attn_merge_wide<128>, grid, dim3(128), 0, s, a);
    else launch_pdl(k_attn_merge<128>, grid, dim3(128), 0, s, a);
  } else if (a.g.d == 64) {
    if (wide) launch_pdl(k_attn_merge_wide<64>, grid, dim3(128), 0, s, a);
    else launch_pdl(k_attn_merge<64>, grid, dim3(128), 0, s, a);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t attention_split(const AttnArgs &a, cudaStream_t s) {
  if (a.n_items <= 0) return cudaSuccess;
  const int rows = attn_query_rows(a.g);
  if (rows > QT) return cudaErrorInvalidValue;
  // a Q tile of 64 rows when the group's queries fit (half the MMA work)
  if (rows <= 64) {
    if (a.g.d == 128) return a.g.kv_fp8 ? launch<128, true, 1>(a, s) : launch<128, false, 1>(a, s);
    if (a.g.d == 64) return a.g.kv_fp8 ? launch<64, true, 1>(a, s) : launch<64, false, 1>(a, s);
  } else {
    if (a.g.d == 128) return a.g.kv_fp8 ? launch<128, true, 2>(a, s) : launch<128, false, 2>(a, s);
    if (a.g.d == 64) return a.g.kv_fp8 ? launch<64, true, 2>(a, s) : launch<64, false, 2>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dfl
