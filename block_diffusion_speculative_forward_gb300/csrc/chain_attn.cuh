// Block attention inside a chained launch (included by chain.cu): the four
// epilogue warps of a chain CTA run it while the weight producer keeps
// streaming the next projection's weights.
//
// For each sequence s and query head j, the gamma block rows (at most 16, one
// mma.sync M tile) attend without a mask to the window's ctx keys and to the
// block's own gamma keys of kv head j / (nq / nkv) ([P1] fields kv_cache,
// ctx_window, layers). Keys come in tiles of 16: ctx tile t holds positions
// p0 + 16 t .. p0 + 16 t + 15 (p0 = the window start rounded down to a page,
// so a tile is one page: K and V of the (layer, kv head) are 16 contiguous
// rows there), and the last tile holds the block keys. An item is a range
// of tiles of one (s, j); the four warps take its tiles in turn, each with
// an online softmax over its tiles (S = Q K^T and O += P V on mma.sync
// m16n8k16, bf16 in, f32 accumulate, P rounded to bf16), K/V pages arriving
// by TMA into a per-warp double buffer. The warps combine in shared memory
// into the item's partial (row max, row sum, unnormalised output); the last
// item of an (s, j) to finish merges the pair's partials, writes the bf16
// output rows and raises head j's ready count.
#pragma once

namespace dfl {
namespace tc {

// Shared memory of the attention part of a chain CTA.
constexpr int CA_D_MAX = 128;
constexpr int CA_QLD = CA_D_MAX + 8;                    // padded Q row (bf16)
constexpr int CA_Q_BYTES = 16 * CA_QLD * 2;             // 4352
constexpr int CA_KV_BYTES = 2 * 16 * CA_D_MAX * 2;      // K tile then V tile: 8 KB
constexpr int CA_WARP_BYTES = 2 * CA_KV_BYTES;          // double buffer: 16 KB
constexpr int CA_Q_OFF = 4 * CA_WARP_BYTES;               // warp buffers first (1024-aligned)
constexpr int CA_BYTES = CA_Q_OFF + CA_Q_BYTES;

__device__ __forceinline__ void ca_ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                           uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ca_ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                             uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ca_mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                       uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t ca_pack(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
// Byte offset of (row r, element col) in a tile of 64-element halves, each
// [16 rows][128 bytes] with the 128-byte swizzle TMA writes.
__device__ __forceinline__ uint32_t ca_sw(int r, int col) {
  return (uint32_t)((col >> 6) * 2048 + r * 128 + ((((col & 63) >> 3) ^ (r & 7)) << 4));
}

// Loads key tile t of an item into buffer `buf` of this warp (lane 0 issues;
// the warp's kv barrier receives the bytes). Ctx tile: page page_ids[...] of
// the pool at (layer, kv head); block tile: the block rows of sequence s.
template <int D>
__device__ __forceinline__ void ca_issue(const ChainAttn &A, const CUtensorMap *maps, int layer,
                                         const SeqMeta &sq, int s, int g, int t, int n_ctx_tiles,
                                         uint32_t buf, uint32_t bar, int *status) {
  constexpr int HALVES = D / 64;
  const uint64_t pol = policy_evict_first();
  mbar_expect_tx(bar, 2 * HALVES * 2048);
  if (t < n_ctx_tiles) {
    const int p0 = sq.ws & ~15;
    const int page_idx = sq.page_base + (p0 + 16 * t) / 16 - sq.ws / 16;
    int page = A.page_ids[page_idx];
    if (page < 0 || page >= A.geo.pages) {
      atomicOr(status, ST_PAGE);
      page = 0;
    }
    const int row_k = (((page * A.geo.L + layer) * 2) * A.geo.nkv + g) * 16;
    const int row_v = row_k + A.geo.nkv * 16;
#pragma unroll
    for (int h = 0; h < HALVES; ++h) {
      tma_load_2d(buf + h * 2048, maps + 0, bar, h * 64, row_k, pol);
      tma_load_2d(buf + HALVES * 2048 + h * 2048, maps + 0, bar, h * 64, row_v, pol);
    }
  } else {
    const int row = s * A.geo.gamma;
#pragma unroll
    for (int h = 0; h < HALVES; ++h) {
      tma_load_2d(buf + h * 2048, maps + 1, bar, g * D + h * 64, row, pol);
      tma_load_2d(buf + HALVES * 2048 + h * 2048, maps + 2, bar, g * D + h * 64, row, pol);
    }
  }
}

// One item on the four epilogue warps (et = 0..127, q = warp & 3).
// Returns false when a wait gave up (the CTA then aborts).
template <int D>
__device__ bool ca_item(const ChainAttn &A, const CUtensorMap *maps, int layer, const ChainPhase &P,
                        const ChainAttnItem it, uint8_t *abase, uint32_t abase_s,
                        uint32_t kv_bar0, uint32_t &kv_par, EpiScratch *sm_epi, int *is_last,
                        volatile int *abort_flag, int *status, int et, int q, int lane) {
  constexpr int NT = D / 8;
  constexpr int HALVES = D / 64;
  const Geo &g = A.geo;
  const int grp = g.nq / g.nkv;
  const int kvh = it.j / grp;
  const SeqMeta sq = A.seq[it.s];
  const int n_ctx = sq.pos - sq.ws;
  const int p0 = sq.ws & ~15;
  const int n_ctx_tiles = n_ctx > 0 ? (sq.pos - p0 + 15) / 16 : 0;
  const int gid = lane >> 2, tig = lane & 3;
  const uint32_t qs = abase_s + CA_Q_OFF;                    // Q [16][CA_QLD]
  bf16 *qp = reinterpret_cast<bf16 *>(abase + CA_Q_OFF);
  const uint32_t wbuf = abase_s + q * CA_WARP_BYTES;
  const uint32_t bar0 = kv_bar0 + q * 16, bar1 = bar0 + 8;  // this warp's two kv barriers

  // this warp's tiles: t0 + q, t0 + q + 4, ...; issue the first two
  const int my_n = it.t1 - it.t0 > q ? (it.t1 - it.t0 - q + 3) / 4 : 0;
  if (lane == 0) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    for (int i = 0; i < 2 && i < my_n; ++i)
      ca_issue<D>(A, maps, layer, sq, it.s, kvh, it.t0 + q + 4 * i, n_ctx_tiles, wbuf + i * CA_KV_BYTES,
                  i ? bar1 : bar0, status);
  }
  // Q rows of the item: block rows s*gamma + r (r < gamma), head j; the rest zero
  for (int idx = et; idx < 16 * (D / 8); idx += 128) {
    const int r = idx / (D / 8), c = idx % (D / 8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < g.gamma)
      v = *reinterpret_cast<const uint4 *>(A.q + ((int64_t)(it.s * g.gamma + r) * g.nq + it.j) * D + c * 8);
    *reinterpret_cast<uint4 *>(qp + r * CA_QLD + c * 8) = v;
  }
  epi_bar();
  uint32_t qf[D / 16][4];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks)
    ca_ldsm_x4(qs + ((lane & 15) * CA_QLD + ks * 16 + (lane >> 4) * 8) * 2, qf[ks][0], qf[ks][1],
               qf[ks][2], qf[ks][3]);

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
  float row_m[2] = {-INFINITY, -INFINITY}, row_l[2] = {0.f, 0.f};
  bool ok = true;
  int waited = 0;
  for (int i = 0; i < my_n; ++i) {
    const int b = i & 1;
    const uint32_t bar = b ? bar1 : bar0;
    if (!mbar_wait_warp(bar, (kv_par >> (q * 2 + b)) & 1u, abort_flag)) { ok = false; break; }
    waited = i + 1;
    kv_par ^= 1u << (q * 2 + b);
    const uint32_t kt = wbuf + b * CA_KV_BYTES, vt = kt + HALVES * 2048;
    const int t = it.t0 + q + 4 * i;
    // S = Q K^T: 16 rows x 16 keys (two n8 tiles)
    float s[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[j][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t b0, b1, b2, b3;
      const int key = (lane >> 4) * 8 + (lane & 7);
      const int col = ks * 16 + ((lane >> 3) & 1) * 8;
      ca_ldsm_x4(kt + ca_sw(key, col), b0, b1, b2, b3);
      ca_mma(s[0], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
      ca_mma(s[1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
    }
    // keys of the tile inside the item: ctx positions in [ws, pos); block keys < gamma
    const bool block = t >= n_ctx_tiles;
    const int kbase = block ? 0 : p0 + 16 * t;
    const int klo = block ? 0 : sq.ws, khi = block ? g.gamma : sq.pos;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = kbase + j * 8 + 2 * tig + e;
          float v = s[j][2 * h + e] * A.scale;
          v = (key >= klo && key < khi) ? v : -INFINITY;
          s[j][2 * h + e] = v;
          mx = fmaxf(mx, v);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(row_m[h], mx);
      const float corr = (row_m[h] == -INFINITY) ? 0.f : __expf(row_m[h] - m_new);
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float v = s[j][2 * h + e];
          const float p = (v == -INFINITY) ? 0.f : __expf(v - m_new);
          s[j][2 * h + e] = p;
          sum += p;
        }
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      row_l[h] = row_l[h] * corr + sum;
      row_m[h] = m_new;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        acc[nt][2 * h] *= corr;
        acc[nt][2 * h + 1] *= corr;
      }
    }
    // O += P V (16 keys, one k16 slice)
    const uint32_t pa0 = ca_pack(s[0][0], s[0][1]), pa1 = ca_pack(s[0][2], s[0][3]);
    const uint32_t pa2 = ca_pack(s[1][0], s[1][1]), pa3 = ca_pack(s[1][2], s[1][3]);
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
      uint32_t b0, b1, b2, b3;
      const int key = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int col = np * 16 + (lane >> 4) * 8;
      ca_ldsm_x4_t(vt + ca_sw(key, col), b0, b1, b2, b3);
      ca_mma(acc[2 * np], pa0, pa1, pa2, pa3, b0, b1);
      ca_mma(acc[2 * np + 1], pa0, pa1, pa2, pa3, b2, b3);
    }
    // the buffer is read: refill it with this warp's tile i + 2
    __syncwarp();
    if (lane == 0 && i + 2 < my_n) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      ca_issue<D>(A, maps, layer, sq, it.s, kvh, t + 8, n_ctx_tiles, kt, bar, status);
    }
  }
  if (!ok && lane == 0) {
    // giving up: let this warp's copies still in flight land (bounded)
    const int issued = my_n < waited + 2 ? my_n : waited + 2;
    for (int i = waited; i < issued; ++i) {
      const int b = i & 1;
      const uint32_t par = (kv_par >> (q * 2 + b)) & 1u;
      const uint64_t t0 = global_ns();
      while (!mbar_test(b ? bar1 : bar0, par) && global_ns() - t0 < 100000000ull) {
      }
      kv_par ^= 1u << (q * 2 + b);
    }
  }
  // every warp has passed its loads' barriers (or gave up): the buffers
  // become the combine area
  if (!epi_all(ok)) return false;
  float *cm = reinterpret_cast<float *>(abase);                // [4][16] max, then [4][16] sum
  float *cacc = cm + 128;                                        // [4][16][D]
  if (tig == 0) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      cm[q * 16 + gid + 8 * h] = row_m[h];
      cm[64 + q * 16 + gid + 8 * h] = row_l[h];
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int h = 0; h < 2; ++h)
      *reinterpret_cast<float2 *>(cacc + (q * 16 + gid + 8 * h) * D + nt * 8 + 2 * tig) =
          make_float2(acc[nt][2 * h], acc[nt][2 * h + 1]);
  epi_bar();
  // thread et: row r = et / 8, D / 8 consecutive dims; the item's partial
  constexpr int PD = D / 8;
  const int r = et >> 3, d0 = (et & 7) * PD;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < 4; ++w) M = fmaxf(M, cm[w * 16 + r]);
  float wt[4], L = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float mw = cm[w * 16 + r];
    wt[w] = (mw == -INFINITY) ? 0.f : __expf(mw - M);
    L += wt[w] * cm[64 + w * 16 + r];
  }
  float *slot = A.ws + (int64_t)it.slot * (16 * D + 32);
#pragma unroll
  for (int e = 0; e < PD; e += 4) {
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float4 c = *reinterpret_cast<const float4 *>(cacc + (w * 16 + r) * D + d0 + e);
      o.x += wt[w] * c.x;
      o.y += wt[w] * c.y;
      o.z += wt[w] * c.z;
      o.w += wt[w] * c.w;
    }
    *reinterpret_cast<float4 *>(slot + r * D + d0 + e) = o;
  }
  if ((et & 7) == 0) {
    slot[16 * D + r] = M;
    slot[16 * D + 16 + r] = L;
  }
  // arrival of the item at its (s, j) pair; the last merges
  epi_bar();
  if (et == 0) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                 : "=r"(old)
                 : "l"(P.arrive + it.s * g.nq + it.j)
                 : "memory");
    *is_last = (old == it.nc - 1);
  }
  epi_bar();
  if (!*is_last) return true;
  // merge: chunks slot0 .. slot0 + nc - 1 of the pair, in order, four
  // partials in flight, with a running max
  float Mp = -INFINITY;
  float o[PD], Lp = 0.f;
#pragma unroll
  for (int e = 0; e < PD; ++e) o[e] = 0.f;
  for (int c0 = 0; c0 < it.nc; c0 += 4) {
    float4 v[4][PD / 4];
    float mc[4], lc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool live = c0 + u < it.nc;
      const float *sl = A.ws + (int64_t)(it.slot0 + (live ? c0 + u : 0)) * (16 * D + 32);
      mc[u] = live ? __ldcg(sl + 16 * D + r) : -INFINITY;
      lc[u] = live ? __ldcg(sl + 16 * D + 16 + r) : 0.f;
#pragma unroll
      for (int e = 0; e < PD / 4; ++e)
        v[u][e] = live ? __ldcg(reinterpret_cast<const float4 *>(sl + r * D + d0) + e)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mx = Mp;
#pragma unroll
    for (int u = 0; u < 4; ++u) mx = fmaxf(mx, mc[u]);
    if (mx > Mp) {
      const float f = (Mp == -INFINITY) ? 0.f : __expf(Mp - mx);
      Lp *= f;
#pragma unroll
      for (int e = 0; e < PD; ++e) o[e] *= f;
      Mp = mx;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = (mc[u] == -INFINITY) ? 0.f : __expf(mc[u] - Mp);
      Lp += w * lc[u];
#pragma unroll
      for (int e = 0; e < PD / 4; ++e) {
        o[4 * e] += w * v[u][e].x;
        o[4 * e + 1] += w * v[u][e].y;
        o[4 * e + 2] += w * v[u][e].z;
        o[4 * e + 3] += w * v[u][e].w;
      }
    }
  }
  if (r < g.gamma) {
    const float inv = 1.f / Lp;
    bf16 *orow = A.o + ((int64_t)(it.s * g.gamma + r) * g.nq + it.j) * D + d0;
#pragma unroll
    for (int e = 0; e < PD; e += 2)
      *reinterpret_cast<__nv_bfloat162 *>(orow + e) = __floats2bfloat162_rn(o[e] * inv, o[e + 1] * inv);
  }
  // publish: head j's ready count (one per sequence) and the pair count
  epi_bar();
  if (et == 0) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(P.flag + it.j), "r"(1) : "memory");
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(P.done), "r"(1) : "memory");
  }
  return true;
}

}  // namespace tc
}  // namespace dfl
