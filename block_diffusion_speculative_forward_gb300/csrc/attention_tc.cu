// Block attention on the 5th-generation tensor cores (bf16 KV cache, head dim
// 128): for each sequence and kv head, the gamma block rows of every query
// head in the GQA group attend, without a mask, to the ctx window and to the
// block's own gamma keys ([P1] fields kv_cache, ctx_window, layers).
//
// Work: the same split-KV items as the mma.sync kernel (attention.cu), run by
// one persistent CTA per SM over a host-balanced list of items. Per item the
// group's gamma x (nq / nkv) <= 128 query vectors are the M = 128 operand;
// keys stream in tiles of 64 (four 16-key pages) through a 4-stage TMA ring
// straight from the paged pool. Per tile:
//   S   = Q K^T   tcgen05, M 128 x N 64 x K 128, into TMEM (double buffered)
//   P   = exp(S * scale - m)  by four softmax warps, one thread per query
//         vector, written to shared memory as bf16 (double buffered)
//   O_t = P V     tcgen05, M 128 x N 128 x K 64 with V as an MN-major operand,
//         into TMEM (double buffered); the softmax thread folds O_t into its
//         register accumulator with the running-max correction.
// Keys outside the item (ragged page edges) are masked to -inf; 16-key groups
// holding no key of the item are neither loaded nor multiplied. An item
// writes its normalised output, or (acc, max, sum) partials for the merge.
// Warp roles: warp 0 TMA producer, warp 1 MMA issuer (and TMEM owner),
// warps 2-5 softmax. Every wait is bounded.
#include <cuda.h>

#include "attention.h"
#include "gemm_tc.h"
#include "tc_ptx.h"

namespace dfl {

namespace {

using namespace tc;

constexpr int AQ = 128;                      // query vectors per tile (MMA M)
constexpr int AD = 128;                      // head dim
constexpr int AK = 64;                       // keys per tile
constexpr int KV_STAGES = 4;
constexpr int Q_BYTES = AQ * AD * 2;         // 32 KB: two 64-column halves
constexpr int Q_HALF = Q_BYTES / 2;
constexpr int P_BYTES = AQ * AK * 2;         // 16 KB
constexpr int KT_BYTES = AK * AD * 2;        // 16 KB: two 64-column halves
constexpr int KT_HALF = KT_BYTES / 2;
constexpr int STAGE_BYTES = 2 * KT_BYTES;    // K tile then V tile
constexpr int GROUP_BYTES = 16 * 128;        // one 16-key page half: 16 rows x 128 B
constexpr int OFF_P = 2 * Q_BYTES;
constexpr int OFF_KV = OFF_P + 2 * P_BYTES;
constexpr int TILE_BYTES = OFF_KV + KV_STAGES * STAGE_BYTES;   // 224 KB
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_S = 0;               // two 64-column S buffers
constexpr uint32_t TMEM_O = 128;             // two 128-column O accumulators (items alternate)

struct Bars {
  uint64_t q_full[2], q_empty[2], kv_full[KV_STAGES], kv_empty[KV_STAGES];
  uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2], o_free[2], drain;
  uint32_t tmem_base;
  uint32_t q_issued, q_parity, kv_issued, kv_parity;
  int abort_flag;
};
constexpr int SMEM = 1024 + TILE_BYTES + (int)sizeof(Bars);
static_assert(SMEM <= 232448, "attention tile exceeds the 227 KB shared-memory limit");

// Key range of an item in the tile's coordinates: ctx items count positions
// (tile j starts at p0 + 64 j, p0 the item's first position rounded down to a
// page), the block item counts its keys from 0.
struct ItemGeo {
  int lo, hi, p0, ntiles;
  bool block;
};

__device__ __forceinline__ ItemGeo item_geo(const AttnItem &it, const SeqMeta &sm, int gamma) {
  ItemGeo r;
  const int n_ctx = sm.pos - sm.ws;
  r.block = it.k0 >= n_ctx;
  if (r.block) {
    r.lo = 0;
    r.hi = gamma;
    r.p0 = 0;
  } else {
    r.lo = sm.ws + it.k0;
    r.hi = sm.ws + it.k1;
    r.p0 = r.lo & ~15;
  }
  r.ntiles = (r.hi - r.p0 + AK - 1) / AK;
  return r;
}

// Bit q: the tile's keys 16q..16q+15 include a key of the item.
__device__ __forceinline__ uint32_t group_mask(const ItemGeo &ig, int j) {
  const int base = ig.p0 + j * AK;
  uint32_t m = 0;
#pragma unroll
  for (int q = 0; q < AK / 16; ++q)
    if (base + 16 * q < ig.hi) m |= 1u << q;
  return m;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *map, uint32_t bar, int x,
                                            int y, int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// Pulls a 2D box of a tensor map into L2 (a hint: no shared memory, no
// barrier, and later loads still see every write).
__device__ __forceinline__ void tma_prefetch_l2(const void *map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(map), "r"(x),
               "r"(y)
               : "memory");
}

// Descriptor of an MN-major operand in the 128-byte swizzle: rows of 64
// consecutive N elements (128 B), 8 K-rows per 1024-byte atom; lbo = bytes
// between 64-wide N blocks, sbo = bytes between 8-row K groups.
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
      "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __launch_bounds__(THREADS, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_pool,
              const __grid_constant__ CUtensorMap map_kb, const __grid_constant__ CUtensorMap map_vb,
              AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  Bars *bar = (Bars *)(smem_raw + (base - raw) + TILE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Geo &g = a.g;
  const int grp = g.nq / g.nkv;
  const int n_q = g.gamma * grp;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bar->q_full[b]), 1);
      mbar_init(smem_u32(&bar->q_empty[b]), 1);
      mbar_init(smem_u32(&bar->s_full[b]), 1);
      mbar_init(smem_u32(&bar->s_empty[b]), 4);
      mbar_init(smem_u32(&bar->p_full[b]), 4);
      mbar_init(smem_u32(&bar->p_empty[b]), 1);
      mbar_init(smem_u32(&bar->o_free[b]), 4);
    }
    for (int s = 0; s < KV_STAGES; ++s) {
      mbar_init(smem_u32(&bar->kv_full[s]), 1);
      mbar_init(smem_u32(&bar->kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&bar->drain), 1);
    bar->abort_flag = 0;
    bar->q_issued = bar->q_parity = bar->kv_issued = bar->kv_parity = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_q) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_pool) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_kb) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_vb) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&bar->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The work list, sequence table and page ids are written by the host before
  // the launch, so they are read before waiting for the previous kernel: warp
  // 0 reads its first item's and pulls that item's first KV_STAGES tiles of
  // K/V pages into L2 (lane 4j + q: group q of tile j); the reads after the
  // wait then hit L1 and L2.
  const int c_begin = a.cta_off[blockIdx.x], c_end = a.cta_off[blockIdx.x + 1];
  if (warp == 0 && c_begin < c_end) {
    const AttnItem it = a.items[c_begin];
    const SeqMeta sm = a.seq[it.s];
    const ItemGeo ig = item_geo(it, sm, g.gamma);
    const int j = lane >> 2, q = lane & 3;
    if (!ig.block && j < KV_STAGES && j < ig.ntiles && ((group_mask(ig, j) >> q) & 1u)) {
      const int pos = ig.p0 + j * AK + 16 * q;
      const int page = a.page_ids[sm.page_base + pos / 16 - sm.ws / 16];
      if (page >= 0 && page < g.pages) {
        const int row_k = (((page * g.L + a.layer) * 2) * g.nkv + it.g) * 16;
        const int row_v = row_k + g.nkv * 16;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          tma_prefetch_l2(&map_pool, h * 64, row_k);
          tma_prefetch_l2(&map_pool, h * 64, row_v);
        }
      }
    }
  }
  pdl_trigger();
  pdl_wait();
  const uint32_t tmem = bar->tmem_base;
  volatile int *abort_flag = &bar->abort_flag;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer ------
    // The whole warp runs the loop (each wait gives one answer per warp);
    // lane 0 arms the barriers and issues Q, and the 16 boxes of a K/V tile
    // (group q, half h, K or V) are issued in parallel by lanes 4q + 2h + kv:
    // one thread issuing them back to back took ~2 us per tile.
    const uint64_t pol_kv = policy_evict_first();
    const uint64_t pol_q = policy_evict_normal();
    uint32_t q_issued = 0, q_par = 0, kv_issued = 0, kv_par = 0;
    int stage = 0;
    uint32_t kv_phase = 0;
    int qi = 0;
    const int lq = lane >> 2, lh = (lane >> 1) & 1, lkv = lane & 1;   // this lane's box (lanes < 16)
    for (int c = c_begin; c < c_end; ++c, ++qi) {
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const AttnItem it = a.items[c];
      const SeqMeta sm = a.seq[it.s];
      const ItemGeo ig = item_geo(it, sm, g.gamma);
      const int qb = qi & 1;
      const uint32_t qph = (qi >> 1) & 1;
      if (!mbar_wait_warp(smem_u32(&bar->q_empty[qb]), qph ^ 1, abort_flag)) break;
      if (lane == 0) {
        const uint32_t qf = smem_u32(&bar->q_full[qb]);
        mbar_expect_tx(qf, 2 * 64 * n_q * 2);
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tma_load_3d(base + qb * Q_BYTES + h * Q_HALF, &map_q, qf, h * 64, it.g * grp,
                      it.s * g.gamma, pol_q);
      }
      q_issued |= 1u << qb;
      q_par = (q_par & ~(1u << qb)) | (qph << qb);
      bool ok = true;
      for (int j = 0; j < ig.ntiles; ++j) {
        if (!mbar_wait_warp(smem_u32(&bar->kv_empty[stage]), kv_phase ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t gm = group_mask(ig, j);
        const uint32_t sb = base + OFF_KV + stage * STAGE_BYTES;
        const uint32_t fb = smem_u32(&bar->kv_full[stage]);
        if (lane == 0) mbar_expect_tx(fb, __popc(gm) * 4 * GROUP_BYTES);
        __syncwarp();
        if (lane < 16 && ((gm >> lq) & 1u)) {
          const uint32_t dst = sb + lkv * KT_BYTES + lh * KT_HALF + lq * GROUP_BYTES;
          if (!ig.block) {
            const int pos = ig.p0 + j * AK + 16 * lq;
            int page = a.page_ids[sm.page_base + pos / 16 - sm.ws / 16];
            if (page < 0 || page >= g.pages) {
              atomicOr(a.status, ST_PAGE);
              page = 0;
            }
            const int row = ((((page * g.L + a.layer) * 2) + lkv) * g.nkv + it.g) * 16;
            tma_load_2d(dst, &map_pool, fb, lh * 64, row, pol_kv);
          } else {
            const int row = it.s * g.gamma + j * AK + 16 * lq;
            tma_load_2d(dst, lkv ? &map_vb : &map_kb, fb, it.g * AD + lh * 64, row, pol_q);
          }
        }
        kv_issued |= 1u << stage;
        kv_par = (kv_par & ~(1u << stage)) | (kv_phase << stage);
        if (++stage == KV_STAGES) {
          stage = 0;
          kv_phase ^= 1;
        }
      }
      if (!ok) break;
    }
    if (lane == 0) {
      bar->q_issued = q_issued;
      bar->q_parity = q_par;
      bar->kv_issued = kv_issued;
      bar->kv_parity = kv_par;
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer --------
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_mn<AQ, AK>();
      const uint32_t idesc_o = idesc_bf16_mn<AQ, AD>() | (1u << 16);   // B (V) MN-major
      int stage = 0;
      uint32_t kv_phase = 0;
      int T = 0, qi = 0;
      bool have_prev = false, prev_first = false;
      int prev_T = 0, prev_stage = 0, prev_qi = 0;
      uint32_t prev_gm = 0;
      bool ok = true;
      // O[item % 2] (+)= P_t V_t; the item's first tile starts the accumulator
      auto issue_pv = [&](int t, int st, uint32_t gm, int item, bool first) -> bool {
        const int pb = t & 1, ob = item & 1;
        if (!mbar_wait(smem_u32(&bar->p_full[pb]), (t >> 1) & 1, abort_flag)) return false;
        if (first && !mbar_wait(smem_u32(&bar->o_free[ob]), ((item >> 1) & 1) ^ 1, abort_flag))
          return false;
        tc_fence_after();
        const uint32_t d = tmem + TMEM_O + ob * AD;
        const uint32_t pa = base + OFF_P + pb * P_BYTES;
        const uint32_t vb = base + OFF_KV + st * STAGE_BYTES + KT_BYTES;
        uint32_t acc = first ? 0u : 1u;
#pragma unroll
        for (int kq = 0; kq < AK / 16; ++kq) {
          if (!((gm >> kq) & 1u)) continue;
          umma_bf16(d, sw128_desc(pa + kq * 32), sw128_desc_mn(vb + kq * 16 * 128, KT_HALF, 1024),
                    idesc_o, acc);
          acc = 1;
        }
        umma_commit(smem_u32(&bar->p_empty[pb]));
        umma_commit(smem_u32(&bar->kv_empty[st]));
        return true;
      };
      for (int c = c_begin; c < c_end && ok && !*abort_flag; ++c, ++qi) {
        const AttnItem it = a.items[c];
        const ItemGeo ig = item_geo(it, a.seq[it.s], g.gamma);
        const int qb = qi & 1;
        if (!mbar_wait(smem_u32(&bar->q_full[qb]), (qi >> 1) & 1, abort_flag)) break;
        const uint32_t qa = base + qb * Q_BYTES;
        for (int j = 0; j < ig.ntiles; ++j, ++T) {
          if (!mbar_wait(smem_u32(&bar->kv_full[stage]), kv_phase, abort_flag)) { ok = false; break; }
          const int sbuf = T & 1;
          if (!mbar_wait(smem_u32(&bar->s_empty[sbuf]), ((T >> 1) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + TMEM_S + sbuf * AK;
          const uint32_t kb = base + OFF_KV + stage * STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < AD / 16; ++kk) {
            const int h = kk >> 2, off = (kk & 3) * 32;
            umma_bf16(d, sw128_desc(qa + h * Q_HALF + off), sw128_desc(kb + h * KT_HALF + off),
                      idesc_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(smem_u32(&bar->s_full[sbuf]));
          if (j == ig.ntiles - 1) umma_commit(smem_u32(&bar->q_empty[qb]));
          if (have_prev && !issue_pv(prev_T, prev_stage, prev_gm, prev_qi, prev_first)) {
            ok = false;
            break;
          }
          have_prev = true;
          prev_T = T;
          prev_stage = stage;
          prev_gm = group_mask(ig, j);
          prev_qi = qi;
          prev_first = (j == 0);
          if (++stage == KV_STAGES) {
            stage = 0;
            kv_phase ^= 1;
          }
        }
      }
      if (ok && have_prev && !*abort_flag) issue_pv(prev_T, prev_stage, prev_gm, prev_qi, prev_first);
    }
  } else {
    // ------------------------------------------------ softmax -----------
    // Every wait here is taken with one answer per warp (the TMEM loads and
    // stores after it are warp-collective).
    // Scores in log2 units (x = s * scale * log2 e, p = 2^(x - m)). O
    // accumulates in TMEM over the item's tiles relative to the reference
    // max m; m moves (and O, l are rescaled) only when a tile's max exceeds
    // it by more than 2^8, so P stays <= 256 and most tiles touch no O.
    constexpr float TAU = 8.f;
    const float scale2 = a.scale * 1.4426950408889634f;
    const int q4 = warp & 3;                 // TMEM lane quarter this warp may access
    const int r = q4 * 32 + lane;            // query vector of this thread
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    int T = 0, qi = 0;
    bool ok = true;
    for (int c = c_begin; c < c_end && ok; ++c, ++qi) {
      const AttnItem it = a.items[c];
      const ItemGeo ig = item_geo(it, a.seq[it.s], g.gamma);
      const int ob = qi & 1;
      const uint32_t o_col = tmem + lane_off + TMEM_O + ob * AD;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < ig.ntiles; ++j, ++T) {
        const int sbuf = T & 1;
        if (!mbar_wait_warp(smem_u32(&bar->s_full[sbuf]), (T >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        float x[AK];
#pragma unroll
        for (int i = 0; i < AK / 16; ++i)
          tmem_ld16_nowait(tmem + lane_off + TMEM_S + sbuf * AK + 16 * i, x + 16 * i);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar->s_empty[sbuf]));
        const int kbase = ig.p0 + j * AK;
        float tmax = -INFINITY;
        if (kbase >= ig.lo && kbase + AK <= ig.hi) {
#pragma unroll
          for (int cc = 0; cc < AK; ++cc) {
            x[cc] *= scale2;
            tmax = fmaxf(tmax, x[cc]);
          }
        } else {
#pragma unroll
          for (int cc = 0; cc < AK; ++cc) {
            const int key = kbase + cc;
            x[cc] = (key >= ig.lo && key < ig.hi) ? x[cc] * scale2 : -INFINITY;
            tmax = fmaxf(tmax, x[cc]);
          }
        }
        if (tmax > m + TAU) {
          if (m != -INFINITY) {
            // O holds tiles < T: wait for PV(T-1), then rescale it in TMEM
            const int t1 = T - 1;
            if (!mbar_wait_warp(smem_u32(&bar->p_empty[t1 & 1]), (t1 >> 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float fac = ex2f(m - tmax);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              float v[64];
#pragma unroll
              for (int i = 0; i < 4; ++i) tmem_ld16_nowait(o_col + hh * 64 + 16 * i, v + 16 * i);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 64; ++e) v[e] *= fac;
#pragma unroll
              for (int i = 0; i < 4; ++i) tmem_st16(o_col + hh * 64 + 16 * i, v + 16 * i);
            }
            tmem_wait_st();
            l *= fac;
          }
          m = tmax;
        }
        const float mm = (m == -INFINITY) ? 0.f : m;
        // P buffer of this tile was last read by PV(T-2)
        if (T >= 2 && !mbar_wait_warp(smem_u32(&bar->p_empty[sbuf]), ((T - 2) >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        float s0 = 0.f, s1 = 0.f;
        // P row (bf16) in the 128B-swizzled K-major layout: 16-byte chunk ch
        // of row r sits at chunk position ch ^ (r % 8)
        const uint32_t prow = base + OFF_P + sbuf * P_BYTES + r * 128;
#pragma unroll
        for (int ch = 0; ch < AK / 8; ++ch) {
          float p[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) p[e] = ex2f(x[ch * 8 + e] - mm);
          s0 += (p[0] + p[1]) + (p[2] + p[3]);
          s1 += (p[4] + p[5]) + (p[6] + p[7]);
          const uint32_t w0 = pack_bf16(p[0], p[1]), w1 = pack_bf16(p[2], p[3]);
          const uint32_t w2 = pack_bf16(p[4], p[5]), w3 = pack_bf16(p[6], p[7]);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                           prow + ((uint32_t)(ch ^ (r & 7)) << 4)),
                       "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                       : "memory");
        }
        l += s0 + s1;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bar->p_full[sbuf]));
      }
      if (!ok) break;
      // the item's last PV, then O out of TMEM
      const int tl = T - 1;
      if (!mbar_wait_warp(smem_u32(&bar->p_empty[tl & 1]), (tl >> 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float m_nat = m * 0.6931471805599453f;
      const bool write = r < n_q;
      const float inv = 1.f / l;
      bf16 *orow = a.o + ((int64_t)(it.s * g.gamma + r / grp) * g.nq + it.g * grp + r % grp) * AD;
      float *ws = a.ws + (int64_t)(it.slot < 0 ? 0 : it.slot) * a.slot_floats;
      // Partial rows leave through this warp's 8 KB slice of the two P
      // buffers (free once the item's last PV is done), 64 columns at a time:
      // a thread stages its row (16-byte chunk c at c ^ (row % 8)), then each
      // warp store covers two whole 256-byte row halves instead of 32
      // scattered 16-byte pieces.
      const uint32_t stg = base + OFF_P + (uint32_t)q4 * (32 * 256);
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        float v[64];
#pragma unroll
        for (int i = 0; i < 4; ++i) tmem_ld16_nowait(o_col + hh * 64 + 16 * i, v + 16 * i);
        tmem_wait_ld();
        if (it.slot < 0) {
          if (!write) continue;
#pragma unroll
          for (int e = 0; e < 64; e += 8) {
            uint4 w;
            w.x = pack_bf16(v[e] * inv, v[e + 1] * inv);
            w.y = pack_bf16(v[e + 2] * inv, v[e + 3] * inv);
            w.z = pack_bf16(v[e + 4] * inv, v[e + 5] * inv);
            w.w = pack_bf16(v[e + 6] * inv, v[e + 7] * inv);
            *reinterpret_cast<uint4 *>(orow + hh * 64 + e) = w;
          }
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c)
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(
                             stg + lane * 256 + ((uint32_t)(c ^ (lane & 7)) << 4)),
                         "f"(v[4 * c]), "f"(v[4 * c + 1]), "f"(v[4 * c + 2]), "f"(v[4 * c + 3])
                         : "memory");
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int i = lane + 32 * k, rr = i >> 4, c = i & 15;
            float4 x;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
                         : "r"(stg + rr * 256 + ((uint32_t)(c ^ (rr & 7)) << 4))
                         : "memory");
            const int row = q4 * 32 + rr;
            if (row < n_q)
              *reinterpret_cast<float4 *>(ws + (int64_t)row * AD + hh * 64 + 4 * c) = x;
          }
          __syncwarp();
        }
      }
      if (write && it.slot >= 0) {
        ws[(int64_t)n_q * AD + r] = m_nat;
        ws[(int64_t)n_q * AD + n_q + r] = l;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bar->o_free[ob]));
    }
  }

  // ---------------------------------------------------------- teardown ----
  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) {
      atomicOr(a.status, ST_TIMEOUT);
      // wait (bounded) for every load this CTA issued to land
      for (int b = 0; b < 2; ++b) {
        if (!((bar->q_issued >> b) & 1u)) continue;
        const uint64_t t0 = global_ns();
        while (!mbar_test(smem_u32(&bar->q_full[b]), (bar->q_parity >> b) & 1u) &&
               global_ns() - t0 < 100000000ull) {
        }
      }
      for (int s = 0; s < KV_STAGES; ++s) {
        if (!((bar->kv_issued >> s) & 1u)) continue;
        const uint64_t t0 = global_ns();
        while (!mbar_test(smem_u32(&bar->kv_full[s]), (bar->kv_parity >> s) & 1u) &&
               global_ns() - t0 < 100000000ull) {
        }
      }
    }
    if (threadIdx.x == 32) {
      umma_commit(smem_u32(&bar->drain));
      const uint64_t t0 = global_ns();
      while (!mbar_test(smem_u32(&bar->drain), 0) && global_ns() - t0 < 100000000ull) {
      }
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                 : "memory");
  }
}

}  // namespace

bool attention_tc_supported(const Geo &g) {
  return !g.kv_fp8 && g.d == AD && attn_query_rows(g) <= AQ && g.B == 16 &&
         (int64_t)g.pages * g.L * 2 * g.nkv * g.B < (1ll << 31);
}

bool attention_tc_maps(const Geo &g, int R_max, const void *q, const void *pool, const void *kb,
                       const void *vb, AttnMaps *m) {
  m->ok = false;
  if (!attention_tc_supported(g)) return true;
  const int grp = g.nq / g.nkv;
  const int64_t qdims[3] = {g.d, g.nq, R_max};
  const int64_t qstr[2] = {(int64_t)g.d * 2, (int64_t)g.nq * g.d * 2};
  const int qbox[3] = {64, grp, g.gamma};
  if (!tc::make_map_3d(&m->q, q, qdims, qstr, qbox)) return false;
  const int64_t pool_rows = (int64_t)g.pages * g.L * 2 * g.nkv * g.B;
  if (!tc::make_map_2d(&m->pool, pool, false, pool_rows, g.d, 16) ||
      !tc::make_map_2d(&m->kb, kb, false, R_max, g.kv, 16) ||
      !tc::make_map_2d(&m->vb, vb, false, R_max, g.kv, 16))
    return false;
  m->ok = true;
  return true;
}

cudaError_t attention_tc(const AttnArgs &a, const AttnMaps &m, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  launch_pdl(k_attn_tc, dim3(a.grid_tc), dim3(THREADS), SMEM, s, m.q, m.pool, m.kb, m.vb, a);
  return cudaGetLastError();
}

int attention_tc_tiles(const Geo &g, const SeqMeta &sm, const AttnItem &it) {
  const int n_ctx = sm.pos - sm.ws;
  if (it.k0 >= n_ctx) return (g.gamma + AK - 1) / AK;
  const int lo = sm.ws + it.k0, hi = sm.ws + it.k1;
  return (hi - (lo & ~15) + AK - 1) / AK;
}

}  // namespace dfl
