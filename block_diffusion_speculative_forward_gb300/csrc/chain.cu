// Few-row proposes (one sequence, or a handful of short blocks) as a few
// persistent launches: each launch walks several weight-streaming GEMMs of
// the layer stack back to back ("phases"), so the weight stream of the next
// projection starts while the current one finishes, and the norms, the q/k
// RoPE, SwiGLU, the residual updates and the lm_head reductions run inside
// the GEMMs instead of as separate kernels ([P1] fields fc, hidden_norm,
// fused_kv_weight, kv_cache, layers, norm, lm_head_shared).
//
// A batch-1 propose of the shipped geometry is
//   prologue (block embed, pack of the new ctx rows)
//   chain [fc, fused K/V + paged write, QKV of layer 0]
//   for each layer l: attention(l); chain [o(l), gate/up(l), down(l), QKV(l+1) or lm_head]
// where every GEMM is "swap AB" (128 weight rows are the MMA's M, the 16
// block rows its N) and is split over all SMs by stream-K, as in gemm_tc.cu.
//
// Warp roles of a CTA (224 threads):
//   warp 0     issues the weight TMA loads of every phase into an 8-stage ring;
//              weights depend on nothing, so it runs ahead across phases
//   warp 1     owns TMEM and issues the MMAs (one thread)
//   warp 2     provides the B operand of each stage by a TMA load of a bf16
//              activation: one written by an earlier kernel, or by an earlier
//              phase (after the producing tile's ready flag), or a normed
//              input RMSNorm(x), which CTA j writes for k-block j (from the f32
//              residual and its per-tile sums of squares) before raising that
//              k-block's ready flag
//   warps 3-6  drain the accumulators and run the phase's epilogue; a tile cut
//              between CTAs is finished by its last arriving contributor,
//              which sums the partials in CTA order
// Phases depend only on earlier phases. A phase's dependency is a count of
// finished tiles (or one tile's flag) in global memory, polled with
// acquire loads; every wait here is bounded (2 s), after which the CTA raises
// the status word and takes the same abort path as gemm_tc.cu. All CTAs are
// resident at once (one per SM), so waiting on another CTA is safe.
#include <cuda.h>

#include <cstddef>

#include "chain.h"
#include "gemm_epi.h"
#include "tc_ptx.h"
#include "chain_attn.cuh"

namespace dfl {
namespace tc {

namespace {

constexpr int CH_THREADS = 224;
constexpr int CH_STAGES = 8;
constexpr int CH_B_BYTES = CHAIN_BN * BK * 2;                 // 2 KB: bf16 B operand
constexpr int CH_STAGE_BYTES = A_BYTES + CH_B_BYTES;          // 18 KB (1024-aligned)
constexpr int CH_EPI_T0 = 96;
constexpr uint32_t CH_TMEM_COLS = 32;

struct ChainSmem {
  uint64_t full[CH_STAGES], empty[CH_STAGES], acc_full[2], acc_empty[2], drain, never;
  uint64_t kvb[8];   // attention: two K/V buffers per epilogue warp
  uint32_t tmem_base;
  uint32_t drain_issued, drain_parity;
  int abort_flag;
  int is_last;
  EpiScratch epi;
};
constexpr int CH_ATTN_OFF = CH_STAGES * CH_STAGE_BYTES;   // the attention area (1024-aligned)
constexpr int CH_SMEM = 1024 + CH_ATTN_OFF + CA_BYTES + (int)sizeof(ChainSmem);
static_assert(CH_SMEM <= 232448, "chain CTA exceeds the 227 KB shared-memory limit");
static_assert(CH_STAGE_BYTES % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
static_assert(sizeof(ChainArgs) <= 32000, "chain parameters exceed the launch limit");

// Stream-K split of one phase's (tile, k-block) iterations over the first
// G = min(CTAs, iterations) CTAs, so that every participating CTA holds at
// least one iteration (a tile's contributors are then exactly the CTAs
// owner(first) .. owner(last)); later CTAs hold none of this phase.
struct Split {
  int64_t total;
  int G;
  __device__ __forceinline__ Split(int64_t total_, int ctas)
      : total(total_), G(total_ < ctas ? (int)total_ : ctas) {}
  __device__ __forceinline__ int64_t begin(int c) const {
    return c >= G ? total : total * c / G;
  }
  // The CTA whose range holds iteration i.
  __device__ __forceinline__ int owner(int64_t i) const {
    int c = (int)((i * G) / total);
    while (c + 1 < G && begin(c + 1) <= i) ++c;
    while (c > 0 && begin(c) > i) --c;
    return c;
  }
};

__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Every lane of the warp polls until *ctr >= target (one answer per warp).
// False when the CTA aborts or the wait runs past the limit (then it aborts).
__device__ bool wait_count_warp(const int *ctr, int target, volatile int *abort_flag) {
  bool ok = true;
  if (ld_acquire(ctr) < target) {
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
      if (ld_acquire(ctr) >= target) break;
      if ((i & 15) == 0) {
        if (*abort_flag) { ok = false; break; }
        if (global_ns() - t0 > TIMEOUT_NS) {
          *abort_flag = 1;
          ok = false;
          break;
        }
      }
    }
  }
  return __all_sync(0xffffffffu, ok) != 0;
}

// ------------------------------------------------------- phase epilogues --
// Residual / ctx-row outputs: out[a, f] (+)= y, the residual tap, and the
// per-tile sums of squares of the updated rows (the next RMSNorm's input).
__device__ __forceinline__ void finish_rows(const ChainPhase &P, EpiScratch *sm,
                                            const float (&v)[16], int f, int tm, int q, int lane,
                                            int et) {
  const bool add = P.kind != CK_FC;
  const bool f_ok = f < P.n_w;
  // every load first (one round trip), then the stores
  float old[16], sq[16];
#pragma unroll
  for (int c = 0; c < 16; ++c)
    old[c] = (add && f_ok && c < P.rows) ? __ldcg(P.out + (int64_t)c * P.n_w + f) : 0.f;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    float y = 0.f;
    if (f_ok && c < P.rows) {
      y = old[c] + v[c];
      P.out[(int64_t)c * P.n_w + f] = y;
      if (P.x_tap) P.x_tap[(int64_t)c * P.n_w + f] = y;
    }
    sq[c] = y * y;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int c = 0; c < 16; ++c) sq[c] += __shfl_xor_sync(0xffffffffu, sq[c], o);
  if (lane == 0) {
#pragma unroll
    for (int c = 0; c < 16; ++c) sm->red_v[q][c] = sq[c];
  }
  epi_bar();
  if (et < 16)
    P.out_ss[tm * 16 + et] = sm->red_v[0][et] + sm->red_v[1][et] + sm->red_v[2][et] + sm->red_v[3][et];
  epi_bar();
}

// Fused ctx K/V rows ([P1] fields fused_kv_weight, kv_cache, yarn_inv_freq):
// W_kv row f is element i of head h of layer l's K (or V). A 128-row tile
// holds whole heads of one kind. K: per-head RMSNorm (k_norm of layer l),
// then RoPE at the row's position; V as it is; both written to the row's
// (page, slot) of the pool, bf16 or E4M3 with the head's scale.
__device__ __forceinline__ void finish_kv(const ChainPhase &P, EpiScratch *sm, const float (&v)[16],
                                          int f, int q, int lane, int *status) {
  const Geo &g = P.geo;
  const int d = g.d, half = d / 2;
  const int fl = q * 32 + lane;
  const int l = f / (2 * g.kv), within = f % (2 * g.kv);
  const int kind = within / g.kv, h = (within % g.kv) / d, i = within % d;
  const int nrows = P.rows < 16 ? P.rows : 16;
  float y[16];
  if (kind == 0) {
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
  }
  epi_bar();
  if (kind == 0) {
    const float gi = __bfloat162float(P.k_norm[l][i]);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      float tot;
      if (d == 128) tot = sm->red_v[0][c] + sm->red_v[1][c] + sm->red_v[2][c] + sm->red_v[3][c];
      else tot = sm->red_v[q & 2][c] + sm->red_v[(q & 2) + 1][c];
      sm->xch[c][fl] = gi * (v[c] * rsqrtf(tot / (float)d + g.eps));
    }
  }
  epi_bar();
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    if (kind == 0) {
      const int pos = c < nrows ? P.ctx_rows[c].pos : 0;
      const float cs = P.ep.cos_t[(int64_t)pos * half + (i % half)];
      const float sn = P.ep.sin_t[(int64_t)pos * half + (i % half)];
      const float a = sm->xch[c][fl], b = sm->xch[c][fl ^ half];
      y[c] = (i < half) ? (a * cs - b * sn) : (a * cs + b * sn);
    } else {
      y[c] = v[c];
    }
  }
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    if (c >= nrows) break;
    const RowMeta rm = P.ctx_rows[c];
    if (rm.seq < 0) continue;   // padding row: computed, never stored
    if (rm.page < 0 || rm.page >= g.pages) {
      if (i == 0) atomicOr(status, ST_PAGE);
      continue;
    }
    const int64_t off = kv_offset(g, rm.page, l, kind, h, rm.slot) + i;
    if (g.kv_fp8) {
      const float s = P.kv_scale[(l * g.nkv + h) * 2 + kind];
      ((uint8_t *)P.pool)[off] = (uint8_t)__nv_cvt_float_to_fp8(y[c] / s, __NV_SATFINITE, __NV_E4M3);
    } else {
      ((bf16 *)P.pool)[off] = __float2bfloat16_rn(y[c]);
    }
  }
  epi_bar();
}

// ---------------------------------------------------------------- kernel --
__global__ void __launch_bounds__(CH_THREADS, 1)
    k_chain(const __grid_constant__ ChainArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  ChainSmem *sm = (ChainSmem *)(gbase + CH_ATTN_OFF + CA_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = (int)gridDim.x, cta = (int)blockIdx.x;
  const int np = a.n_phases;

  if (threadIdx.x == 0) {
    for (int s = 0; s < CH_STAGES; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 2);   // the weight copy's arrival + the B operand's
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm->acc_full[b]), 1);
      mbar_init(smem_u32(&sm->acc_empty[b]), 4);
    }
    mbar_init(smem_u32(&sm->drain), 1);
    mbar_init(smem_u32(&sm->never), 1);   // nothing ever arrives (test hook)
    for (int b = 0; b < 8; ++b) mbar_init(smem_u32(&sm->kvb[b]), 1);
    sm->abort_flag = 0;
    sm->drain_issued = 0;
    sm->drain_parity = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    pdl_trigger();
  }
  if (warp == 0) {
    for (int p = lane; p < np; p += 32)
      if (a.ph[p].kind != CK_ATTN) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(a.maps + a.ph[p].map_w) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(a.maps + a.ph[p].map_b) : "memory");
      }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sm->tmem_base)),
                 "r"(CH_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int *abort_flag = &sm->abort_flag;

  if (warp == 0) {
    // ------------------------------------------- weight producer ------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0, issued = 0, parity = 0;
      bool ok = true;
      for (int p = 0; p < np && ok; ++p) {
        const ChainPhase &P = a.ph[p];
        const Split sp((int64_t)P.tiles_m * P.kb, G);
        const int64_t e = sp.begin(cta + 1);
        if (sp.begin(cta) >= e) continue;   // no weights here (attention, or a short phase)
        int t = (int)(sp.begin(cta) / P.kb), k = (int)(sp.begin(cta) % P.kb);
        for (int64_t it = sp.begin(cta); it < e; ++it) {
          if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, abort_flag)) { ok = false; break; }
          const uint32_t fb = smem_u32(&sm->full[stage]);
          mbar_expect_tx(fb, A_BYTES);
          tma_load_2d(base + stage * CH_STAGE_BYTES, a.maps + P.map_w, fb, k * BK, t * BM, pol);
          if (++k == P.kb) { k = 0; ++t; }
          issued |= 1u << stage;
          parity = (parity & ~(1u << stage)) | (phase << stage);
          if (++stage == CH_STAGES) { stage = 0; phase ^= 1; }
        }
      }
      sm->drain_issued = issued;
      sm->drain_parity = parity;
    }
    pdl_wait();
  } else if (warp == 1) {
    // ------------------------------------------- MMA issuer -----------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_mn<BM, CHAIN_BN>();
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int p = 0; p < np && ok; ++p) {
        const ChainPhase &P = a.ph[p];
        const Split sp((int64_t)P.tiles_m * P.kb, G);
        const int64_t b = sp.begin(cta), e = sp.begin(cta + 1);
        for (int64_t it = b; it < e && ok;) {
          const int k0 = (int)(it % P.kb);
          const int k1 = (int)((int64_t)P.kb < k0 + (e - it) ? (int64_t)P.kb : k0 + (e - it));
          if (!mbar_wait(smem_u32(&sm->acc_empty[acc]), acc_phase ^ 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + acc * CHAIN_BN;
          for (int k = k0; k < k1; ++k) {
            if (!mbar_wait(smem_u32(&sm->full[stage]), phase, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = base + stage * CH_STAGE_BYTES;
            const uint32_t sb = sa + A_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              umma_bf16(d, sw128_desc(sa + kk * 32), sw128_desc(sb + kk * 32), idesc,
                        (k > k0 || kk > 0) ? 1u : 0u);
            umma_commit(smem_u32(&sm->empty[stage]));
            if (++stage == CH_STAGES) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          umma_commit(smem_u32(&sm->acc_full[acc]));
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
          it += k1 - k0;
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------- B operand ------------
    pdl_wait();
    const uint64_t pol_b = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int p = 0; p < np && ok; ++p) {
      const ChainPhase &P = a.ph[p];
      const Split sp((int64_t)P.tiles_m * P.kb, G);
      const int64_t b = sp.begin(cta), e = sp.begin(cta + 1);
      const bool need_dep = P.dep >= 0 && !P.dep_tile;
      if (P.b_norm && cta < P.kb) {
        // this CTA's share of the normed operand: k-block cta of
        // h = bf16(gain * x * rinv(row)), written once to the phase's bf16
        // buffer, then its ready flag
        if (need_dep && !wait_count_warp(a.ph[P.dep].done, a.ph[P.dep].tiles_m, abort_flag)) {
          ok = false;
          break;
        }
        float rinv = 0.f;   // lane r < 16: 1 / sqrt(mean square of row r + eps)
        if (lane < 16 && lane < P.rows) {
          // the row's per-tile sums (at most 16 tiles), all loads in flight at once
          const int nt = P.k / 128;
          float sv[CHAIN_MAX_K_NORM / 128];
#pragma unroll
          for (int j = 0; j < CHAIN_MAX_K_NORM / 128; ++j) sv[j] = j < nt ? __ldcg(P.nss + j * 16 + lane) : 0.f;
          float t = 0.f;
#pragma unroll
          for (int j = 0; j < CHAIN_MAX_K_NORM / 128; ++j) t += sv[j];
          rinv = rsqrtf(t / (float)P.k + P.ep.eps);
        }
        // lane: row r, 32 consecutive features (half hh of the k-block)
        const int r = lane & 15, hh = lane >> 4;
        const float rr = __shfl_sync(0xffffffffu, rinv, r);
        const int f0 = cta * BK + hh * 32;
        uint32_t w[16];
        if (r < P.rows) {
          const float4 *xs = reinterpret_cast<const float4 *>(P.nsrc + (int64_t)r * P.k + f0);
          const uint4 *gs = reinterpret_cast<const uint4 *>(P.ngain + f0);
          float4 xv[8];
          uint4 gw[4];
#pragma unroll
          for (int u = 0; u < 8; ++u) xv[u] = __ldcg(xs + u);
#pragma unroll
          for (int u = 0; u < 4; ++u) gw[u] = __ldg(gs + u);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const bf16 *gv = reinterpret_cast<const bf16 *>(&gw[u]);
            const float x8[8] = {xv[2 * u].x, xv[2 * u].y, xv[2 * u].z, xv[2 * u].w,
                                 xv[2 * u + 1].x, xv[2 * u + 1].y, xv[2 * u + 1].z, xv[2 * u + 1].w};
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              __nv_bfloat162 h2 = __floats2bfloat162_rn(
                  __bfloat162float(gv[2 * e2]) * (x8[2 * e2] * rr),
                  __bfloat162float(gv[2 * e2 + 1]) * (x8[2 * e2 + 1] * rr));
              w[4 * u + e2] = *reinterpret_cast<uint32_t *>(&h2);
            }
          }
        } else {
#pragma unroll
          for (int u = 0; u < 16; ++u) w[u] = 0u;   // rows past the call's rows: zero
        }
        uint4 *dst = reinterpret_cast<uint4 *>(P.hbuf + (int64_t)r * P.k + f0);
#pragma unroll
        for (int u = 0; u < 4; ++u) dst[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        if (P.kind == CK_LM && r < P.rows) {
          // the lm_head's normed rows for the debug taps
          if (P.z_tap) {
            uint4 *zt = reinterpret_cast<uint4 *>(P.z_tap + (int64_t)r * P.k + f0);
#pragma unroll
            for (int u = 0; u < 4; ++u) zt[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
          }
          const int j = r % P.ep.lm_gamma - P.ep.lm_first;
          if (P.z_rows && j >= 0 && j < P.ep.nd) {
            uint4 *zr = reinterpret_cast<uint4 *>(P.z_rows +
                                                  (int64_t)((r / P.ep.lm_gamma) * P.ep.nd + j) * P.k + f0);
#pragma unroll
            for (int u = 0; u < 4; ++u) zr[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
          }
        }
        // publish: the warp's stores are ordered before lane 0's release by
        // the warp barrier (release is cumulative); consumers acquire, then
        // fence the async proxy before their TMA reads
        __syncwarp();
        if (lane == 0) {
          asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(P.hflag + cta), "r"(1) : "memory");
          asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(P.hdone), "r"(1) : "memory");
        }
      }
      if (b == e) continue;
      if (need_dep && !P.b_norm &&
          !wait_count_warp(a.ph[P.dep].done, a.ph[P.dep].tiles_m, abort_flag)) {
        ok = false;
        break;
      }
      // B = a bf16 activation, TMA per stage. A normed operand's k-block k
      // waits for its ready flag; with a tile dependency, k-block k waits for
      // tile k of phase dep; either until every k-block or tile is ready.
      const ChainPhase *D = (P.dep >= 0 && P.dep_tile) ? &a.ph[P.dep] : nullptr;
      const int *rflag = P.b_norm ? P.hflag : D ? D->flag : nullptr;
      const int *rdone = P.b_norm ? P.hdone : D ? D->done : nullptr;
      const int rall = P.b_norm ? P.kb : D ? D->tiles_m : 0;
      const int rdiv = P.b_norm ? 1 : P.dep_div, rneed = P.b_norm ? 1 : P.dep_need;
      bool all_ready = rflag == nullptr;
      int k = (int)(b % P.kb);
      for (int64_t it = b; it < e; ++it) {
        if (!mbar_wait_warp(smem_u32(&sm->empty[stage]), phase ^ 1, abort_flag)) { ok = false; break; }
        bool acquired = false;
        if (!all_ready) {
          acquired = true;
          if (ld_acquire(rdone) >= rall) all_ready = true;
          else if (!wait_count_warp(rflag + k / rdiv, rneed, abort_flag)) { ok = false; break; }
        }
        if (lane == 0) {
          // what the acquire made visible to the generic proxy, for the TMA
          if (acquired) asm volatile("fence.proxy.async.global;" ::: "memory");
          const uint32_t fb = smem_u32(&sm->full[stage]);
          mbar_expect_tx(fb, CH_B_BYTES);
          tma_load_2d(base + stage * CH_STAGE_BYTES + A_BYTES, a.maps + P.map_b, fb, k * BK, 0, pol_b);
        }
        if (++k == P.kb) k = 0;
        if (++stage == CH_STAGES) { stage = 0; phase ^= 1; }
      }
    }
  } else {
    // ------------------------------------------- epilogue -------------
    pdl_wait();
    const int et = (int)threadIdx.x - CH_EPI_T0;
    const int q = warp & 3;                  // TMEM lane quarter of this warp
    const int f_local = q * 32 + lane;       // weight row within the tile
    int acc = 0;
    uint32_t acc_phase = 0;
    bool live = true;
    if (a.fault_ns > 0 && et == 0)
      live = fault_wait(smem_u32(&sm->never), (uint64_t)a.fault_ns, abort_flag);
    live = epi_all(live);
    uint32_t kv_par = 0;   // per warp and buffer: parity of the next K/V arrival
    for (int p = 0; p < np && live; ++p) {
      const ChainPhase &P = a.ph[p];
      if (P.kind == CK_ATTN) {
        // block attention: items cta, cta + G, ... of the call, once the QKV
        // phase (and the fused ctx K/V phase of this launch, if any) is done
        bool ok = true;
        if (warp == 3) {
          if (P.dep >= 0) ok = wait_count_warp(a.ph[P.dep].done, a.ph[P.dep].tiles_m, abort_flag);
          if (ok && P.dep2 >= 0) ok = wait_count_warp(a.ph[P.dep2].done, a.ph[P.dep2].tiles_m, abort_flag);
        }
        live = epi_all(ok);
        const int n_items = live ? *a.attn.count : 0;
        uint8_t *abase = gbase + CH_ATTN_OFF;
        const uint32_t abase_s = base + CH_ATTN_OFF;
        const uint32_t kvb0 = smem_u32(&sm->kvb[0]);
        for (int i = cta; i < n_items && live; i += G) {
          const ChainAttnItem it = a.attn.items[i];
          live = a.attn.geo.d == 128
                     ? ca_item<128>(a.attn, a.maps + a.map_pool, P.attn_layer, P, it, abase, abase_s, kvb0, kv_par, &sm->epi,
                                    &sm->is_last, abort_flag, a.status, et, q, lane)
                     : ca_item<64>(a.attn, a.maps + a.map_pool, P.attn_layer, P, it, abase, abase_s, kvb0, kv_par, &sm->epi,
                                   &sm->is_last, abort_flag, a.status, et, q, lane);
          live = epi_all(live);
        }
        continue;
      }
      const Split sp((int64_t)P.tiles_m * P.kb, G);
      const int64_t b = sp.begin(cta), e = sp.begin(cta + 1);
      bool res_seen = P.res_dep < 0;
      for (int64_t it = b; it < e;) {
        const int t = (int)(it / P.kb);
        const int k0 = (int)(it % P.kb);
        const int k1 = (int)((int64_t)P.kb < k0 + (e - it) ? (int64_t)P.kb : k0 + (e - it));
        const bool whole = (k0 == 0 && k1 == P.kb);
        const int f = t * BM + f_local;
        if (!epi_all(mbar_wait(smem_u32(&sm->acc_full[acc]), acc_phase, abort_flag))) {
          live = false;
          break;
        }
        tc_fence_after();
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + acc * CHAIN_BN, v);
        tc_fence_before();
        if (lane == 0) mbar_arrive(smem_u32(&sm->acc_empty[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
        bool finisher = whole;
        if (!whole) {
          // this CTA's partial of the tile, thread-major (16 contiguous floats)
          const int slot = 2 * (P.slot_set * G + cta) + (it == b ? 0 : 1);
          float4 *dst = reinterpret_cast<float4 *>(a.ws + ((int64_t)slot * BM + f_local) * CHAIN_BN);
#pragma unroll
          for (int c = 0; c < 4; ++c) dst[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
          // arrival: the partial stores of all 128 threads are ordered before
          // one thread's acquire-release add by the barrier; the last
          // contributor's add acquires every earlier contributor's partials,
          // and the barrier after it carries that to the other threads
          epi_bar();
          const int c_lo = sp.owner((int64_t)t * P.kb);
          const int c_hi = sp.owner((int64_t)t * P.kb + P.kb - 1);
          if (et == 0) {
            int old;
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(P.arrive + t) : "memory");
            sm->is_last = (old == c_hi - c_lo);
          }
          epi_bar();
          finisher = sm->is_last != 0;
          if (finisher) {
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = 0.f;
            // contributors in ascending order, four partials in flight
            for (int c0 = c_lo; c0 <= c_hi; c0 += 4) {
              float4 r[4][4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int cc = c0 + u;
                if (cc <= c_hi) {
                  const int sl = 2 * (P.slot_set * G + cc) +
                                 ((cc == c_lo && sp.begin(cc) < (int64_t)t * P.kb) ? 1 : 0);
                  const float4 *src = reinterpret_cast<const float4 *>(
                      a.ws + ((int64_t)sl * BM + f_local) * CHAIN_BN);
#pragma unroll
                  for (int c = 0; c < 4; ++c) r[u][c] = __ldcg(src + c);
                } else {
#pragma unroll
                  for (int c = 0; c < 4; ++c) r[u][c] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
              }
#pragma unroll
              for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                  v[4 * c] += r[u][c].x;
                  v[4 * c + 1] += r[u][c].y;
                  v[4 * c + 2] += r[u][c].z;
                  v[4 * c + 3] += r[u][c].w;
                }
            }
          }
        }
        if (finisher && !res_seen) {
          // the residual rows this epilogue adds to were written by another
          // phase's epilogues: take their count with acquire semantics
          bool ok = true;
          if (warp == 3) ok = wait_count_warp(a.ph[P.res_dep].done, a.ph[P.res_dep].tiles_m, abort_flag);
          if (!epi_all(ok)) {
            live = false;
            break;
          }
          res_seen = true;
        }
        if (finisher) {
          switch (P.kind) {
            case CK_FC:
            case CK_O:
            case CK_DOWN: finish_rows(P, &sm->epi, v, f, t, q, lane, et); break;
            case CK_KV: finish_kv(P, &sm->epi, v, f, q, lane, a.status); break;
            case CK_QKV: finish16<EPI_TC_QKV>(P.ep, &sm->epi, v, f, t, 0, q, lane, et); break;
            case CK_GU: finish16<EPI_TC_SWIGLU>(P.ep, &sm->epi, v, f, t, 0, q, lane, et); break;
            default: finish16<EPI_TC_LMHEAD>(P.ep, &sm->epi, v, f, t, 0, q, lane, et); break;
          }
          // publish: every thread's stores (ordered by the barrier), then
          // the tile's flag and count with release semantics
          epi_bar();
          if (et == 0) {
            asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(P.flag + t), "r"(1) : "memory");
            asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(P.done), "r"(1) : "memory");
          }
        }
        if (!whole) epi_bar();   // is_last is reused by the next split tile
        it += k1 - k0;
      }
    }
  }

  // ---------------------------------------------------------- teardown ----
  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) {
      atomicOr(a.status, ST_TIMEOUT);
      // let this CTA's own copies land (bounded: a stage whose B arrival is
      // missing never completes, and its weight copy has long landed)
      for (int s = 0; s < CH_STAGES; ++s) {
        if (!((sm->drain_issued >> s) & 1u)) continue;
        const uint32_t par = (sm->drain_parity >> s) & 1u;
        const uint64_t t0 = global_ns();
        while (!mbar_test(smem_u32(&sm->full[s]), par) && global_ns() - t0 < 100000000ull) {
        }
      }
    }
    if (threadIdx.x == 32) {
      umma_commit(smem_u32(&sm->drain));
      const uint64_t t0 = global_ns();
      while (!mbar_test(smem_u32(&sm->drain), 0) && global_ns() - t0 < 100000000ull) {
      }
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(CH_TMEM_COLS)
                 : "memory");
  }
}

// -------------------------------------------------------------- prologue --
// Block embed ([P1] fields gamma, mask_token_id, embed_tokens_shared) with
// the per-tile sums of squares of each row (the first RMSNorm's input), and
// the pack of the new ctx rows from the callers' stacks (zero for padding).
__global__ void k_chain_prologue(const bf16 *__restrict__ E, const SeqMeta *__restrict__ seq,
                                 int R, int gamma, int H, int V, uint32_t mask_token,
                                 float *__restrict__ x, float *__restrict__ ss, float *x_tap,
                                 const RowMeta *__restrict__ rows, int S, bf16 *__restrict__ pack,
                                 int *status) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  if (b >= R) {
    const RowMeta rm = rows[b - R];
    uint4 *dst = reinterpret_cast<uint4 *>(pack + (int64_t)(b - R) * S);
    const uint4 *src = reinterpret_cast<const uint4 *>(rm.src);
    for (int e = threadIdx.x; e < S / 8; e += blockDim.x)
      dst[e] = (rm.seq < 0 || !src) ? make_uint4(0u, 0u, 0u, 0u) : src[e];
    return;
  }
  const int i = b % gamma;
  uint32_t tok = i == 0 ? (uint32_t)seq[b / gamma].token : mask_token;
  if (tok >= (uint32_t)V) {
    if (threadIdx.x == 0) atomicOr(status, ST_TOKEN);
    tok = 0;
  }
  // thread t: features 8t .. 8t+7; 16 threads per 128-feature tile
  const int f0 = 8 * threadIdx.x;
  float s = 0.f;
  if (f0 < H) {
    const uint4 raw = *reinterpret_cast<const uint4 *>(E + (int64_t)tok * H + f0);
    const bf16 *e = reinterpret_cast<const bf16 *>(&raw);
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = __bfloat162float(e[j]);
      s += v[j] * v[j];
    }
    float4 *xo = reinterpret_cast<float4 *>(x + (int64_t)b * H + f0);
    xo[0] = make_float4(v[0], v[1], v[2], v[3]);
    xo[1] = make_float4(v[4], v[5], v[6], v[7]);
    if (x_tap) {
      float4 *to = reinterpret_cast<float4 *>(x_tap + (int64_t)b * H + f0);
      to[0] = xo[0];
      to[1] = xo[1];
    }
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (f0 < H && (threadIdx.x & 15) == 0) ss[(threadIdx.x >> 4) * 16 + b] = s;
}

}  // namespace

int chain_smem() { return CH_SMEM; }

cudaError_t chain(const ChainArgs &a, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_chain, cudaFuncAttributeMaxDynamicSharedMemorySize, CH_SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaError_t e = launch_pdl(k_chain, dim3(num_sms()), dim3(CH_THREADS), CH_SMEM, s, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace tc

cudaError_t chain_prologue(const bf16 *E, const SeqMeta *seq, int R, const Geo &g,
                           uint32_t mask_token, float *x, float *ss, float *x_tap,
                           const RowMeta *rows, int m, bf16 *pack, int *status, cudaStream_t s) {
  if (g.H > 8 * 256 || g.H % 128) return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(tc::k_chain_prologue, dim3(R + m), dim3(256), 0, s, E, seq, R,
                             g.gamma, g.H, g.V, mask_token, x, ss, x_tap, rows, g.S, pack, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dfl
