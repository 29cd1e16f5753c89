// The shared lm_head over the full vocab fused with the per-row reductions
// of the draft rows ([P1] fields lm_head_shared, lm_head_shared_fp8; [P3]
// propose argument grammar_bitmask, last_confidence): for every draft row and
// every 256-row vocab tile, the tile's max logit, its lowest argmax and
// sum exp(logit - max), with grammar-masked tokens excluded. No
// [rows, vocab] logits tensor is written.
//
// Orientation: the draft rows are the MMA's A operand (M = 128 rows, rows
// past the call's count are zero-filled by TMA) and 256 vocab rows are B
// (N = 256), so the accumulator row of TMEM lane i is draft row i: each
// epilogue thread reduces its own row over the tile's 256 columns with no
// cross-thread traffic. At one sequence the kernel is bound by the vocab
// stream (1.02 GB bf16), at many sequences by the tensor cores.
//
// CTAs form groups of n_rt (one CTA per 128-row tile of draft rows); a group
// walks a contiguous range of vocab tiles in step, so the group's CTAs stream
// the same weight tile at the same time and L2 serves all but the first
// (the weight matrix is read from HBM about once). In each CTA a TMA producer
// warp, a single-thread MMA issuer and four epilogue warps share a 4-stage
// ring and two TMEM accumulators. Every wait is bounded.
#include <cuda.h>

#include "gemm_tc.h"
#include "internal.h"
#include "tc_ptx.h"

namespace dfl {
namespace tc {

namespace {

constexpr int LM_M = 128;                   // draft rows per tile
constexpr int LM_N = 256;                   // vocab rows per tile
constexpr int LM_BK = 64;
constexpr int LM_A = LM_M * LM_BK * 2;      // 16 KB
constexpr int LM_B = LM_N * LM_BK * 2;      // 32 KB
constexpr int LM_STAGE = LM_A + LM_B;       // 48 KB
constexpr int LM_STAGES = 4;
constexpr int LM_THREADS = 192;

struct LmSmem {
  uint64_t full[LM_STAGES], empty[LM_STAGES], acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
  uint32_t drain_issued, drain_parity;
  int abort_flag;
  uint32_t mwords[LM_N / 32][LM_M];   // grammar-mask words of the current tile, per row
};
constexpr int LM_SMEM = 1024 + LM_STAGES * LM_STAGE + (int)sizeof(LmSmem);

// Folds 16 consecutive logits (masked ones already -inf) of one row into the
// row's running (max m, lowest argmax id, sum exp(x - m)). Branch-free apart
// from the rare max update; ties keep the lower vocab id since chunks arrive
// in increasing id order.
__device__ __forceinline__ void lm_merge16(const float (&x)[16], int v0, float &m, int &id,
                                           float &s) {
  float lm = x[0];
#pragma unroll
  for (int c = 1; c < 16; ++c) lm = fmaxf(lm, x[c]);
  int li = 15;
#pragma unroll
  for (int c = 14; c >= 0; --c) li = (x[c] == lm) ? c : li;
  if (lm > m) {
    s *= __expf(m - lm);    // 0 while m is still -inf
    m = lm;
    id = v0 + li;
  }
  const float mm = (m == -INFINITY) ? 0.f : m;
  float e0 = 0.f, e1 = 0.f, e2 = 0.f, e3 = 0.f;
#pragma unroll
  for (int c = 0; c < 16; c += 4) {
    e0 += __expf(x[c] - mm);
    e1 += __expf(x[c + 1] - mm);
    e2 += __expf(x[c + 2] - mm);
    e3 += __expf(x[c + 3] - mm);
  }
  s += (e0 + e1) + (e2 + e3);
}

__global__ void __launch_bounds__(LM_THREADS, 1)
    k_lmhead(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
             LmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  LmSmem *sm = (LmSmem *)(smem_raw + (base - raw) + LM_STAGES * LM_STAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb = p.k / LM_BK;
  const int n_rt = (p.m_act + LM_M - 1) / LM_M;
  const int n_vt = (p.n_w + LM_N - 1) / LM_N;
  // this CTA: row tile rt, vocab tiles [vt_begin, vt_end) of its group
  const int n_groups = gridDim.x / n_rt;
  const int rt = blockIdx.x % n_rt, grp = blockIdx.x / n_rt;
  const int vt_begin = (int)((int64_t)n_vt * grp / n_groups);
  const int vt_end = (int)((int64_t)n_vt * (grp + 1) / n_groups);
  // local tile index t walks the group's vocab tiles
  const int t_begin = vt_begin, t_end = vt_end;

  if (threadIdx.x == 0) {
    for (int s = 0; s < LM_STAGES; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 1);
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm->acc_full[b]), 1);
      mbar_init(smem_u32(&sm->acc_empty[b]), 4);
    }
    mbar_init(smem_u32(&sm->drain), 1);
    sm->abort_flag = 0;
    sm->drain_issued = 0;
    sm->drain_parity = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    pdl_trigger();
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_x) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_w) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sm->tmem_base)),
                 "r"(512u)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int *abort_flag = &sm->abort_flag;
  const int64_t n_it = (int64_t)(t_end - t_begin) * kb;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer ------
    if (lane == 0) {
      // weight tiles are read by the n_rt CTAs of the group: normal L2 priority
      const uint64_t pol_w = n_rt > 1 ? policy_evict_normal() : policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      uint32_t issued = 0, parity = 0;
      const int n_pre = (int)(n_it < LM_STAGES ? n_it : LM_STAGES);
      // weight tiles first: they do not depend on the previous kernel
      for (int j = 0; j < n_pre; ++j) {
        const int t = t_begin + j / kb, k = j % kb;
        const uint32_t fb = smem_u32(&sm->full[j]);
        mbar_expect_tx(fb, LM_STAGE);
        tma_load_2d(base + j * LM_STAGE + LM_A, &map_w, fb, k * LM_BK, t * LM_N, pol_w);
        issued |= 1u << j;
      }
      pdl_wait();
      for (int j = 0; j < n_pre; ++j) {
        const int k = j % kb;
        tma_load_2d(base + j * LM_STAGE, &map_x, smem_u32(&sm->full[j]), k * LM_BK, rt * LM_M,
                    pol_x);
      }
      int t = t_begin + n_pre / kb, k = n_pre % kb;
      int stage = n_pre % LM_STAGES;
      uint32_t phase = (n_pre == LM_STAGES) ? 1u : 0u;
      for (int64_t j = n_pre; j < n_it && !*abort_flag; ++j) {
        if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, abort_flag)) break;
        const uint32_t sa = base + stage * LM_STAGE;
        const uint32_t fb = smem_u32(&sm->full[stage]);
        mbar_expect_tx(fb, LM_STAGE);
        tma_load_2d(sa + LM_A, &map_w, fb, k * LM_BK, t * LM_N, pol_w);
        tma_load_2d(sa, &map_x, fb, k * LM_BK, rt * LM_M, pol_x);
        issued |= 1u << stage;
        parity = (parity & ~(1u << stage)) | (phase << stage);
        if (++k == kb) { k = 0; ++t; }
        if (++stage == LM_STAGES) { stage = 0; phase ^= 1; }
      }
      sm->drain_issued = issued;
      sm->drain_parity = parity;
    } else {
      pdl_wait();
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer --------
    pdl_wait();
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_mn<LM_M, LM_N>();
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int t = t_begin; t < t_end && !*abort_flag; ++t) {
        if (!mbar_wait(smem_u32(&sm->acc_empty[acc]), acc_phase ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * LM_N;
        bool ok = true;
        for (int k = 0; k < kb; ++k) {
          if (!mbar_wait(smem_u32(&sm->full[stage]), phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = base + stage * LM_STAGE;
#pragma unroll
          for (int kk = 0; kk < LM_BK / 16; ++kk)
            umma_bf16(d, sw128_desc(sa + kk * 32), sw128_desc(sa + LM_A + kk * 32), idesc,
                      (k > 0 || kk > 0) ? 1u : 0u);
          umma_commit(smem_u32(&sm->empty[stage]));
          if (++stage == LM_STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        umma_commit(smem_u32(&sm->acc_full[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
  } else {
    // ------------------------------------------------ epilogue ----------
    pdl_wait();
    const int q = warp & 3;
    const int row_local = q * 32 + lane;   // TMEM lane = draft row within the row tile
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = t_begin; t < t_end; ++t) {
      const int vt = t;
      const int a = rt * LM_M + row_local;
      const bool row_ok = a < p.m_act;
      // this row's grammar-mask words for the tile; each thread reads back
      // only its own row, so no barrier is needed
      if (p.bitmask) {
#pragma unroll
        for (int w = 0; w < LM_N / 32; ++w) {
          const int word = (vt * LM_N) / 32 + w;
          sm->mwords[w][row_local] =
              (row_ok && word < p.mask_words)
                  ? (uint32_t)p.bitmask[(int64_t)(a / p.nd) * p.mask_words + word]
                  : 0xffffffffu;
        }
      }
      // one decision per warp: the TMEM loads below are warp-collective
      if (!mbar_wait_warp(smem_u32(&sm->acc_full[acc]), acc_phase, abort_flag)) break;
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + acc * LM_N;
      float m = -INFINITY, s = 0.f;
      int id = INT32_MAX;
#pragma unroll 1
      for (int c0 = 0; c0 < LM_N; c0 += 32) {
        const uint32_t word = p.bitmask ? sm->mwords[c0 >> 5][row_local] : 0xffffffffu;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float x[16];
          tmem_ld16(tbase + c0 + 16 * h, x);
          const int v0 = vt * LM_N + c0 + 16 * h;
          const uint32_t bits = word >> (16 * h);
          if (p.wscale) {
            if (v0 + 16 <= p.n_w) {
              const float4 *w4 = reinterpret_cast<const float4 *>(p.wscale + v0);
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const float4 f = __ldg(w4 + c);
                x[4 * c] *= f.x;
                x[4 * c + 1] *= f.y;
                x[4 * c + 2] *= f.z;
                x[4 * c + 3] *= f.w;
              }
            } else {
#pragma unroll
              for (int c = 0; c < 16; ++c) x[c] *= (v0 + c < p.n_w) ? __ldg(p.wscale + v0 + c) : 0.f;
            }
          }
          if (p.gscale != 0.f) {
#pragma unroll
            for (int c = 0; c < 16; ++c) x[c] *= p.gscale;
          }
#pragma unroll
          for (int c = 0; c < 16; ++c)
            x[c] = (v0 + c < p.n_w && ((bits >> c) & 1u)) ? x[c] : -INFINITY;
          lm_merge16(x, v0, m, id, s);
        }
      }
      tc_fence_before();
      if (lane == 0) mbar_arrive(smem_u32(&sm->acc_empty[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
      if (row_ok) {
        LmPartial r;
        r.max = m;
        r.id = id;
        r.sum = s;
        r.pad = 0;
        p.out[(int64_t)a * n_vt + vt] = r;
      }
    }
  }

  // ---------------------------------------------------------- teardown ----
  __syncthreads();
  if (*abort_flag) {
    if (threadIdx.x == 0) {
      atomicOr(p.status, ST_TIMEOUT);
      for (int s = 0; s < LM_STAGES; ++s) {
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
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u)
                 : "memory");
  }
}

}  // namespace

cudaError_t lmhead(const CUtensorMap &map_x, const CUtensorMap &map_w, const LmArgs &p,
                   cudaStream_t s) {
  if (p.m_act <= 0) return cudaSuccess;
  if (p.k % LM_BK) return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e =
        cudaFuncSetAttribute(k_lmhead, cudaFuncAttributeMaxDynamicSharedMemorySize, LM_SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int n_rt = (p.m_act + LM_M - 1) / LM_M;
  const int n_vt = (p.n_w + LM_N - 1) / LM_N;
  int groups = num_sms() / n_rt;
  if (groups < 1) groups = 1;
  if (groups > n_vt) groups = n_vt;
  const int grid = groups * n_rt;
  return launch_pdl(k_lmhead, dim3(grid), dim3(LM_THREADS), LM_SMEM, s, map_x, map_w, p);
}

int lmhead_vocab_tiles(int vocab) { return (vocab + LM_N - 1) / LM_N; }

}  // namespace tc
}  // namespace dfl
