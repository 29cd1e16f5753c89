// Weight-only low-precision lm_head over the draft rows ([P1] fields
// lm_head_shared_fp8 and lm_head_nvfp4, [P1]/[P3] last_confidence and the
// grammar bitmask of propose): the vocab table streams from HBM as its codes
// and never exists in 16-bit form anywhere.
//
//   FP8:   logit[a, v] = s_v * sum_k z[a, k] * e4m3(c[v, k])
//   NVFP4: logit[a, v] = g * sum_k z[a, k] * e2m1(c[v, k]) * e4m3(s[v, k / 16])
//
// It serves proposes of at most 16 draft rows (batch 1), where the table's
// bytes bound the step; wider proposes are bound by tensor-core work and
// multiply by the table widened to bf16 once (see build_device_side).
//
// z (the final-normed draft rows) is not quantised: the weight is
// dequantised, the activations are not. The product runs on the tensor cores
// as kind::f16 with f16 operands: the vocab rows as A (M = 128 rows per tile)
// and the 16 draft rows as B (N = 16), read from an f16 copy of the rows
// (every bf16 value down to 2^-17 in magnitude is an f16 value, so that copy
// changes no product a logit of any weight here can feel).
//
// Why A comes from tensor memory: at the HBM rate an SM receives about 22
// code bytes per cycle; dequantising into shared memory would add a 16-bit
// write and the MMA's read (4 bytes per element) on top of the codes' TMA
// write and read, beyond shared memory's 128 bytes per cycle for FP4 and at
// its limit for FP8. So converter warps read each row's codes (TMA-staged,
// 128-byte swizzled, conflict-free), convert them in registers and store f16
// pairs straight into TMEM with tcgen05.st; the MMA reads A from TMEM and only
// the small B tile from shared memory.
//
// Granularity: every hand-off between the converters and the MMA issuer (a
// TMEM slot signalled full, its MMAs, a commit that frees the slot) costs the
// issuer a fixed few hundred cycles, measured, on top of about 64 cycles per
// N = 16 MMA. So a slot carries 256 K (128 TMEM columns, 16 MMAs per
// hand-off) and a code stage carries the same 256 K.
//
// Exactness of the dequantisation: every E4M3 value and every E2M1 x E4M3
// product (at most 5 significant bits, magnitudes 2^-10 .. 2688) is an f16
// value, which the hardware FP8 / FP4 -> f16 conversions and one f16
// multiply produce; the per-row scale (FP8) or global scale (NVFP4)
// multiplies the fp32 logit in the epilogue.
//
// Work: vocab tiles of 128 rows, one persistent CTA per SM walking tiles
// c, c + G, ...; each tile runs the whole reduction (K = hidden) into a
// double-buffered TMEM accumulator, and the epilogue writes the tile's
// per-row (max, lowest argmax, sum exp) partial, as the bf16 lm_head does.
// The draft rows stay resident in shared memory for the whole launch: loaded
// once, so no load of them ever queues behind the code stream.
//
// Warp roles (352 threads): warp 0 issues the code (and scale) TMA loads into
// their ring, which the converters release as soon as the codes are in
// registers; warp 10 loads the draft rows; warp 1 owns TMEM and issues MMAs;
// warps 2-5 run the epilogue; warps 6-9 convert (converting a slot takes less
// time than its 16 MMAs, so one warpgroup keeps the issuer fed). Every wait
// is bounded; on a timeout the CTA raises the status word, drains its own
// copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include <cstddef>

#include "gemm_epi.h"
#include "gemm_tc.h"
#include "internal.h"
#include "tc_ptx.h"

namespace dfl {
namespace tc {

namespace {

constexpr int LP_THREADS = 352;
constexpr int LP_KS = 256;              // K elements per code stage and per A slot
constexpr int LP_SUB = LP_KS / 64;      // 64-K sub-blocks (4 MMAs each) per slot
constexpr int LP_SLOT_COLS = LP_KS / 2; // f16 pairs: 128 TMEM columns per slot
constexpr int LP_TMEM_COLS = 512;
constexpr int LP_SMEM_MAX = 232448;     // dynamic shared memory per CTA
constexpr int LP_K_RES = 2048;          // widest reduction with resident draft rows

struct LpSmem {
  uint64_t cfull[8], cempty[8], zfull;
  uint64_t a_full[4], a_empty[4], acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t c_issued, c_parity, z_issued;
  int abort_flag;
  EpiScratch epi;
};

constexpr int LP_BN = 16;               // draft rows (the MMA's N)

template <int FMT>
struct LpCfg {
  // one stage = 256 K of 128 vocab rows: FP8 two 128-byte boxes per row,
  // NVFP4 one (two codes a byte) plus 16 block-scale bytes
  static constexpr int CODE_BYTES = FMT == LM_LOWP_FP8 ? 2 * 128 * 128 : 128 * 128;
  static constexpr int SCALE_BYTES = FMT == LM_LOWP_NVFP4 ? 128 * 16 : 0;
  static constexpr int CSTAGE = CODE_BYTES + SCALE_BYTES;
  static constexpr int Z_TILE = LP_BN * 128;                   // 16 rows x 64 f16
  static constexpr int Z_BYTES = (LP_K_RES / 64) * Z_TILE;     // the resident draft rows
  static constexpr int CFIT = (LP_SMEM_MAX - 1024 - (int)sizeof(LpSmem) - Z_BYTES) / CSTAGE;
  static constexpr int CSTAGES = CFIT > 8 ? 8 : CFIT;
  static constexpr int SMEM = 1024 + Z_BYTES + CSTAGES * CSTAGE + (int)sizeof(LpSmem);
  static_assert(CSTAGES >= 3, "three code stages at least");
  static_assert(SMEM <= LP_SMEM_MAX, "shared memory");
  static_assert(CSTAGE % 1024 == 0 && Z_TILE % 1024 == 0,
                "swizzled tiles stay 1024-byte aligned");
  // TMEM: the two accumulators (32 columns), then the A slots
  static constexpr int A_COL0 = 2 * LP_BN;
  static constexpr int A_SLOTS = (LP_TMEM_COLS - A_COL0) / LP_SLOT_COLS;   // 3
  static_assert(A_SLOTS >= 2 && A_SLOTS <= 4, "A slots");
};

__device__ __forceinline__ uint32_t halfraw2_bits(__half2_raw r) {
  return (uint32_t)r.x | ((uint32_t)r.y << 16);
}

// 16 E4M3 codes -> 8 f16 pairs of their exact values (the row scale comes
// later); element 2c in the low half.
__device__ __forceinline__ void fp8_chunk(const uint4 &v, uint32_t *out) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[2 * i] = halfraw2_bits(
        __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xFFFFu), __NV_E4M3));
    out[2 * i + 1] = halfraw2_bits(
        __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3));
  }
}

// 16 bytes = 32 E2M1 codes (element 2j in the low nibble) with the block
// scales of elements 0-15 (s0) and 16-31 (s1), f16 pairs -> 16 f16 pairs of
// e2m1 * scale (exact).
__device__ __forceinline__ void fp4_chunk(const uint4 &v, __half2 s0, __half2 s1, uint32_t *out) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 s = i < 2 ? s0 : s1;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const __half2_raw r =
          __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((w[i] >> (8 * b)) & 0xFFu), __NV_E2M1);
      const __half2 x = __hmul2(*reinterpret_cast<const __half2 *>(&r), s);
      out[4 * i + b] = *reinterpret_cast<const uint32_t *>(&x);
    }
  }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

template <int FMT>
__global__ void __launch_bounds__(LP_THREADS, 1)
    k_lm_lowp(const __grid_constant__ CUtensorMap map_c, const __grid_constant__ CUtensorMap map_s,
              const __grid_constant__ CUtensorMap map_z, GemmParams p) {
  using C = LpCfg<FMT>;
  constexpr int BN = LP_BN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;          // z tiles, then the code ring
  const uint32_t cbase = base + C::Z_BYTES;
  LpSmem *sm = (LpSmem *)(smem_raw + (base - raw) + C::Z_BYTES + C::CSTAGES * C::CSTAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int n_items = p.tiles_m;
  const int G = (int)gridDim.x;
  const int my_items = (int)blockIdx.x < n_items ? (n_items - (int)blockIdx.x + G - 1) / G : 0;
  const int n_st = p.k / LP_KS;
  const int64_t total = (int64_t)my_items * n_st;      // stages (= A slots filled) of this CTA
  // (vocab tile, stage) of the CTA's j-th stage
  auto item_of = [&](int64_t j, int *tm, int *s) {
    *tm = (int)blockIdx.x + (int)(j / n_st) * G;
    *s = (int)(j % n_st);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::CSTAGES; ++s) {
      mbar_init(smem_u32(&sm->cfull[s]), 1);
      mbar_init(smem_u32(&sm->cempty[s]), 4);   // the converter warps
    }
    mbar_init(smem_u32(&sm->zfull), 1);
    for (int s = 0; s < C::A_SLOTS; ++s) {
      mbar_init(smem_u32(&sm->a_full[s]), 4);   // the converter warps
      mbar_init(smem_u32(&sm->a_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm->acc_full[b]), 1);
      mbar_init(smem_u32(&sm->acc_empty[b]), 4);
    }
    mbar_init(smem_u32(&sm->drain), 1);
    sm->abort_flag = 0;
    sm->c_issued = sm->c_parity = sm->z_issued = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (threadIdx.x == 0) pdl_trigger();
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_c) : "memory");
    if (FMT == LM_LOWP_NVFP4) asm volatile("prefetch.tensormap [%0];" ::"l"(&map_s) : "memory");
  }
  if (warp == 10 && lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(&map_z) : "memory");
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sm->tmem_base)),
                 "r"((uint32_t)LP_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int *abort_flag = &sm->abort_flag;

  if (warp == 0) {
    // ------------------------------------------- code producer ----------
    // (the codes are weights: nothing the previous kernel writes)
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      uint32_t issued = 0, parity = 0;
      int stage = 0;
      uint32_t phase = 0;
      for (int64_t j = 0; j < total && !*abort_flag; ++j) {
        if (j >= C::CSTAGES &&
            !mbar_wait_idle(smem_u32(&sm->cempty[stage]), phase ^ 1, abort_flag, 64))
          break;
        int tm, s;
        item_of(j, &tm, &s);
        const uint32_t sb = cbase + stage * C::CSTAGE;
        const uint32_t fb = smem_u32(&sm->cfull[stage]);
        mbar_expect_tx(fb, C::CSTAGE);
        // (x counts 4-byte words of the byte tables: a 128-byte box is 32)
        if (FMT == LM_LOWP_FP8) {
          tma_load_2d(sb, &map_c, fb, s * 64, tm * 128, pol_w);
          tma_load_2d(sb + 128 * 128, &map_c, fb, s * 64 + 32, tm * 128, pol_w);
        } else {
          tma_load_2d(sb, &map_c, fb, s * 32, tm * 128, pol_w);
          tma_load_2d(sb + C::CODE_BYTES, &map_s, fb, s * 4, tm * 128, pol_w);
        }
        issued |= 1u << stage;
        parity = (parity & ~(1u << stage)) | (phase << stage);
        if (++stage == C::CSTAGES) { stage = 0; phase ^= 1; }
      }
      sm->c_issued = issued;
      sm->c_parity = parity;
    }
  } else if (warp == 10) {
    // ------------------------------------------- draft rows ---------------
    pdl_wait();
    if (lane == 0 && total > 0) {
      // every 64-K tile of the rows, once, behind one barrier
      const uint32_t fb = smem_u32(&sm->zfull);
      mbar_expect_tx(fb, (uint32_t)(p.k / 64) * C::Z_TILE);
      for (int t = 0; t < p.k / 64; ++t)
        tma_load_2d(base + t * C::Z_TILE, &map_z, fb, 64 * t, 0, policy_evict_last());
      sm->z_issued = 1;
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer --------
    pdl_wait();
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_mn<BM, BN>();
      int slot = 0, acc = 0;
      uint32_t a_phase = 0, acc_phase = 0;
      bool ok = my_items == 0 || mbar_wait(smem_u32(&sm->zfull), 0, abort_flag);   // the rows
      for (int i = 0; i < my_items && ok; ++i) {
        if (!mbar_wait_idle(smem_u32(&sm->acc_empty[acc]), acc_phase ^ 1, abort_flag, 64)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        for (int s = 0; s < n_st && ok; ++s) {
          if (!mbar_wait(smem_u32(&sm->a_full[slot]), a_phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = tmem + C::A_COL0 + slot * LP_SLOT_COLS;
          for (int u = 0; u < LP_SUB; ++u) {
            const int g = s * LP_SUB + u;   // 64-K sub-block of the item
            // the descriptor's start address counts 16-byte units: +2 per 16 K
            const uint64_t bd = sw128_desc(base + g * C::Z_TILE);
            const uint32_t au = a + u * 32;
            if (g == 0)
              umma_bf16_tmem_a(d, au, bd, idesc, 0u);
            else
              umma_bf16_tmem_a_acc(d, au, bd, idesc);
#pragma unroll
            for (int kk = 1; kk < 4; ++kk) umma_bf16_tmem_a_acc(d, au + kk * 8, bd + 2 * kk, idesc);
          }
          umma_commit(smem_u32(&sm->a_empty[slot]));
          if (++slot == C::A_SLOTS) { slot = 0; a_phase ^= 1; }
        }
        if (!ok) break;
        umma_commit(smem_u32(&sm->acc_full[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
  } else if (warp < 6) {
    // ------------------------------------------------ epilogue ----------
    pdl_wait();
    const int q = warp & 3;
    const int et = (int)threadIdx.x - 64;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int i = 0; i < my_items; ++i) {
      const int tm = (int)blockIdx.x + i * G;
      const int f = tm * BM + q * 32 + lane;
      if (!epi_all(mbar_wait_idle(smem_u32(&sm->acc_full[acc]), acc_phase, abort_flag, 256)))
        break;
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + acc * BN;
      for (int cb = 0; cb < BN; cb += 16) {
        float v[16];
        tmem_ld16(tbase + cb, v);
        if (p.epi == EPI_TC_STORE_F32) {
          // the logits themselves (debug taps): out[a, f], scaled as the partials are
          float sc = p.gscale != 0.f ? p.gscale : 1.f;
          if (p.wscale && f < p.n_w) sc *= p.wscale[f];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int a = cb + e;
            if (a < p.m_act && f < p.n_w)
              static_cast<float *>(p.out)[(int64_t)a * p.ldo + f] = v[e] * sc;
          }
        } else {
          finish16<EPI_TC_LMHEAD>(p, &sm->epi, v, f, tm, cb, q, lane, et);
        }
      }
      tc_fence_before();
      if (lane == 0) mbar_arrive(smem_u32(&sm->acc_empty[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  } else {
    // ------------------------------------------------ converters --------
    // One warpgroup fills the slot of every stage (stage j goes to A slot
    // j % A_SLOTS), 64 K per tcgen05.st, one signal per slot.
    const int q = warp & 3;
    const int r = q * 32 + lane;   // vocab row of the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    for (int64_t j = 0; j < total; ++j) {
      const int stage = (int)(j % C::CSTAGES);
      const uint32_t phase = (uint32_t)((j / C::CSTAGES) & 1);
      const int slot = (int)(j % C::A_SLOTS);
      const uint32_t a_phase = (uint32_t)((j / C::A_SLOTS) & 1);
      if (!mbar_wait_warp_idle(smem_u32(&sm->cfull[stage]), phase, abort_flag, 32)) break;
      const uint32_t sb = cbase + stage * C::CSTAGE;
      __half2 sc[16];
      if (FMT == LM_LOWP_NVFP4) {
        // the row's 16 block scales of this stage (exact in f16)
        const uint4 sv = lds128(sb + C::CODE_BYTES + r * 16);
        const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int b = 0; b < 16; ++b) {
          const __half_raw hr =
              __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)((sw[b >> 2] >> (8 * (b & 3))) & 0xFFu),
                                      __NV_E4M3);
          const __half h = *reinterpret_cast<const __half *>(&hr);
          sc[b] = __halves2half2(h, h);
        }
      }
      if (!mbar_wait_warp_idle(smem_u32(&sm->a_empty[slot]), a_phase ^ 1, abort_flag, 32)) break;
      tc_fence_after();
      const uint32_t ta = tmem + lane_base + C::A_COL0 + slot * LP_SLOT_COLS;
#pragma unroll
      for (int u = 0; u < LP_SUB; ++u) {
        uint32_t w[32];
        if (FMT == LM_LOWP_FP8) {
          // 64 codes: box u / 2 of the stage, its 16-byte chunks 4 (u & 1) ..
          // + 3 (128-byte swizzled: chunk c of row r sits at c ^ (r & 7))
          const uint32_t row = sb + (u >> 1) * 128 * 128 + r * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int ch = 4 * (u & 1) + c;
            fp8_chunk(lds128(row + (uint32_t)((ch ^ (r & 7)) * 16)), w + 8 * c);
          }
        } else {
          // 64 elements: 16-byte chunks 2u, 2u + 1 (32 elements, two scale blocks each)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int ch = 2 * u + c;
            fp4_chunk(lds128(sb + r * 128 + (uint32_t)((ch ^ (r & 7)) * 16)), sc[2 * ch],
                      sc[2 * ch + 1], w + 16 * c);
          }
        }
        if (u == LP_SUB - 1) {
          // the stage's codes are in registers now
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm->cempty[stage]));
        }
        tmem_st32(ta + u * 32, w);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm->a_full[slot]));
    }
    tmem_wait_st();
  }

  // ---------------------------------------------------------- teardown ----
  __syncthreads();
  if (*abort_flag) {
    // let this CTA's own copies land before its shared memory goes away
    if (threadIdx.x == 0) {
      atomicOr(p.status, ST_TIMEOUT);
      for (int s = 0; s <= C::CSTAGES; ++s) {
        const bool code = s < C::CSTAGES;
        if (!(code ? (sm->c_issued >> s) & 1u : sm->z_issued)) continue;
        const uint32_t par = code ? (sm->c_parity >> s) & 1u : 0u;
        const uint32_t bar = smem_u32(code ? &sm->cfull[s] : &sm->zfull);
        const uint64_t t0 = global_ns();
        while (!mbar_test(bar, par) && global_ns() - t0 < 100000000ull) {
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
                 "r"((uint32_t)LP_TMEM_COLS)
                 : "memory");
  }
}

template <int FMT>
cudaError_t launch_lp(const CUtensorMap &mc, const CUtensorMap &ms, const CUtensorMap &mz,
                      const GemmParams &p, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_lm_lowp<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         LpCfg<FMT>::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int grid = p.tiles_m < num_sms() ? p.tiles_m : num_sms();
  cudaError_t e = launch_pdl(k_lm_lowp<FMT>, dim3(grid), dim3(LP_THREADS), LpCfg<FMT>::SMEM, s,
                             mc, ms, mz, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool lm_lowp_fits(int m_act, int k) { return m_act <= LP_BN && k <= LP_K_RES && k % LP_KS == 0; }

cudaError_t lm_lowp(int fmt, const CUtensorMap &map_codes, const CUtensorMap &map_scales,
                    const CUtensorMap &map_z, const GemmParams &p, cudaStream_t s) {
  if (p.m_act <= 0) return cudaSuccess;
  if (!lm_lowp_fits(p.m_act, p.k)) return cudaErrorInvalidValue;
  if (fmt == LM_LOWP_FP8) return launch_lp<LM_LOWP_FP8>(map_codes, map_scales, map_z, p, s);
  if (fmt == LM_LOWP_NVFP4) return launch_lp<LM_LOWP_NVFP4>(map_codes, map_scales, map_z, p, s);
  return cudaErrorInvalidValue;
}

}  // namespace tc
}  // namespace dfl
