// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05 + TMEM),
// operands staged by TMA, for every dense contraction of the draft head:
// fc, the fused ctx K/V projection, the per-layer QKV / o / gate-up / down
// projections and the shared lm_head ([P1] fields fc, fused_kv_weight,
// layers, lm_head_shared).
//
//   Y[a, f] = sum_k X[a, k] * W[f, k]      (X activations, W a linear weight)
//
// The weight is the MMA's A operand (128 weight rows per tile, M = 128) and
// the activations are B (BN rows, N = BN), so a batch-1 step of 16 block rows
// still runs full-width MMAs while every weight byte is read once ("swap AB").
// Both operands are K-major, 64-element (128-byte) K slices in the 128-byte
// swizzled layout TMA writes.
//
// One persistent CTA per SM walks a contiguous range of the (tile, k-block)
// iteration space (stream-K), so every SM streams the same number of weight
// bytes whatever the tile count. A tile whose k-range is split between CTAs is
// finished by its last arriving contributor, which sums the contributors'
// partials in a fixed order (deterministic) and runs the epilogue; nothing
// spins on another CTA.
//
// Warp roles (192 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues MMAs from one thread, warps 2-5 (one per TMEM lane quarter) drain the
// double-buffered accumulator and run the epilogue. Every mbarrier wait is
// bounded; on timeout the CTA raises the status word, stops issuing work,
// waits (bounded) for its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <cstdio>
#include <mutex>

#include "internal.h"
#include "gemm_tc.h"
#include "tc_ptx.h"
#include "gemm_epi.h"

namespace dfl {
namespace tc {

constexpr int NUM_THREADS = 192;
// K elements per pipeline stage (iteration): two 64-element TMA boxes per
// operand and 8 MMAs behind one commit. Every commit hand-off costs the MMA
// issuer a fixed few hundred cycles (measured), which at one commit per 4
// MMAs held the tensor pipe to about half its rate at N = 256 and left the
// batch-1 weight stream little slack. A K that is not a multiple of 128 reads
// an all-zero second box at its end (the copy's out-of-bounds fill).
constexpr int KS = 2 * BK;

template <int BN, int EPI>
struct Cfg {
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int HALF_BYTES = A_BYTES + B_BYTES;   // one 64-K box of each operand
  static constexpr int STAGE_BYTES = 2 * HALF_BYTES;
  // Up to 64 rows: 4 stages (8 x 16 KB of weight tiles in flight per SM,
  // which the batch-1 weight stream needs). Partial mode reserves no
  // exchange buffer.
  static constexpr bool kPartial = (EPI == EPI_TC_PARTIAL);
  static constexpr int STAGES = (BN <= 64) ? 4 : (BN <= 128 ? 3 : 2);
  static_assert(STAGES <= 8, "the barrier arrays in Smem hold 8 stages");
  static constexpr int TMEM_COLS = (2 * BN < 32) ? 32 : 2 * BN;
  static constexpr int EXTRA = kPartial ? 1536 : 10240;   // Smem (without / with xch)
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + EXTRA;
};

// -------------------------------------------------------- stream-K map --
struct Part {
  int64_t total;  // tiles * kb
  int G;          // CTAs
  __device__ __forceinline__ int64_t begin(int c) const { return total * c / G; }
  // The CTA whose range holds iteration i.
  __device__ int owner(int64_t i) const {
    int c = (int)((i * G) / total);
    while (c + 1 < G && begin(c + 1) <= i) ++c;
    while (c > 0 && begin(c) > i) --c;
    return c;
  }
};

// ----------------------------------------------------------- epilogues --
struct Smem {
  uint64_t full[8], empty[8], acc_full[2], acc_empty[2], drain, never;
  uint32_t tmem_base;
  uint32_t drain_issued, drain_parity;
  int abort_flag;
  int is_last;
  EpiScratch epi;   // its exchange buffer comes last (fused epilogues only)
};
// Partial mode reserves shared memory only up to the exchange buffer, which it never touches.
static_assert(offsetof(Smem, epi) + offsetof(EpiScratch, xch) <= 1536,
              "Smem head must fit the partial-mode reservation");

// ---------------------------------------------------------------- kernel --
template <int BN, int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
              GemmParams p) {
  using C = Cfg<BN, EPI>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *gbase = smem_raw + (base - raw);
  Smem *sm = (Smem *)(gbase + C::STAGES * C::STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int kb = (p.k + KS - 1) / KS;   // iterations (K steps) per tile
  const int tiles = p.tiles_m * p.tiles_n;
  const Part part{(int64_t)tiles * kb, (int)gridDim.x};
  // Iteration range of this CTA. Stream-K: a contiguous range of (tile,
  // k-block) iterations, tile = it / kb. Data-parallel: whole tiles
  // blockIdx.x, blockIdx.x + G, ...; iteration it is k-block it % kb of the
  // CTA's (it / kb)-th tile.
  const bool dp = p.dp != 0;
  const int n_dp = dp ? (tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  const int64_t it_begin = dp ? 0 : part.begin(blockIdx.x);
  const int64_t it_end = dp ? (int64_t)n_dp * kb : part.begin(blockIdx.x + 1);
  const int t_step = dp ? (int)gridDim.x : 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 1);
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm->acc_full[b]), 1);
      mbar_init(smem_u32(&sm->acc_empty[b]), 4);
    }
    mbar_init(smem_u32(&sm->drain), 1);
    mbar_init(smem_u32(&sm->never), 1);   // nothing ever arrives (test hook)
    sm->abort_flag = 0;
    sm->drain_issued = 0;
    sm->drain_parity = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (threadIdx.x == 0) pdl_trigger();
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_w) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&map_x) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sm->tmem_base)),
                 "r"((uint32_t)C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int *abort_flag = &sm->abort_flag;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer ------
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
      uint32_t issued = 0, parity = 0;   // per stage: loads issued, phase they complete
      const int64_t n_it = it_end - it_begin;
      // Weights do not depend on the previous kernel: fill the first stages
      // with weight tiles before waiting for it, then add the activations.
      const int n_pre = (int)(n_it < C::STAGES ? n_it : C::STAGES);
      // (tile, k-block) of it_begin
      int t0 = dp ? (int)blockIdx.x : (int)(it_begin / kb), k0 = (int)(it_begin % kb);
      {
        int t = t0, k = k0;
        for (int j = 0; j < n_pre; ++j) {
          const uint32_t fb = smem_u32(&sm->full[j]);
          mbar_expect_tx(fb, C::STAGE_BYTES);
#pragma unroll
          for (int h = 0; h < 2; ++h)
            tma_load_2d(base + j * C::STAGE_BYTES + h * C::HALF_BYTES, &map_w, fb,
                        k * KS + h * BK, (t % p.tiles_m) * BM, pol_w);
          issued |= 1u << j;
          if (++k == kb) { k = 0; t += t_step; }
        }
      }
      pdl_wait();
      int t = t0, k = k0;
      for (int j = 0; j < n_pre; ++j) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tma_load_2d(base + j * C::STAGE_BYTES + h * C::HALF_BYTES + A_BYTES, &map_x,
                      smem_u32(&sm->full[j]), k * KS + h * BK, (t / p.tiles_m) * BN, pol_x);
        if (++k == kb) { k = 0; t += t_step; }
      }
      int stage = n_pre % C::STAGES;
      uint32_t phase = (n_pre == C::STAGES) ? 1u : 0u;
      for (int64_t j = n_pre; j < n_it && !*abort_flag; ++j) {
        if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, abort_flag)) break;
        const uint32_t sa = base + stage * C::STAGE_BYTES;
        const uint32_t fb = smem_u32(&sm->full[stage]);
        mbar_expect_tx(fb, C::STAGE_BYTES);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          tma_load_2d(sa + h * C::HALF_BYTES, &map_w, fb, k * KS + h * BK, (t % p.tiles_m) * BM,
                      pol_w);
          tma_load_2d(sa + h * C::HALF_BYTES + A_BYTES, &map_x, fb, k * KS + h * BK,
                      (t / p.tiles_m) * BN, pol_x);
        }
        issued |= 1u << stage;
        parity = (parity & ~(1u << stage)) | (phase << stage);
        if (++k == kb) { k = 0; t += t_step; }
        if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
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
      const uint32_t idesc = idesc_bf16_mn<BM, BN>();
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int64_t it = it_begin; it < it_end && !*abort_flag;) {
        const int k0 = (int)(it % kb);
        const int k1 = (int)((int64_t)kb < (int64_t)k0 + (it_end - it) ? (int64_t)kb : (int64_t)k0 + (it_end - it));
        if (!mbar_wait(smem_u32(&sm->acc_empty[acc]), acc_phase ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        bool ok = true;
        for (int k = k0; k < k1; ++k) {
          if (!mbar_wait(smem_u32(&sm->full[stage]), phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = base + stage * C::STAGE_BYTES;
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = sw128_desc(sa + h * C::HALF_BYTES + kk * 32);
              const uint64_t bd = sw128_desc(sa + h * C::HALF_BYTES + A_BYTES + kk * 32);
              umma_bf16(d, ad, bd, idesc, (k > k0 || h > 0 || kk > 0) ? 1u : 0u);
            }
          umma_commit(smem_u32(&sm->empty[stage]));
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        umma_commit(smem_u32(&sm->acc_full[acc]));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
        it += k1 - k0;
      }
    }
  } else {
    // ------------------------------------------------ epilogue ----------
    pdl_wait();
    const int q = warp & 3;                  // TMEM lane quarter of this warp
    const int f_local = q * 32 + lane;       // weight row within the tile
    int acc = 0;
    uint32_t acc_phase = 0;
    // test hook: one epilogue thread waits on a barrier nothing arrives on
    // until the limit runs out, which aborts the CTA mid-stream
    bool live = true;
    if (p.fault_ns > 0 && threadIdx.x == 64)
      live = fault_wait(smem_u32(&sm->never), (uint64_t)p.fault_ns, abort_flag);
    live = epi_all(live);
    for (int64_t it = it_begin; live && it < it_end;) {
      const int t = dp ? (int)blockIdx.x + (int)(it / kb) * (int)gridDim.x : (int)(it / kb);
      const int k0 = (int)(it % kb);
      const int k1 = (int)((int64_t)kb < (int64_t)k0 + (it_end - it) ? (int64_t)kb : (int64_t)k0 + (it_end - it));
      const int tm = t % p.tiles_m, tn = t / p.tiles_m;
      const int f = tm * BM + f_local;
      const bool whole = (k0 == 0 && k1 == kb);
      // all 128 epilogue threads take the same decision (named barriers and
      // warp-collective TMEM loads follow)
      if (!epi_all(mbar_wait(smem_u32(&sm->acc_full[acc]), acc_phase, abort_flag))) break;
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + acc * BN;
      // partial slot of this CTA for this tile: its first or its last segment
      const int slot = 2 * blockIdx.x + (it == it_begin ? 0 : 1);
      float *ws = p.ws + (int64_t)slot * BN * BM;
      // up to 64 accumulator columns per TMEM round trip
      constexpr int CH = BN < 64 ? BN : 64;
      for (int cb = 0; cb < BN; cb += CH) {
        float vv[CH / 16][16];
#pragma unroll
        for (int i = 0; i < CH / 16; ++i) tmem_ld16_nowait(tbase + cb + 16 * i, vv[i]);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < CH / 16; ++i) {
          const int c0 = cb + 16 * i;
          const float(&v)[16] = vv[i];
          if (EPI == EPI_TC_PARTIAL) {
            // [BN rows][128 features]: coalesced for this store and for the
            // consumer, which reads along features
#pragma unroll
            for (int c = 0; c < 16; ++c) ws[(int64_t)(c0 + c) * BM + f_local] = v[c];
          } else if (whole) {
            finish16<EPI>(p, &sm->epi, v, f, tm, tn * BN + c0, q, lane, (int)threadIdx.x - 64);
          } else {
            // thread-major partial: this thread's BN columns are contiguous
            float4 *dst = reinterpret_cast<float4 *>(ws + (int64_t)f_local * BN + c0);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              dst[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
          }
        }
      }
      tc_fence_before();
      if (lane == 0) mbar_arrive(smem_u32(&sm->acc_empty[acc]));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
      if (!whole && EPI != EPI_TC_PARTIAL) {
        // stream-K fixup: the last contributor of the tile sums the partials
        __threadfence();
        epi_bar();
        const int c_lo = part.owner((int64_t)t * kb);
        const int c_hi = part.owner((int64_t)t * kb + kb - 1);
        if (threadIdx.x == 64) {
          const int old = atomicAdd(&p.counters[t], 1);
          sm->is_last = (old == c_hi - c_lo);
        }
        epi_bar();
        if (sm->is_last) {
          __threadfence();
          for (int c0 = 0; c0 < BN; c0 += 16) {
            float v[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = 0.f;
            // contributors in ascending order, four partial reads in flight
            for (int cc0 = c_lo; cc0 <= c_hi; cc0 += 4) {
              float4 r[4][4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int cc = cc0 + u;
                if (cc <= c_hi) {
                  const int sl =
                      2 * cc + ((cc == c_lo && part.begin(cc) < (int64_t)t * kb) ? 1 : 0);
                  const float4 *src = reinterpret_cast<const float4 *>(
                      p.ws + (int64_t)sl * BN * BM + (int64_t)f_local * BN + c0);
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
            finish16<EPI>(p, &sm->epi, v, f, tm, tn * BN + c0, q, lane, (int)threadIdx.x - 64);
          }
          if (threadIdx.x == 64) p.counters[t] = 0;
        }
        epi_bar();
      }
      it += k1 - k0;
    }
  }

  // ---------------------------------------------------------- teardown ----
  __syncthreads();
  if (*abort_flag) {
    // Let this CTA's own copies and MMAs land before its shared memory and
    // TMEM go away; each wait is bounded (100 ms).
    if (threadIdx.x == 0) {
      atomicOr(p.status, ST_TIMEOUT);
      for (int s = 0; s < C::STAGES; ++s) {
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
                 "r"((uint32_t)C::TMEM_COLS)
                 : "memory");
  }
}

// ============================================================ host side ==
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
int g_num_sms = 0;

void init_driver() {
  cudaDriverEntryPointQueryResult q;
  void *fn = nullptr;
  if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &fn, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
}

template <int BN, int EPI>
cudaError_t set_smem_attr() {
  static bool done = false;
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(k_gemm_tc<BN, EPI>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg<BN, EPI>::SMEM);
  if (e == cudaSuccess) done = true;
  return e;
}

template <int BN, int EPI>
cudaError_t launch_bn(const CUtensorMap &mw, const CUtensorMap &mx, const GemmParams &p, int grid,
                      cudaStream_t s) {
  cudaError_t e = set_smem_attr<BN, EPI>();
  if (e != cudaSuccess) return e;
  e = launch_pdl(k_gemm_tc<BN, EPI>, dim3(grid), dim3(NUM_THREADS), Cfg<BN, EPI>::SMEM, s, mw, mx, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int EPI>
cudaError_t launch_epi(int bn, const CUtensorMap &mw, const CUtensorMap &mx, const GemmParams &p,
                       int grid, cudaStream_t s) {
  switch (bn) {
    case 16: return launch_bn<16, EPI>(mw, mx, p, grid, s);
    case 32: return launch_bn<32, EPI>(mw, mx, p, grid, s);
    case 64: return launch_bn<64, EPI>(mw, mx, p, grid, s);
    case 128: return launch_bn<128, EPI>(mw, mx, p, grid, s);
    case 256: return launch_bn<256, EPI>(mw, mx, p, grid, s);
  }
  return cudaErrorInvalidValue;
}
}  // namespace

int num_sms() {
  std::call_once(g_once, init_driver);
  return g_num_sms;
}

bool make_map_2d(CUtensorMap *map, const void *base, bool fp8, int64_t rows, int64_t cols,
                 int box_rows) {
  std::call_once(g_once, init_driver);
  if (!g_encode) return false;
  const int esz = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * esz)};
  cuuint32_t box[2] = {(cuuint32_t)(128 / esz), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        2, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_map_u8(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int box_bytes,
                 int box_rows, bool swizzle128) {
  std::call_once(g_once, init_driver);
  if (!g_encode || cols % 4 || box_bytes % 4) return false;
  // moved as 4-byte elements (the same bytes and layout; the copy engine
  // walks a box by elements, so wider elements move a byte table faster)
  cuuint64_t dims[2] = {(cuuint64_t)(cols / 4), (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols};
  cuuint32_t box[2] = {(cuuint32_t)(box_bytes / 4), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_map_3d(CUtensorMap *map, const void *base, const int64_t dims[3],
                 const int64_t strides_bytes[2], const int box[3]) {
  std::call_once(g_once, init_driver);
  if (!g_encode) return false;
  cuuint64_t d[3] = {(cuuint64_t)dims[0], (cuuint64_t)dims[1], (cuuint64_t)dims[2]};
  cuuint64_t st[2] = {(cuuint64_t)strides_bytes[0], (cuuint64_t)strides_bytes[1]};
  cuuint32_t bx[3] = {(cuuint32_t)box[0], (cuuint32_t)box[1], (cuuint32_t)box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), d, st,
                        bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int pick_bn(int m_act) {
  if (m_act <= 16) return 16;
  if (m_act <= 32) return 32;
  if (m_act <= 64) return 64;
  if (m_act <= 128) return 128;
  return 256;
}

bool partial_ok(int m_act, int n_w, int k) {
  const int bn = pick_bn(m_act);
  const int ks = (k + KS - 1) / KS;
  const int64_t total = (int64_t)((n_w + BM - 1) / BM) * ((m_act + bn - 1) / bn) * ks;
  int grid = num_sms();
  if (total < grid) grid = (int)total;
  return grid > 0 && (total + grid - 1) / grid <= ks && total * grid < (1ll << 31);
}

int pick_bn_dp(int m_act, int n_w, int k) {
  // Data-parallel tile width: the smallest modelled time of the tensor work
  // (waves of whole tiles; an M 128 x N bn x K 16 MMA issues in bn / 2
  // cycles at ~1.9 GHz) and of the operand stream out of L2 (~20 TB/s).
  const int G = num_sms();
  const int kb = k / BK;
  const int cap = pick_bn(m_act);
  int best = cap;
  double best_t = 1e30;
  for (int bn = cap; bn >= 64; bn /= 2) {
    const int64_t tiles = (int64_t)((n_w + BM - 1) / BM) * ((m_act + bn - 1) / bn);
    const int64_t waves = (tiles + G - 1) / G;
    const double t_mma = (double)waves * kb * (BK / 16) * (bn / 2) / 1.9e9;
    const double t_l2 = (double)tiles * kb * (A_BYTES + bn * BK * 2) / 20e12;
    const double t = t_mma > t_l2 ? t_mma : t_l2;
    if (t < best_t) {
      best_t = t;
      best = bn;
    }
  }
  return best;
}

cudaError_t gemm(const CUtensorMap &map_w, const CUtensorMap &map_x, int bn, GemmParams p,
                 cudaStream_t s, Partials *view) {
  if (p.m_act <= 0 || p.n_w <= 0) return cudaSuccess;
  if (p.k % BK) return cudaErrorInvalidValue;
  p.tiles_m = (p.n_w + BM - 1) / BM;
  p.tiles_n = (p.m_act + bn - 1) / bn;
  const int ks = (p.k + KS - 1) / KS;
  const int64_t total = (int64_t)p.tiles_m * p.tiles_n * ks;
  int grid = num_sms();
  if (p.grid_cap > 0 && p.grid_cap < grid) grid = p.grid_cap;
  if (p.dp) {
    // whole tiles per CTA: fused epilogues only, no fixup
    if (p.epi == EPI_TC_PARTIAL || p.epi == EPI_TC_LMHEAD) return cudaErrorInvalidValue;
    const int tiles = p.tiles_m * p.tiles_n;
    if (tiles < grid) grid = tiles;
  }
  if (total < grid) grid = (int)total;
  if (grid < 1) grid = 1;
  if (p.epi == EPI_TC_PARTIAL) {
    if ((total + grid - 1) / grid > ks || !view) return cudaErrorInvalidValue;
    view->ws = p.ws;
    view->dense = nullptr;
    view->ld = 0;
    view->tiles_m = p.tiles_m;
    view->kb = ks;
    view->G = grid;
    view->bn = bn;
    view->total = (int)total;
  }
  switch (p.epi) {
    case EPI_TC_STORE_F32: return launch_epi<EPI_TC_STORE_F32>(bn, map_w, map_x, p, grid, s);
    case EPI_TC_ADD_F32: return launch_epi<EPI_TC_ADD_F32>(bn, map_w, map_x, p, grid, s);
    case EPI_TC_STORE_BF16: return launch_epi<EPI_TC_STORE_BF16>(bn, map_w, map_x, p, grid, s);
    case EPI_TC_LMHEAD: return launch_epi<EPI_TC_LMHEAD>(bn, map_w, map_x, p, grid, s);
    case EPI_TC_QKV: return launch_epi<EPI_TC_QKV>(bn, map_w, map_x, p, grid, s);
    case EPI_TC_SWIGLU: return launch_epi<EPI_TC_SWIGLU>(bn, map_w, map_x, p, grid, s);
    case EPI_TC_PARTIAL: return launch_epi<EPI_TC_PARTIAL>(bn, map_w, map_x, p, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tc

// ------------------------------------------------------- lm_head merge --
// Merges the (max, lowest argmax, sum exp) partials of one draft row over all
// vocab tiles: draft id (or -1 when no token is allowed) and the top-1
// softmax probability 1 / sum_v exp(l_v - max).
__device__ __forceinline__ void lm_merge(float &m, int &id, float &s, float m2, int id2,
                                         float s2) {
  const float M = fmaxf(m, m2);
  const int I = (m > m2 || (m == m2 && id < id2)) ? id : id2;
  const float a = (m == -INFINITY) ? 0.f : s * __expf(m - M);
  const float b = (m2 == -INFINITY) ? 0.f : s2 * __expf(m2 - M);
  m = M;
  id = I;
  s = a + b;
}

__global__ void k_lm_reduce(const LmPartial *__restrict__ part, int tiles,
                            int32_t *__restrict__ row_id, float *__restrict__ row_p1) {
  __shared__ float sm_m[32], sm_s[32];
  __shared__ int sm_i[32];
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const LmPartial *pr = part + (int64_t)r * tiles;
  float m = -INFINITY, s = 0.f;
  int id = INT32_MAX;
  for (int t = threadIdx.x; t < tiles; t += blockDim.x) {
    const LmPartial q = pr[t];
    lm_merge(m, id, s, q.max, q.id, q.sum);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, id, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lm_merge(m, id, s, m2, i2, s2);
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { sm_m[w] = m; sm_i[w] = id; sm_s[w] = s; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) lm_merge(m, id, s, sm_m[i], sm_i[i], sm_s[i]);
    const bool none = (m == -INFINITY);
    row_id[r] = none ? -1 : id;
    row_p1[r] = none ? 0.f : 1.f / s;
  }
}

cudaError_t lm_reduce(const LmPartial *part, int rows, int tiles, int32_t *row_id, float *row_p1,
                      cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(k_lm_reduce, dim3(rows), dim3(256), 0, s, part, tiles, row_id, row_p1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dfl
