// dflash_gemm_noalloc: the tensor-core GEMM with its scratch in a fixed,
// file-scope device array instead of memory obtained from cudaMalloc.
//
// Why it exists: some callers may not allocate device memory once they are
// running. A serving engine that reserves the whole GPU up front (weights,
// KV cache, activations carved from one arena) cannot have a library call
// cudaMalloc behind its back: the allocation can fail when the arena owns
// everything, and cudaMalloc/cudaFree synchronise the whole device, which
// stalls every other stream of a latency-critical decode loop. This entry
// point lets such a caller run the GEMM with nothing but the inputs and the
// output it passes in.
//
// The scratch (the stream-K partial tiles, the per-tile arrival counters and
// a status word) lives in `g_noalloc_scratch` below. Every GPU that loads the
// library holds that array until the process exits. All calls share it, so
// two calls that run at the same time on the GPU (different streams, or
// different host threads) race on it; callers must order such calls.
#include <cuda_runtime.h>

#include <mutex>

#include "dflash.h"
#include "gemm_tc.h"
#include "internal.h"

namespace {

// Limits of the fixed scratch: at most 16 activation rows (the 16-row tile),
// at most kMaxCtas persistent CTAs, at most kMaxTiles 128-row weight tiles.
constexpr int kMaxRows = 16;
constexpr int kMaxCtas = 160;
constexpr int kMaxTiles = 4096;
constexpr size_t kWsFloats = (size_t)2 * kMaxCtas * kMaxRows * 128;   // 2.5 MiB
constexpr size_t kScratchBytes = kWsFloats * sizeof(float) + (kMaxTiles + 64) * sizeof(int);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};   // device address of g_noalloc_scratch per device

// Looks up (once per device, with that device current) the device address of
// the scratch array; the host-side symbol itself is not a device pointer.
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" DFLASH_API int dflash_gemm_noalloc(const void *w, const void *x, float *y, int32_t m,
                                               int32_t n_w, int32_t k, void *stream) {
  if (!w || !x || !y || m <= 0 || n_w <= 0 || k <= 0 || k % 64) return DFLASH_EINVAL;
  if (m > kMaxRows || (n_w + 127) / 128 > kMaxTiles) return DFLASH_EINVAL;
  if (((uintptr_t)w | (uintptr_t)x) & 15) return DFLASH_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  void *base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return DFLASH_ECUDA;
  float *ws = (float *)base;
  int *status = (int *)((unsigned char *)base + kWsFloats * sizeof(float));
  int *counters = status + 64;
  const int bn = dfl::tc::pick_bn(m);   // 16 for every m this entry accepts
  CUtensorMap mw, mx;
  if (!dfl::tc::make_map_2d(&mw, w, false, n_w, k, 128) ||
      !dfl::tc::make_map_2d(&mx, x, false, m, k, bn))
    return DFLASH_ECUDA;
  const int tiles = (n_w + 127) / 128;
  // The status word and the counters must start at zero; the array keeps
  // whatever the previous call left.
  if (cudaMemsetAsync(status, 0, sizeof(int) * ((size_t)tiles + 64), s) != cudaSuccess)
    return DFLASH_ECUDA;
  dfl::GemmParams p{};
  p.m_act = m;
  p.n_w = n_w;
  p.k = k;
  p.epi = dfl::EPI_TC_STORE_F32;
  p.out = y;
  p.ldo = n_w;
  p.grid_cap = kMaxCtas;
  p.ws = ws;
  p.counters = counters;
  p.status = status;
  if (dfl::tc::gemm(mw, mx, bn, p, s) != cudaSuccess) return DFLASH_ECUDA;
  int st = 0;
  if (cudaMemcpyAsync(&st, status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return DFLASH_ECUDA;
  return st ? DFLASH_EDEVICE : DFLASH_OK;
}
