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
};

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
  // stream-K
  float *ws;          // partial slots: 2 * grid * BN * 128 floats
  int *counters;      // per tile, zero between launches
  int grid_cap;       // 0 = one CTA per SM
  // lm_head
  const int32_t *bitmask;  // [n_seq][mask_words] or NULL
  int mask_words;
  int nd;             // draft rows per sequence (row a belongs to sequence a / nd)
  LmPartial *lm_part; // [m_act][tiles_m]
  int *status;
  // filled by the launcher
  int tiles_m, tiles_n;
};

namespace tc {
int num_sms();
int pick_bn(int m_act);
// 2-D row-major map [rows, cols], box = 128 bytes of a row x box_rows rows, 128B swizzle.
bool make_map_2d(CUtensorMap *map, const void *base, bool fp8, int64_t rows, int64_t cols,
                 int box_rows);
cudaError_t gemm(const CUtensorMap &map_w, const CUtensorMap &map_x, int bn, GemmParams p,
                 cudaStream_t s);
// Bytes of stream-K partial workspace for the widest tile and a full grid.
inline size_t ws_floats(int grid) { return (size_t)2 * grid * 256 * 128; }
}  // namespace tc

// Merges the lm_head partials of each draft row: (argmax id or -1, top-1 prob).
cudaError_t lm_reduce(const LmPartial *part, int rows, int tiles, int32_t *row_id, float *row_p1,
                      cudaStream_t s);

}  // namespace dfl
