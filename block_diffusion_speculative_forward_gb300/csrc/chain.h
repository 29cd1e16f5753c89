// The multi-phase weight-streaming kernel of few-row proposes (chain.cu):
// its phases, arguments and launchers.
#pragma once

#include <cuda.h>

#include "gemm_tc.h"
#include "internal.h"

namespace dfl {

// What a phase computes after its GEMM y[a, f] = sum_k B[a, k] W[f, k].
enum ChainKind : int {
  CK_FC = 0,   // ctx rows: c = y (f32) and per-tile sums of squares (hidden_norm's input)
  CK_KV,       // fused ctx K/V: k_norm + RoPE on K heads, paged write of K and V
  CK_QKV,      // block QKV: per-head q/k RMSNorm + RoPE, bf16 q, k, v
  CK_O,        // o_proj: residual x += y, per-tile sums of squares
  CK_GU,       // gate/up: SwiGLU into u (bf16), tile-ready flags for the down phase
  CK_DOWN,     // down: residual x += y, per-tile sums of squares, residual tap
  CK_LM,       // lm_head: per (draft row, vocab tile) max / lowest argmax / sum exp
  CK_ATTN,     // block attention (no weights): o rows per head, head-ready counts in flag
};

// One attention item: sequence s, query head j, key tiles [t0, t1) of the
// sequence (ctx tiles of 16 positions from the window start's page, then one
// tile of block keys); its partial goes to slot `slot`; the pair (s, j) has
// nc items in slots slot0 .. slot0 + nc - 1.
struct ChainAttnItem {
  int32_t s, j, t0, t1, slot, slot0, nc, pad;
};

// The attention phase of a launch (at most one, and first in its launch).
struct ChainAttn {
  Geo geo;
  int layer;
  float scale;               // 1 / sqrt(head_dim)
  const SeqMeta *seq;
  const int32_t *page_ids;
  const int *count;          // device: items of the call
  const ChainAttnItem *items;
  const bf16 *q;             // [R, nq * d]
  bf16 *o;                   // [R, nq * d]
  float *ws;                 // item partials: [16 * d + 32] f32 each
};

constexpr int CHAIN_MAX_PHASES = 48;
constexpr int CHAIN_BN = 16;        // activation rows of every phase (one MMA N)
constexpr int CHAIN_BK = 64;        // reduction elements per stage
constexpr int CHAIN_MAX_K_NORM = 2048;   // the widest normed input (hidden) the chain takes

struct ChainPhase {
  int kind;
  int map_w, map_b;      // tensor maps (indices into ChainArgs::maps) of the weight and the B operand
  int slot_set;          // which of the three stream-K partial sets the phase uses
  int attn_layer;        // CK_ATTN: the layer
  int n_w, k;            // weight rows (outputs), reduction length (multiple of 64)
  int rows;              // valid activation rows (<= 16)
  int tiles_m, kb;       // n_w / 128 rounded up, k / 64
  // B operand: TMA of the bf16 activation map b of this phase. b_norm = 1:
  // that activation is hbuf = RMSNorm(nsrc; ngain) [16, k], which CTA j
  // writes for k-block j from the f32 rows nsrc [rows, k] and their per-tile
  // sums of squares nss [k/128][16] (rows past `rows` are zero), then sets
  // hflag[j] and counts hdone
  int b_norm;
  const float *nsrc;
  const float *nss;
  const bf16 *ngain;
  bf16 *hbuf;
  int *hflag;            // [kb] (zero at launch)
  int *hdone;            // (zero at launch)
  // dependency of the B operand on an earlier phase of the same launch:
  // dep < 0 none; dep_tile 0: every tile of phase dep finished; 1: k-block j
  // waits for tile j of phase dep
  int dep, dep_tile;
  // with dep_tile: k-block j waits until flag[j / dep_div] of phase dep
  // reaches dep_need (1 for a tile flag; the sequence count for a head)
  int dep_div, dep_need;
  // CK_ATTN: a second phase whose tiles must all be finished first (the
  // fused ctx K/V of the same launch), or -1
  int dep2;
  // the epilogue reads residual rows another phase of the launch wrote
  // (res_dep >= 0): it takes that phase's finished-tile count (all of them)
  // with acquire semantics before its first finished tile
  int res_dep;
  int *arrive;           // [tiles_m] stream-K arrival counters (zero at launch)
  int *flag;             // [tiles_m] 1 once the tile's epilogue has finished (zero at launch)
  int *done;             // tiles finished (zero at launch)
  // CK_FC / CK_O / CK_DOWN
  float *out;            // [rows, n_w] f32 (FC: stored; O/DOWN: the residual, added to)
  float *out_ss;         // [tiles_m][16] per-tile sums of squares of out
  float *x_tap;          // CK_DOWN: copy of the updated residual, or NULL
  // CK_LM: the normed rows the phase multiplies, for the debug taps (CTA 0
  // writes them): draft rows [n_seq * nd, k] and every block row [rows, k]
  bf16 *z_rows, *z_tap;
  // CK_KV
  const RowMeta *ctx_rows;
  const bf16 *const *k_norm;
  void *pool;
  const float *kv_scale;
  Geo geo;
  // epilogue parameters of CK_QKV / CK_GU / CK_LM (and the RoPE tables)
  GemmParams ep;
};

struct ChainArgs {
  int n_phases;
  ChainPhase ph[CHAIN_MAX_PHASES];
  ChainAttn attn;        // the CK_ATTN phases' work (their layer is per phase)
  const CUtensorMap *maps;   // device table of the launch's tensor maps
  int map_pool, map_kb, map_vb;   // attention: KV pool rows, block K and V
  float *ws;             // stream-K partials: set s uses slots [2 G s, 2 G (s + 1)) of 16 x 128 f32
  int *status;
  int64_t fault_ns;      // test hook, as GemmParams::fault_ns
};

namespace tc {
// Shared memory of one chain CTA (bytes, dynamic).
int chain_smem();
// Launches one chain over every SM (one persistent CTA each). The phases run
// in order; each CTA walks its stream-K range of every phase.
cudaError_t chain(const ChainArgs &a, cudaStream_t s);
}  // namespace tc

// The rows of a chained propose before its first chain: block embed (x,
// per-tile sums of squares, residual tap) of R rows and the pack of m new
// ctx rows.
cudaError_t chain_prologue(const bf16 *E, const SeqMeta *seq, int R, const Geo &g,
                           uint32_t mask_token, float *x, float *ss, float *x_tap,
                           const RowMeta *rows, int m, bf16 *pack, int *status, cudaStream_t s);

}  // namespace dfl
