// Device side of a head: weights as the kernels see them, scratch buffers,
// and the kernel sequence of prefill and propose.
#pragma once

#include <vector>

#include "attention.h"
#include "chain.h"
#include "dflash.h"
#include "gemm_tc.h"
#include "internal.h"

struct dflash_handle;
struct dflash_state;

namespace dfl {

struct Weights {
  const bf16 *embed = nullptr, *lm_head = nullptr, *fc = nullptr, *hidden_norm = nullptr,
             *norm = nullptr;
  const uint8_t *lm_fp8 = nullptr;
  const float *lm_scale = nullptr, *inv_freq = nullptr, *kv_scale = nullptr;
  bool lm_is_fp8 = false;
  // lm_head streamed as codes (tc::LM_LOWP_FP8 / LM_LOWP_NVFP4; 0 = bf16):
  // code and block-scale maps, and the factor every logit takes (NVFP4)
  int lm_lowp = 0;
  CUtensorMap map_lm_codes, map_lm_scales;
  float lm_gscale = 0.f;
  std::vector<LayerW> layers;
  const bf16 *const *k_norm_dev = nullptr;  // device array of L k_norm gains
  bf16 *w_kv = nullptr;                     // [L*2*kv, H], rows [K0; V0; K1; V1; ...]
  float *cos_t = nullptr, *sin_t = nullptr; // [max_seq_len + gamma][d/2]
  void *pool = nullptr;                     // [pages][L][K|V][nkv][B][d]
  // TMA maps of the weights (box: 128 weight rows x 64 K)
  CUtensorMap map_fc, map_wkv, map_lm, map_lm256;
  std::vector<CUtensorMap> map_qkv, map_o, map_gu, map_down;
};

// Activation operands of the tensor-core GEMMs, one TMA map per tile width.
enum ActBuf { ACT_H = 0, ACT_O, ACT_U, ACT_Z, ACT_PACK, ACT_C, ACT_Z16, ACT_COUNT };
constexpr int BN_COUNT = 5;   // 16, 32, 64, 128, 256
inline int bn_index(int bn) { return bn == 16 ? 0 : bn == 32 ? 1 : bn == 64 ? 2 : bn == 128 ? 3 : 4; }

struct Buffers {
  float *x = nullptr;          // [R, H] residual
  bf16 *h = nullptr;           // [R, H] normed GEMM input
  bf16 *q = nullptr, *kb = nullptr, *vb = nullptr, *o = nullptr;
  bf16 *u = nullptr;           // [R, I]
  float *qkv_dense = nullptr;  // [R, qkv_w] f32 QKV of a many-row call
  bf16 *z = nullptr;           // [D, H] final-normed draft rows
  uint16_t *z16 = nullptr;     // [D, H] the same rows as f16 bits (streamed lm_head operand)
  int32_t *row_id = nullptr;
  float *row_p1 = nullptr;
  bf16 *ctx_pack = nullptr;    // [M, S]
  float *ctx_fc = nullptr;     // [M, H]
  bf16 *ctx_c = nullptr;       // [M, H]
  float *ctx_kv = nullptr;     // [M, L*2*kv]
  int *status = nullptr;
  char *out_dev = nullptr, *out_host = nullptr;
  size_t out_bytes = 0, off_drafts = 0, off_nout = 0, off_conf = 0;
  float *tap_x = nullptr;
  bf16 *tap_z = nullptr;
  float *tap_logits = nullptr;
  cudaEvent_t probe_begin = nullptr, probe_end = nullptr;  // around the lm_head stage
  cudaEvent_t step_begin = nullptr, step_end = nullptr;    // around the whole device step
  CUtensorMap act_map[ACT_COUNT][BN_COUNT];
  float *ws = nullptr;          // stream-K partials
  int *counters = nullptr;      // stream-K tile arrival counters (zero between launches)
  int n_counters = 0;
  LmPartial *lm_part = nullptr; // [D_max][vocab tiles]
  float *attn_ws = nullptr;     // split-KV attention partial slots
  AttnMaps attn_maps;           // tensor-core attention operands (ok = false: mma.sync kernel)
  int attn_grid_tc = 0;         // persistent CTAs of the tensor-core attention
  int attn_slots = 0;           // slot capacity
  int64_t attn_slot_floats = 0; // n_q*d + 2*n_q per slot
  int64_t fault_ns = 0;         // test hook of every GEMM launch (GemmParams::fault_ns)
  // few-row (chained) proposes
  float *ss_in = nullptr;       // [H/128][16] per-tile sums of squares of the residual entering a layer
  float *ss_mid = nullptr;      // [H/128][16] ... of the residual after o_proj
  float *ss_c = nullptr;        // [H/128][16] ... of the new ctx rows (hidden_norm's input)
  int *chain_sync = nullptr;    // per launch and phase: arrival counters, tile flags, tile count
  bf16 *hn = nullptr;           // [2][16][H] normed residual rows (gate/up input; QKV or lm_head input)
  CUtensorMap map_hn[2];        // their B-operand maps, box 16 rows x 64
  float *ca_ws = nullptr;       // chained attention partials: [16 * d + 32] f32 per item
  CUtensorMap *map_table = nullptr;   // device: the chained path's tensor maps (MT_* rows)
  CUtensorMap ca_pool, ca_kb, ca_vb;   // chained attention operands, box 16 rows x 64
  bool ca_pool_ok = false;
  int chain_sync_ints = 0;
  bool use_chain = true;        // few-row proposes take the chained path when it applies
  int last_chained = 0;         // the last forward took the chained path
};

// Cuts every (sequence, kv head) key range of the call into split-KV items
// (ctx chunks plus one block-key item) within the workspace's slot capacity.
// With grid_tc > 0 the items are also balanced over grid_tc persistent CTAs
// of the tensor-core kernel: CTA b runs items [cta_off[b], cta_off[b + 1]).
// Returns false (and no items) when even one chunk per window needs more
// slots than slot_cap; a handle's capacity always holds its widest call.
int attn_ctx_waves(int grid_tc);
bool build_attn_work(const Geo &g, const std::vector<SeqMeta> &seq, int slot_cap, int grid_tc,
                     std::vector<AttnItem> *items, std::vector<AttnPair> *pairs,
                     std::vector<int32_t> *cta_off);
// The same for a given SM count (the chunk size aims at three SM waves);
// needs no device, so host-side tests can call it.
bool build_attn_work_sms(const Geo &g, const std::vector<SeqMeta> &seq, int slot_cap,
                         int grid_tc, int sms, std::vector<AttnItem> *items,
                         std::vector<AttnPair> *pairs, std::vector<int32_t> *cta_off);

struct CallMeta {
  const SeqMeta *seq = nullptr;
  const RowMeta *rows = nullptr;
  const int32_t *page_ids = nullptr;
  const AttnItem *items = nullptr;
  const AttnPair *pairs = nullptr;
  const int32_t *cta_off = nullptr;   // tensor-core attention schedule (grid_tc + 1)
  const int *counts = nullptr;   // device: items, pairs, chained attention items
  const ChainAttnItem *citems = nullptr;   // chained path: attention items of the call
  int n_seq = 0, n_rows = 0, n_items = 0, n_pairs = 0;
  int cap_items = 0, cap_pairs = 0;
};

// The attention work of a chained call: per (sequence, query head), its key
// tiles (the window's ctx pages, then one tile of block keys) cut into at
// most `ctas` / pairs chunks. Items are listed pair by pair.
void build_chain_attn_items(const Geo &g, const std::vector<SeqMeta> &seq, int ctas,
                            std::vector<ChainAttnItem> *items);
// Item capacity of a head's chained calls.
int chain_attn_capacity(const Geo &g);

// Rows of the device table of a head's chained-path tensor maps: fixed
// operands, then per layer l its QKV, o_proj, gate/up and down weights.
enum : int {
  MT_EMPTY = 0, MT_POOL = 1, MT_KB = 2, MT_VB = 3,   // pool, kb, vb consecutive (attention)
  MT_FC = 4, MT_WKV = 5, MT_LM = 6,
  MT_PACK = 7, MT_CTXC = 8, MT_HN_MID = 9, MT_HN_IN = 10, MT_O16 = 11, MT_U16 = 12,
  MT_LAYERS = 13
};
inline int mt_layer(int l, int which) { return MT_LAYERS + 4 * l + which; }
inline int mt_count(int L) { return MT_LAYERS + 4 * L; }

// Ints of chained-propose counters a head needs (every launch of one forward).
int chain_sync_capacity(const Geo &g);
// Whether a call of n_rows new ctx rows and R block rows takes the chained path.
bool chain_applies(const Geo &g, const Buffers &B, int n_rows, int R);

int build_device_side(const dflash_config &c, const Geo &g, const dflash_weights *w, int R_max,
                      int D_max, int M_ctx, Weights *W, Buffers *B, std::vector<void *> *dev,
                      std::vector<void *> *host);
const char *last_build_error();

// Kernels launched by this library since load (all handles).
int64_t launch_count();
void count_launches(int n);

// Ctx rows: pack, fc GEMM, hidden_norm, fused K/V GEMM, k_norm + RoPE + paged write.
int ctx_append(const Geo &g, const Weights &W, const Buffers &B, const RowMeta *rows, int m,
               int M_ctx, cudaStream_t s);

// The whole propose forward for the call's sequences; results land in B.out_dev.
int forward(const Geo &g, const dflash_config &c, const Weights &W, const Buffers &B,
            const CallMeta &cm, int nd, const int32_t *bitmask, int M_ctx, cudaStream_t s);

cudaError_t gather_kv_rows(const Geo &g, const Weights &W, const Buffers &B, const RowMeta *rows,
                           int n, int layer, float *k_out, float *v_out, cudaStream_t s);

int propose_impl(dflash_handle *h, int n, dflash_state *const *states,
                 const uint32_t *last_tokens, const int64_t *positions,
                 const void *const *new_rows, const int32_t *n_new, int num_drafts,
                 const int32_t *bitmask, uint32_t *drafts, int32_t *n_out, float *conf,
                 void *stream);

}  // namespace dfl
