// Device-side construction of a head and the kernel sequence of one propose.
//
// Sources: [P1] "Struct BlockDiffusionDraftHead" (spark_model docs),
// [P2] "BlockDiffusionDraftHead" (metrale docs).
#include <atomic>
#include <cstdio>
#include <cstring>
#include <functional>
#include <queue>
#include <string>

#include <algorithm>
#include <cmath>

#include "chain.h"
#include "consumers.h"
#include "forward.h"

namespace dfl {

namespace {
thread_local std::string g_build_err;

int berr(int code, const char *what, cudaError_t e) {
  char buf[384];
  snprintf(buf, sizeof buf, "%s: %s", what, cudaGetErrorString(e));
  g_build_err = buf;
  return code;
}

#define BK(call)                                                  \
  do {                                                            \
    cudaError_t e_ = (call);                                      \
    if (e_ != cudaSuccess) return berr(DFLASH_ECUDA, #call, e_);  \
  } while (0)

template <class T>
int dalloc(std::vector<void *> *dev, T **p, size_t count) {
  *p = nullptr;
  if (count == 0) return DFLASH_OK;
  void *q = nullptr;
  cudaError_t e = cudaMalloc(&q, count * sizeof(T));
  if (e != cudaSuccess) return berr(DFLASH_ENOMEM, "cudaMalloc", e);
  dev->push_back(q);
  *p = (T *)q;
  return DFLASH_OK;
}

#define BA(ptr, count)                               \
  do {                                               \
    int r_ = dalloc(dev, &(ptr), (size_t)(count));   \
    if (r_) return r_;                               \
  } while (0)
}  // namespace

const char *last_build_error() { return g_build_err.c_str(); }

namespace {
std::atomic<int64_t> g_launches{0};
}
int64_t launch_count() { return g_launches.load(); }
void count_launches(int n) { g_launches += n; }

int build_device_side(const dflash_config &c, const Geo &g, const dflash_weights *w, int R_max,
                      int D_max, int M_ctx, Weights *W, Buffers *B, std::vector<void *> *dev,
                      std::vector<void *> *host) {
  if (!w->embed || (c.lm_head_dtype == 0 && !w->lm_head) || !w->fc || !w->hidden_norm ||
      !w->norm || !w->inv_freq || !w->layers) {
    g_build_err = "a required weight pointer is NULL";
    return DFLASH_EINVAL;
  }
  if (c.lm_head_dtype == 1 && (!w->lm_head_fp8 || !w->lm_head_scale)) {
    g_build_err = "lm_head_dtype 1 needs lm_head_fp8 and lm_head_scale";
    return DFLASH_EINVAL;
  }
  if (c.lm_head_dtype == 2 && (!w->lm_head_nvfp4 || !w->lm_head_nvfp4_scale ||
                               !(w->lm_head_nvfp4_global > 0.f))) {
    g_build_err = "lm_head_dtype 2 needs lm_head_nvfp4, lm_head_nvfp4_scale and a positive global";
    return DFLASH_EINVAL;
  }
  if (c.kv_dtype == 1 && !w->kv_scale) {
    g_build_err = "kv_dtype 1 needs kv_scale";
    return DFLASH_EINVAL;
  }
  W->embed = (const bf16 *)w->embed;
  W->lm_head = (const bf16 *)w->lm_head;
  W->lm_fp8 = (const uint8_t *)w->lm_head_fp8;
  W->lm_scale = w->lm_head_scale;
  W->lm_is_fp8 = c.lm_head_dtype == 1;
  W->fc = (const bf16 *)w->fc;
  W->hidden_norm = (const bf16 *)w->hidden_norm;
  W->norm = (const bf16 *)w->norm;
  W->inv_freq = w->inv_freq;
  W->kv_scale = w->kv_scale;
  const size_t H = g.H, kv = g.kv, I = g.I, qd = (size_t)g.nq * g.d;
  // Stitched weights: fused ctx K/V [L*2*kv, H] ([P1]/[P2] field
  // fused_kv_weight, rows [K0; V0; K1; V1; ...]) and, per layer, QKV
  // [q; k; v] and gate-up [gate; up], each one GEMM operand.
  BA(W->w_kv, (size_t)g.L * 2 * kv * H);
  bf16 *w_qkv = nullptr, *w_gu = nullptr;
  BA(w_qkv, (size_t)g.L * g.qkv_w * H);
  BA(w_gu, (size_t)g.L * 2 * I * H);
  std::vector<const bf16 *> knorm(g.L);
  W->layers.resize(g.L);
  for (int l = 0; l < g.L; ++l) {
    const void *const *p = w->layers + (size_t)l * 11;
    for (int t = 0; t < 11; ++t)
      if (!p[t]) {
        g_build_err = "a layer weight pointer is NULL";
        return DFLASH_EINVAL;
      }
    LayerW &L = W->layers[l];
    L.in_norm = (const bf16 *)p[0];
    L.q_norm = (const bf16 *)p[4];
    L.k_norm = (const bf16 *)p[5];
    L.post_norm = (const bf16 *)p[7];
    L.w_o = (const bf16 *)p[6];
    L.w_down = (const bf16 *)p[10];
    bf16 *qkv = w_qkv + (size_t)l * g.qkv_w * H;
    BK(cudaMemcpy(qkv, p[1], qd * H * 2, cudaMemcpyDeviceToDevice));
    BK(cudaMemcpy(qkv + qd * H, p[2], kv * H * 2, cudaMemcpyDeviceToDevice));
    BK(cudaMemcpy(qkv + (qd + kv) * H, p[3], kv * H * 2, cudaMemcpyDeviceToDevice));
    L.w_qkv = qkv;
    // gate/up rows alternate: row 2j = gate j, row 2j+1 = up j, so the two
    // inputs of SwiGLU feature j sit in adjacent accumulator lanes.
    bf16 *gu = w_gu + (size_t)l * 2 * I * H;
    BK(cudaMemcpy2D(gu, 2 * H * 2, p[8], H * 2, H * 2, I, cudaMemcpyDeviceToDevice));
    BK(cudaMemcpy2D(gu + H, 2 * H * 2, p[9], H * 2, H * 2, I, cudaMemcpyDeviceToDevice));
    L.w_gu = gu;
    bf16 *kvl = W->w_kv + (size_t)l * 2 * kv * H;
    BK(cudaMemcpy(kvl, p[2], kv * H * 2, cudaMemcpyDeviceToDevice));
    BK(cudaMemcpy(kvl + kv * H, p[3], kv * H * 2, cudaMemcpyDeviceToDevice));
    knorm[l] = L.k_norm;
  }
  const bf16 **kn = nullptr;
  BA(kn, (size_t)g.L);
  BK(cudaMemcpy(kn, knorm.data(), sizeof(void *) * g.L, cudaMemcpyHostToDevice));
  W->k_norm_dev = kn;
  // Low-precision lm_head ([P1] fields lm_head_shared_fp8, lm_head_nvfp4):
  // the codes stream as they are (lm_lowp.cu), dequantised on chip. FP8:
  // logits s_v * <z, codes_v>; NVFP4: g * <z, e2m1 * scale>.
  bool ok_lm = true;
  if (c.lm_head_dtype == 1) {
    W->lm_lowp = tc::LM_LOWP_FP8;
    ok_lm = tc::make_map_u8(&W->map_lm_codes, W->lm_fp8, g.V, H, 128, 128, true);
  } else if (c.lm_head_dtype == 2) {
    W->lm_lowp = tc::LM_LOWP_NVFP4;
    W->lm_gscale = w->lm_head_nvfp4_global;
    ok_lm = tc::make_map_u8(&W->map_lm_codes, w->lm_head_nvfp4, g.V, H / 2, 128, 128, true) &&
            tc::make_map_u8(&W->map_lm_scales, w->lm_head_nvfp4_scale, g.V, H / 16, 16, 128,
                            false);
  }
  // A propose with more than 16 draft rows is no longer bound by the table's
  // bytes but by tensor-core work, where converting the codes once per row
  // chunk costs more than it saves: those calls multiply by the table widened
  // to bf16 (exactly) once here, made only when such a call is possible.
  const void *lm_operand = W->lm_head;
  if (W->lm_lowp && (D_max > 16 || !tc::lm_lowp_fits(1, g.H))) {
    bf16 *wide = nullptr;
    BA(wide, (size_t)g.V * H);
    BK(widen_lm_table(c.lm_head_dtype, W->lm_lowp == tc::LM_LOWP_FP8
                                           ? W->lm_fp8 : (const uint8_t *)w->lm_head_nvfp4,
                      (const uint8_t *)w->lm_head_nvfp4_scale, g.V, H, wide, 0));
    BK(cudaDeviceSynchronize());
    lm_operand = wide;
  }
  // TMA maps of every weight operand.
  {
    bool ok = ok_lm && tc::make_map_2d(&W->map_fc, W->fc, false, H, g.S, 128) &&
              tc::make_map_2d(&W->map_wkv, W->w_kv, false, (int64_t)g.L * 2 * kv, H, 128) &&
              (!lm_operand ||
               (tc::make_map_2d(&W->map_lm, lm_operand, false, g.V, H, 128) &&
                tc::make_map_2d(&W->map_lm256, lm_operand, false, g.V, H, 256)));
    W->map_qkv.resize(g.L);
    W->map_o.resize(g.L);
    W->map_gu.resize(g.L);
    W->map_down.resize(g.L);
    for (int l = 0; l < g.L && ok; ++l) {
      const LayerW &L = W->layers[l];
      ok = tc::make_map_2d(&W->map_qkv[l], L.w_qkv, false, g.qkv_w, H, 128) &&
           tc::make_map_2d(&W->map_o[l], L.w_o, false, H, qd, 128) &&
           tc::make_map_2d(&W->map_gu[l], L.w_gu, false, 2 * I, H, 128) &&
           tc::make_map_2d(&W->map_down[l], L.w_down, false, H, I, 128);
    }
    if (!ok) {
      g_build_err = "cuTensorMapEncodeTiled failed for a weight operand";
      return DFLASH_ECUDA;
    }
  }
  // The chained few-row path reads norm gains 16 bytes at a time, and runs
  // the bf16 lm_head in its last phase.
  {
    auto al = [](const void *q) { return ((uintptr_t)q & 15) == 0; };
    bool ok = al(W->hidden_norm) && al(W->norm);
    for (const LayerW &L : W->layers) ok = ok && al(L.in_norm) && al(L.post_norm);
    B->use_chain = ok && c.lm_head_dtype == 0;
  }
  // RoPE table for every position a block row can reach.
  const int max_pos = c.max_seq_len + g.gamma;
  BA(W->cos_t, (size_t)max_pos * (g.d / 2));
  BA(W->sin_t, (size_t)max_pos * (g.d / 2));
  // YaRN's attention temperature scales every rotated q and k: folded into the table
  const float rope_scale = c.rope_attn_factor > 0.f ? c.rope_attn_factor : 1.f;
  BK(rope_table(W->inv_freq, max_pos, g.d / 2, rope_scale, W->cos_t, W->sin_t, 0));
  // KV pool.
  const size_t elem = g.kv_fp8 ? 1 : 2;
  const size_t pool_elems = (size_t)g.pages * g.L * 2 * g.nkv * g.B * g.d;
  if (pool_elems) {
    void *pool = nullptr;
    cudaError_t e = cudaMalloc(&pool, pool_elems * elem);
    if (e != cudaSuccess) return berr(DFLASH_ENOMEM, "KV pool cudaMalloc", e);
    dev->push_back(pool);
    W->pool = pool;
    BK(cudaMemset(pool, 0, pool_elems * elem));
  }
  // Scratch.
  BA(B->x, (size_t)R_max * H);
  BA(B->h, (size_t)R_max * std::max(H, I));
  BA(B->q, (size_t)R_max * qd);
  BA(B->kb, (size_t)R_max * kv);
  BA(B->vb, (size_t)R_max * kv);
  BA(B->o, (size_t)R_max * qd);
  BA(B->qkv_dense, (size_t)R_max * g.qkv_w);
  BA(B->u, (size_t)R_max * I);
  BA(B->z, (size_t)D_max * H);
  BA(B->z16, (size_t)D_max * H);
  BA(B->row_id, (size_t)D_max);
  BA(B->row_p1, (size_t)D_max);
  BA(B->ctx_pack, (size_t)M_ctx * g.S);
  BA(B->ctx_fc, (size_t)M_ctx * H);
  BA(B->ctx_c, (size_t)std::max(M_ctx, CHAIN_BN) * H);   // the chained path writes 16 rows
  BA(B->ctx_kv, (size_t)M_ctx * g.L * 2 * kv);
  BA(B->status, 4);
  BK(cudaMemset(B->status, 0, 16));
  // Stream-K workspace and counters; lm_head partials.
  const int sms = tc::num_sms();
  BA(B->ws, tc::ws_floats(sms));
  const int vt = (g.V + 127) / 128;
  B->n_counters = std::max(vt * ((D_max + 255) / 256 + 1),
                           ((std::max({g.qkv_w, 2 * g.I, g.L * 2 * g.kv, g.H}) + 127) / 128) *
                               ((std::max(R_max, M_ctx) + 15) / 16));
  BA(B->counters, (size_t)B->n_counters);
  BK(cudaMemset(B->counters, 0, sizeof(int) * (size_t)B->n_counters));
  BA(B->lm_part, (size_t)D_max * vt);
  // Few-row chained proposes: per-tile sums of squares of the residual and
  // of the new ctx rows, and every launch's tile counters and flags.
  {
    const int ht = (g.H + 127) / 128;
    BA(B->ss_in, (size_t)ht * 16);
    BA(B->ss_mid, (size_t)ht * 16);
    BA(B->ss_c, (size_t)ht * 16);
    B->chain_sync_ints = chain_sync_capacity(g);
    BA(B->chain_sync, (size_t)B->chain_sync_ints);
    BA(B->hn, (size_t)2 * CHAIN_BN * H);
    BA(B->ca_ws, (size_t)chain_attn_capacity(g) * (16 * g.d + 32));
    B->ca_pool_ok = W->pool != nullptr;
    if ((B->ca_pool_ok &&
         !tc::make_map_2d(&B->ca_pool, W->pool, false, (int64_t)g.pages * g.L * 2 * g.nkv * g.B,
                          g.d, 16)) ||
        !tc::make_map_2d(&B->ca_kb, B->kb, false, R_max, kv, 16) ||
        !tc::make_map_2d(&B->ca_vb, B->vb, false, R_max, kv, 16) ||
        !tc::make_map_2d(&B->map_hn[0], B->hn, false, CHAIN_BN, H, CHAIN_BN) ||
        !tc::make_map_2d(&B->map_hn[1], B->hn + (size_t)CHAIN_BN * H, false, CHAIN_BN, H, CHAIN_BN)) {
      g_build_err = "cuTensorMapEncodeTiled failed for a normed activation";
      return DFLASH_ECUDA;
    }
  }
  // Split-KV attention partials: at most two ctx chunks per (sequence, kv
  // head) beyond 3 x SMs, plus one block-key item each.
  {
    const int n_q = attn_query_rows(g);
    if (n_q > 128) {
      g_build_err = "gamma * (num_q_heads / num_kv_heads) must be <= 128";
      return DFLASH_EINVAL;
    }
    // slots start on 16 bytes (vector stores and loads of partial rows)
    B->attn_slot_floats = ((int64_t)n_q * g.d + 2 * n_q + 3) & ~(int64_t)3;
    // The tensor-core kernel reads whole 16-row blocks of the block K/V
    // rows (masked past gamma): keep never-written rows finite.
    BK(cudaMemset(B->kb, 0, sizeof(bf16) * (size_t)R_max * kv));
    BK(cudaMemset(B->vb, 0, sizeof(bf16) * (size_t)R_max * kv));
    if (!attention_tc_maps(g, R_max, B->q, W->pool, B->kb, B->vb, &B->attn_maps)) {
      g_build_err = "cuTensorMapEncodeTiled failed for an attention operand";
      return DFLASH_ECUDA;
    }
    B->attn_grid_tc = B->attn_maps.ok ? sms : 0;
    B->attn_slots = attn_ctx_waves(B->attn_grid_tc) * sms + 3 * c.max_batch * g.nkv + 64;
    BA(B->attn_ws, (size_t)B->attn_slots * B->attn_slot_floats);
  }
  // TMA maps of the activation operands, one per tile width.
  {
    struct A { int id; const void *p; int64_t rows, cols; } acts[ACT_COUNT] = {
        {ACT_H, B->h, R_max, (int64_t)H}, {ACT_O, B->o, R_max, (int64_t)qd},
        {ACT_U, B->u, R_max, (int64_t)I}, {ACT_Z, B->z, D_max, (int64_t)H},
        {ACT_PACK, B->ctx_pack, M_ctx, (int64_t)g.S}, {ACT_C, B->ctx_c, M_ctx, (int64_t)H},
        {ACT_Z16, B->z16, D_max, (int64_t)H}};   // 16-bit elements: TMA moves f16 as bf16
    const int bns[BN_COUNT] = {16, 32, 64, 128, 256};
    for (auto &a : acts)
      for (int j = 0; j < BN_COUNT; ++j)
        if (!tc::make_map_2d(&B->act_map[a.id][j], a.p, false, a.rows, a.cols, bns[j])) {
          g_build_err = "cuTensorMapEncodeTiled failed for an activation operand";
          return DFLASH_ECUDA;
        }
  }
  // the chained path's tensor maps, in device memory (its launch parameters
  // hold only their rows)
  {
    std::vector<CUtensorMap> t(mt_count(g.L));
    memset(t.data(), 0, sizeof(CUtensorMap) * t.size());
    if (B->ca_pool_ok) t[MT_POOL] = B->ca_pool;
    t[MT_KB] = B->ca_kb;
    t[MT_VB] = B->ca_vb;
    t[MT_FC] = W->map_fc;
    t[MT_WKV] = W->map_wkv;
    t[MT_LM] = W->map_lm;
    t[MT_PACK] = B->act_map[ACT_PACK][bn_index(16)];
    t[MT_CTXC] = B->act_map[ACT_C][bn_index(16)];
    t[MT_HN_MID] = B->map_hn[0];
    t[MT_HN_IN] = B->map_hn[1];
    t[MT_O16] = B->act_map[ACT_O][bn_index(16)];
    t[MT_U16] = B->act_map[ACT_U][bn_index(16)];
    for (int l = 0; l < g.L; ++l) {
      t[mt_layer(l, 0)] = W->map_qkv[l];
      t[mt_layer(l, 1)] = W->map_o[l];
      t[mt_layer(l, 2)] = W->map_gu[l];
      t[mt_layer(l, 3)] = W->map_down[l];
    }
    BA(B->map_table, t.size());
    BK(cudaMemcpy(B->map_table, t.data(), sizeof(CUtensorMap) * t.size(), cudaMemcpyHostToDevice));
  }
  const int nb = c.max_batch;
  B->off_drafts = 16;
  B->off_nout = (B->off_drafts + (size_t)D_max * 4 + 15) & ~(size_t)15;
  B->off_conf = (B->off_nout + (size_t)nb * 4 + 15) & ~(size_t)15;
  B->out_bytes = B->off_conf + (size_t)nb * 4;
  BA(B->out_dev, B->out_bytes);
  void *hp = nullptr;
  BK(cudaMallocHost(&hp, B->out_bytes));
  host->push_back(hp);
  B->out_host = (char *)hp;
  BK(cudaDeviceSynchronize());
  return DFLASH_OK;
}

#define FK(call)                                                  \
  do {                                                            \
    cudaError_t e_ = (call);                                      \
    if (e_ != cudaSuccess) return berr(DFLASH_ECUDA, #call, e_);  \
  } while (0)

// A kernel launch of this library: checked and counted.
#define LK(call)          \
  do {                    \
    FK(call);             \
    count_launches(1);    \
  } while (0)

namespace {
// One tensor-core GEMM: out[m_act, n_w] (epi)= act[m_act, k] * W[n_w, k]^T.
// dp: whole tiles per CTA, tile width from the data-parallel cost model.
cudaError_t tc_gemm(const Buffers &B, const CUtensorMap &map_w, ActBuf act, int m_act, int n_w,
                    int k, int epi, void *out, int ldo, cudaStream_t s, bool dp = false) {
  GemmParams p{};
  p.m_act = m_act;
  p.n_w = n_w;
  p.k = k;
  p.epi = epi;
  p.out = out;
  p.ldo = ldo;
  p.ws = B.ws;
  p.counters = B.counters;
  p.status = B.status;
  p.fault_ns = B.fault_ns;
  p.dp = dp;
  const int bn = dp ? tc::pick_bn_dp(m_act, n_w, k) : tc::pick_bn(m_act);
  return tc::gemm(map_w, B.act_map[act][bn_index(bn)], bn, p, s);
}
}  // namespace

namespace {

// A projection whose consumer reads it through a Partials view: split-K
// partials when the shape allows (no inter-CTA fixup in the GEMM), otherwise
// a dense f32 store into `dense` [m_act, n_w].
int project(const Buffers &B, const CUtensorMap &map_w, ActBuf act, int m_act, int n_w, int k,
            float *dense, Partials *view, cudaStream_t s) {
  GemmParams p{};
  p.m_act = m_act;
  p.n_w = n_w;
  p.k = k;
  p.ws = B.ws;
  p.counters = B.counters;
  p.status = B.status;
  p.fault_ns = B.fault_ns;
  const int bn = tc::pick_bn(m_act);
  if (tc::partial_ok(m_act, n_w, k)) {
    p.epi = EPI_TC_PARTIAL;
    LK(tc::gemm(map_w, B.act_map[act][bn_index(bn)], bn, p, s, view));
  } else {
    p.epi = EPI_TC_STORE_F32;
    p.out = dense;
    p.ldo = n_w;
    LK(tc::gemm(map_w, B.act_map[act][bn_index(bn)], bn, p, s));
    *view = Partials{};
    view->dense = dense;
    view->ld = n_w;
  }
  return DFLASH_OK;
}

}  // namespace

int ctx_append(const Geo &g, const Weights &W, const Buffers &B, const RowMeta *rows, int m,
               int M_ctx, cudaStream_t s) {
  const int kvw = g.L * 2 * g.kv;
  for (int a = 0; a < m; a += M_ctx) {
    const int mb = std::min(M_ctx, m - a);
    const RowMeta *r = rows + a;
    LK(pack_rows(r, mb, g.S, B.ctx_pack, s));
    Partials fcv, kvv;
    int rc = project(B, W.map_fc, ACT_PACK, mb, g.H, g.S, B.ctx_fc, &fcv, s);
    if (rc) return rc;
    AddNormArgs an{};
    an.x = nullptr;
    an.has_y = true;
    an.y = fcv;
    an.g = W.hidden_norm;
    an.eps = g.eps;
    an.n = g.H;
    an.out = B.ctx_c;
    LK(add_norm(an, mb, s));
    rc = project(B, W.map_wkv, ACT_C, mb, kvw, g.H, B.ctx_kv, &kvv, s);
    if (rc) return rc;
    LK(ctx_kv_write(kvv, mb, r, g, W.k_norm_dev, W.cos_t, W.sin_t, W.pool, W.kv_scale, B.status,
                    s));
  }
  return DFLASH_OK;
}

int chain_sync_capacity(const Geo &g) {
  auto t = [](int64_t n) { return (int)((n + 127) / 128); };
  // per phase: arrival counters and flags per tile, the tile count, the
  // normed operand's k-block count and flags (+ padding); see forward_chain
  auto ph = [](int tiles, int k) { return 2 * tiles + 4 + (k / CHAIN_BK + 3) / 4 * 4; };
  const int first = ph(t(g.H), g.S) + ph(t((int64_t)g.L * 2 * g.kv), g.H) + ph(t(g.qkv_w), g.H);
  // the attention phase counts (sequence, head) pairs: at most 16 sequences
  const int layer = ph(16 * g.nq, 0) + ph(t(g.H), g.nq * g.d) + ph(t(2 * (int64_t)g.I), g.H) +
                    ph(t(g.H), g.I) + std::max(ph(t(g.qkv_w), g.H), ph(t(g.V), g.H));
  return first + g.L * layer + 64;
}

bool chain_applies(const Geo &g, const Buffers &B, int n_rows, int R) {
  // bf16 cache in pages of 16 for the in-launch attention; every phase of
  // the forward in one launch
  return B.use_chain && 3 + 5 * g.L <= CHAIN_MAX_PHASES && R <= CHAIN_BN && n_rows <= CHAIN_BN && g.H <= CHAIN_MAX_K_NORM &&
         g.H % 128 == 0 && g.S % CHAIN_BK == 0 && g.I % CHAIN_BK == 0 && B.chain_sync &&
         !g.kv_fp8 && g.B == 16 && (g.d == 64 || g.d == 128) && g.gamma <= CHAIN_BN;
}

int chain_attn_capacity(const Geo &g) { return tc::num_sms() + (CHAIN_BN / 2) * g.nq + 16; }

void build_chain_attn_items(const Geo &g, const std::vector<SeqMeta> &seq, int ctas,
                            std::vector<ChainAttnItem> *items) {
  items->clear();
  const int pairs = (int)seq.size() * g.nq;
  const int nc_target = std::max(1, ctas / std::max(1, pairs));
  for (int s = 0; s < (int)seq.size(); ++s) {
    const int n_ctx = seq[s].pos - seq[s].ws;
    const int p0 = seq[s].ws & ~15;
    const int T = (n_ctx > 0 ? (seq[s].pos - p0 + 15) / 16 : 0) + 1;   // + the block tile
    int nc = std::min(nc_target, T);
    const int chunk = (T + nc - 1) / nc;
    nc = (T + chunk - 1) / chunk;
    for (int j = 0; j < g.nq; ++j) {
      const int slot0 = (int)items->size();
      for (int c = 0; c < nc; ++c)
        items->push_back({s, j, c * chunk, std::min(T, (c + 1) * chunk), slot0 + c, slot0, nc, 0});
    }
  }
}

namespace {

// The chained propose of few rows (see chain.cu): the prologue (block embed,
// pack of the new ctx rows), then one persistent launch whose phases are the
// new ctx rows (fc, fused K/V), layer 0's QKV, and per layer the attention,
// o_proj, gate/up, down and the next QKV (or the lm_head); then the row merge
// of the lm_head partials and the chain of drafts.
int forward_chain(const Geo &g, const dflash_config &c, const Weights &W, const Buffers &B,
                  const CallMeta &cm, int nd, const int32_t *bitmask, cudaStream_t s) {
  if (B.step_begin && B.step_end) FK(cudaEventRecordWithFlags(B.step_begin, s, cudaEventRecordExternal));
  const int n = cm.n_seq, R = n * g.gamma, D = n * nd, m = cm.n_rows;
  const int qd = g.nq * g.d;
  FK(cudaMemsetAsync(B.chain_sync, 0, sizeof(int) * (size_t)B.chain_sync_ints, s));
  LK(chain_prologue(W.embed, cm.seq, R, g, c.mask_token_id, B.x, B.ss_in, B.tap_x, cm.rows, m,
                    B.ctx_pack, B.status, s));
  int *sync = B.chain_sync;
  ChainArgs a{};
  int np = 0, weight_phases = 0;
  // appends a phase: its counters from the sync area, its tensor maps, and
  // (weight phases) the next of three stream-K partial sets in turn, so a set
  // is reused only by a phase that depends on the set's previous user
  auto add = [&](int kind, int n_w, int k, int rows, int map_w, int map_b) -> ChainPhase & {
    ChainPhase &P = a.ph[np++];
    P = ChainPhase{};
    P.kind = kind;
    P.n_w = n_w;
    P.k = k;
    P.rows = rows;
    // the attention phase has no weights; its "tiles" are the (sequence,
    // head) pairs, whose count `done` reaches when every pair is merged
    P.tiles_m = kind == CK_ATTN ? n * g.nq : (n_w + 127) / 128;
    P.kb = k / CHAIN_BK;
    P.map_w = map_w;
    P.map_b = map_b;
    P.slot_set = kind == CK_ATTN ? 0 : weight_phases++ % 3;
    P.dep = -1;
    P.dep2 = -1;
    P.res_dep = -1;
    P.arrive = sync;
    P.flag = sync + P.tiles_m;
    P.done = sync + 2 * P.tiles_m;
    P.hdone = P.done + 1;
    P.hflag = sync + 2 * P.tiles_m + 4;
    sync += 2 * P.tiles_m + 4 + (P.kb + 3) / 4 * 4;
    P.geo = g;
    P.ep.m_act = rows;
    P.ep.n_w = n_w;
    P.ep.k = k;
    P.ep.eps = g.eps;
    P.ep.status = B.status;
    P.ep.tiles_m = P.tiles_m;
    P.ep.tiles_n = 1;
    P.ep.cos_t = W.cos_t;
    P.ep.sin_t = W.sin_t;
    return P;
  };
  auto normed = [](ChainPhase &P, const float *src, const float *ss, const bf16 *gain, bf16 *h) {
    P.b_norm = 1;
    P.nsrc = src;
    P.nss = ss;
    P.ngain = gain;
    P.hbuf = h;
  };
  bf16 *const hn_mid = B.hn, *const hn_in = B.hn + (size_t)CHAIN_BN * g.H;
  auto add_qkv = [&](int l) -> int {
    ChainPhase &P = add(CK_QKV, g.qkv_w, g.H, R, mt_layer(l, 0), MT_HN_IN);
    normed(P, B.x, B.ss_in, W.layers[l].in_norm, hn_in);
    P.ep.seq = cm.seq;
    P.ep.gamma = g.gamma;
    P.ep.head_dim = g.d;
    P.ep.q_rows = qd;
    P.ep.k_rows = g.kv;
    P.ep.q_norm = W.layers[l].q_norm;
    P.ep.k_norm = W.layers[l].k_norm;
    P.ep.q_out = B.q;
    P.ep.k_out = B.kb;
    P.ep.v_out = B.vb;
    return np - 1;
  };
  // new ctx rows: fc, hidden_norm, fused K/V with the paged write
  int kv_phase = -1;
  if (m > 0) {
    ChainPhase &fc = add(CK_FC, g.H, g.S, m, MT_FC, MT_PACK);
    fc.out = B.ctx_fc;
    fc.out_ss = B.ss_c;
    const int fc_i = np - 1;
    ChainPhase &kv = add(CK_KV, g.L * 2 * g.kv, g.H, m, MT_WKV, MT_CTXC);
    normed(kv, B.ctx_fc, B.ss_c, W.hidden_norm, B.ctx_c);
    kv.dep = fc_i;
    kv.ctx_rows = cm.rows;
    kv.k_norm = W.k_norm_dev;
    kv.pool = W.pool;
    kv.kv_scale = W.kv_scale;
    kv_phase = np - 1;
  }
  int qkv_i = add_qkv(0);
  for (int l = 0; l < g.L; ++l) {
    const LayerW &L = W.layers[l];
    // attention of layer l once its QKV (and the new ctx rows' K/V) are in
    ChainPhase &at = add(CK_ATTN, 0, 0, R, MT_EMPTY, MT_EMPTY);
    at.dep = qkv_i;
    at.dep2 = l == 0 ? kv_phase : -1;
    at.attn_layer = l;
    const int at_i = np - 1;
    ChainPhase &o = add(CK_O, g.H, qd, R, mt_layer(l, 1), MT_O16);
    o.dep = at_i;
    o.dep_tile = 1;
    o.dep_div = g.d / CHAIN_BK;   // k-block j reads head j * 64 / d
    o.dep_need = n;               // every sequence's rows of that head
    o.out = B.x;
    o.out_ss = B.ss_mid;
    const int o_i = np - 1;
    ChainPhase &gu = add(CK_GU, 2 * g.I, g.H, R, mt_layer(l, 2), MT_HN_MID);
    normed(gu, B.x, B.ss_mid, L.post_norm, hn_mid);
    gu.dep = o_i;
    gu.ep.u_out = B.u;
    const int gu_i = np - 1;
    ChainPhase &dn = add(CK_DOWN, g.H, g.I, R, mt_layer(l, 3), MT_U16);
    dn.dep = gu_i;
    dn.dep_tile = 1;
    dn.dep_div = 1;
    dn.dep_need = 1;
    dn.res_dep = o_i;
    dn.out = B.x;
    dn.out_ss = B.ss_in;
    dn.x_tap = B.tap_x ? B.tap_x + (size_t)(l + 1) * R * g.H : nullptr;
    const int dn_i = np - 1;
    if (l + 1 < g.L) {
      qkv_i = add_qkv(l + 1);
      a.ph[qkv_i].dep = dn_i;
    } else {
      ChainPhase &lm = add(CK_LM, g.V, g.H, R, MT_LM, MT_HN_IN);
      normed(lm, B.x, B.ss_in, W.norm, hn_in);
      lm.dep = dn_i;
      lm.ep.wscale = W.lm_is_fp8 ? W.lm_scale : nullptr;
      lm.ep.bitmask = bitmask;
      lm.ep.mask_words = (g.V + 31) / 32;
      lm.ep.nd = nd;
      lm.ep.lm_gamma = g.gamma;
      lm.ep.lm_first = g.draft0;
      lm.ep.lm_part = B.lm_part;
      lm.z_rows = B.z;
      lm.z_tap = B.tap_z;
    }
  }
  a.n_phases = np;
  a.attn.geo = g;
  a.attn.scale = (float)(1.0 / std::sqrt((double)g.d));
  a.attn.seq = cm.seq;
  a.attn.page_ids = cm.page_ids;
  a.attn.count = cm.counts + 2;
  a.attn.items = cm.citems;
  a.attn.q = B.q;
  a.attn.o = B.o;
  a.attn.ws = B.ca_ws;
  a.maps = B.map_table;
  a.map_pool = MT_POOL;
  a.map_kb = MT_POOL + 1;
  a.map_vb = MT_POOL + 2;
  a.ws = B.ws;
  a.status = B.status;
  a.fault_ns = B.fault_ns;
  LK(tc::chain(a, s));
  LK(lm_reduce(B.lm_part, D, (g.V + 127) / 128, B.row_id, B.row_p1, s));
  // (the lm_head runs inside the single launch: no separate lm_head probe here)
  if (B.tap_logits) {
    GemmParams p{};
    p.m_act = D;
    p.n_w = g.V;
    p.k = g.H;
    p.epi = EPI_TC_STORE_F32;
    p.out = B.tap_logits;
    p.ldo = g.V;
    p.wscale = W.lm_is_fp8 ? W.lm_scale : nullptr;
    p.ws = B.ws;
    p.counters = B.counters;
    p.status = B.status;
    const int bn = tc::pick_bn(D);
    LK(tc::gemm(W.map_lm, B.act_map[ACT_Z][bn_index(bn)], bn, p, s));
  }
  LK(finalize(B.row_id, B.row_p1, n, nd, B.status, (uint32_t *)(B.out_dev + B.off_drafts),
              (int32_t *)(B.out_dev + B.off_nout), (float *)(B.out_dev + B.off_conf),
              (int32_t *)B.out_dev, s));
  if (B.step_begin && B.step_end) FK(cudaEventRecordWithFlags(B.step_end, s, cudaEventRecordExternal));
  return DFLASH_OK;
}

}  // namespace

int forward(const Geo &g, const dflash_config &c, const Weights &W, const Buffers &B,
            const CallMeta &cm, int nd, const int32_t *bitmask, int M_ctx, cudaStream_t s) {
  if (chain_applies(g, B, cm.n_rows, cm.n_seq * g.gamma))
    return forward_chain(g, c, W, B, cm, nd, bitmask, s);
  if (B.step_begin && B.step_end) FK(cudaEventRecordWithFlags(B.step_begin, s, cudaEventRecordExternal));
  if (cm.n_rows) {
    int rc = ctx_append(g, W, B, cm.rows, cm.n_rows, M_ctx, s);
    if (rc) return rc;
  }
  const int n = cm.n_seq, R = n * g.gamma, D = n * nd;
  const int qd = g.nq * g.d;
  const int bnR = tc::pick_bn(R);
  // Many rows: the fused QKV and gate/up GEMMs run whole tiles per CTA
  // (data-parallel, epilogue in the GEMM); few rows: split-K partials read by
  // the consumer kernels, so every SM streams weights.
  // Many rows: QKV and gate/up run whole tiles per CTA (data-parallel; QKV
  // stored dense for the q/k pass, SwiGLU in the epilogue). Few rows: every
  // GEMM is split-K over all SMs (one SM streams only ~35 GB/s from HBM, so
  // the weight stream needs them all) and the consumers read the partials.
  const bool dp = R > 64;
  // Few rows, but gate/up has 128-row tiles for at least half the SMs: whole
  // tiles per CTA there too. Its stream-K fixup tail (partial write, fence,
  // atomic, the other contributors' partials) cost ~4 us per layer at batch
  // 1; whole tiles on 96 of the 152 SMs take the weight stream at ~45 GB/s
  // per SM, and the down projection's CTAs start on the idle SMs and load
  // their first weight stages meanwhile (measured 13.5 -> 10.3 us per
  // gate/up, 676 -> 652 us per propose).
  const bool gu_dp_few = !dp && 2 * ((2 * g.I + 127) / 128) >= tc::num_sms();
  const int bn_qkv = dp ? tc::pick_bn_dp(R, g.qkv_w, g.H) : bnR;
  const int bn_gu = dp ? tc::pick_bn_dp(R, 2 * g.I, g.H) : bnR;
  LK(embed_block(W.embed, cm.seq, n, g, c.mask_token_id, B.x, B.status, s));
  // The residual update of each o/down projection is applied by the RMSNorm
  // that follows it (pending), or by the GEMM itself when the partial mode
  // does not fit the shape.
  Partials pending{};
  bool has_pending = false;
  for (int l = 0; l < g.L; ++l) {
    const LayerW &L = W.layers[l];
    {
      AddNormArgs an{};
      an.x = B.x;
      an.has_y = has_pending;
      an.y = pending;
      an.g = L.in_norm;
      an.eps = g.eps;
      an.n = g.H;
      an.out = B.h;
      an.x_tap = B.tap_x ? B.tap_x + (size_t)l * R * g.H : nullptr;
      LK(add_norm(an, R, s));
    }
    // (at batch 1 the partials and a separate norm + RoPE pass measured
    // faster than the fused stream-K epilogue: 757 vs 791 us per step)
    const bool part = !dp && tc::partial_ok(R, g.qkv_w, g.H);
    if (dp) {
      // whole-tile QKV into a dense f32 buffer, then per-head q/k RMSNorm + RoPE
      GemmParams p{};
      p.m_act = R;
      p.n_w = g.qkv_w;
      p.k = g.H;
      p.epi = EPI_TC_STORE_F32;
      p.out = B.qkv_dense;
      p.ldo = g.qkv_w;
      p.ws = B.ws;
      p.counters = B.counters;
      p.status = B.status;
      p.fault_ns = B.fault_ns;
      p.dp = 1;
      LK(tc::gemm(W.map_qkv[l], B.act_map[ACT_H][bn_index(bn_qkv)], bn_qkv, p, s));
      QkvPostArgs qp{};
      qp.g = g;
      qp.y.dense = B.qkv_dense;
      qp.y.ld = g.qkv_w;
      qp.seq = cm.seq;
      qp.q_norm = L.q_norm;
      qp.k_norm = L.k_norm;
      qp.cos_t = W.cos_t;
      qp.sin_t = W.sin_t;
      qp.q = B.q;
      qp.kb = B.kb;
      qp.vb = B.vb;
      LK(qkv_post(qp, R, s));
    } else if (part) {
      // QKV partials, then per-head q/k RMSNorm + RoPE
      QkvPostArgs qp{};
      qp.g = g;
      int rc = project(B, W.map_qkv[l], ACT_H, R, g.qkv_w, g.H, nullptr, &qp.y, s);
      if (rc) return rc;
      qp.seq = cm.seq;
      qp.q_norm = L.q_norm;
      qp.k_norm = L.k_norm;
      qp.cos_t = W.cos_t;
      qp.sin_t = W.sin_t;
      qp.q = B.q;
      qp.kb = B.kb;
      qp.vb = B.vb;
      LK(qkv_post(qp, R, s));
    } else {
      // QKV with per-head q/k RMSNorm + RoPE fused in the epilogue
      GemmParams p{};
      p.m_act = R;
      p.n_w = g.qkv_w;
      p.k = g.H;
      p.epi = EPI_TC_QKV;
      p.ws = B.ws;
      p.counters = B.counters;
      p.status = B.status;
      p.fault_ns = B.fault_ns;
      p.seq = cm.seq;
      p.gamma = g.gamma;
      p.head_dim = g.d;
      p.q_rows = qd;
      p.k_rows = g.kv;
      p.q_norm = L.q_norm;
      p.k_norm = L.k_norm;
      p.cos_t = W.cos_t;
      p.sin_t = W.sin_t;
      p.eps = g.eps;
      p.q_out = B.q;
      p.k_out = B.kb;
      p.v_out = B.vb;
      LK(tc::gemm(W.map_qkv[l], B.act_map[ACT_H][bn_index(bnR)], bnR, p, s));
    }
    {
      AttnArgs a{};
      a.g = g;
      a.q = B.q;
      a.kb = B.kb;
      a.vb = B.vb;
      a.o = B.o;
      a.seq = cm.seq;
      a.page_ids = cm.page_ids;
      a.pool = W.pool;
      a.kv_scale = W.kv_scale;
      a.layer = l;
      a.scale = (float)(1.0 / std::sqrt((double)g.d));
      a.items = cm.items;
      a.n_items = cm.cap_items;
      a.pairs = cm.pairs;
      a.n_pairs = cm.cap_pairs;
      a.counts = cm.counts;
      a.ws = B.attn_ws;
      a.slot_floats = B.attn_slot_floats;
      a.status = B.status;
      a.cta_off = cm.cta_off;
      a.grid_tc = B.attn_grid_tc;
      if (B.attn_maps.ok) {
        LK(attention_tc(a, B.attn_maps, s));
        LK(attention_merge(a, s));
      } else {
        LK(attention_split(a, s));
      }
      if (cm.cap_pairs) count_launches(1);
    }
    // o_proj: residual added by the post-attention norm (or by the GEMM)
    has_pending = tc::partial_ok(R, g.H, qd);
    if (has_pending) {
      int rc = project(B, W.map_o[l], ACT_O, R, g.H, qd, nullptr, &pending, s);
      if (rc) return rc;
    } else {
      LK(tc_gemm(B, W.map_o[l], ACT_O, R, g.H, qd, EPI_TC_ADD_F32, B.x, g.H, s));
    }
    {
      AddNormArgs an{};
      an.x = B.x;
      an.has_y = has_pending;
      an.y = pending;
      an.g = L.post_norm;
      an.eps = g.eps;
      an.n = g.H;
      an.out = B.h;
      LK(add_norm(an, R, s));
    }
    {
      // gate/up with SwiGLU in the GEMM's epilogue: whole tiles for many rows
      // (and for few when the tiles cover half the SMs), otherwise the split-K
      // fixup (one kernel instead of partials plus a separate SwiGLU pass)
      GemmParams p{};
      p.m_act = R;
      p.n_w = 2 * g.I;
      p.k = g.H;
      p.epi = EPI_TC_SWIGLU;
      p.ws = B.ws;
      p.counters = B.counters;
      p.status = B.status;
      p.fault_ns = B.fault_ns;
      p.u_out = B.u;
      p.dp = dp || gu_dp_few;
      LK(tc::gemm(W.map_gu[l], B.act_map[ACT_H][bn_index(bn_gu)], bn_gu, p, s));
    }
    has_pending = tc::partial_ok(R, g.H, g.I);
    if (has_pending) {
      int rc = project(B, W.map_down[l], ACT_U, R, g.H, g.I, nullptr, &pending, s);
      if (rc) return rc;
    } else {
      LK(tc_gemm(B, W.map_down[l], ACT_U, R, g.H, g.I, EPI_TC_ADD_F32, B.x, g.H, s));
    }
  }
  {
    // last residual update, the final norm of the draft rows (and the taps)
    AddNormArgs an{};
    an.x = B.x;
    an.has_y = has_pending;
    an.y = pending;
    an.g = W.norm;
    an.eps = g.eps;
    an.n = g.H;
    an.out = nullptr;
    an.x_tap = B.tap_x ? B.tap_x + (size_t)g.L * R * g.H : nullptr;
    an.z_tap = B.tap_z;
    an.z = B.z;
    an.nd = nd;
    an.gamma = g.gamma;
    an.first = g.draft0;
    an.z16 = W.lm_lowp ? B.z16 : nullptr;
    LK(add_norm(an, R, s));
  }
  if (B.probe_begin && B.probe_end) FK(cudaEventRecordWithFlags(B.probe_begin, s, cudaEventRecordExternal));
  const int vt = (g.V + 127) / 128;
  if (W.lm_lowp && tc::lm_lowp_fits(D, g.H)) {
    // codes streamed and dequantised on chip (the draft rows resident),
    // per-row partials over 128-row vocab tiles
    GemmParams p{};
    p.m_act = D;
    p.n_w = g.V;
    p.k = g.H;
    p.tiles_m = vt;
    p.epi = EPI_TC_LMHEAD;
    p.wscale = W.lm_is_fp8 ? W.lm_scale : nullptr;
    p.gscale = W.lm_gscale;
    p.status = B.status;
    p.bitmask = bitmask;
    p.mask_words = (g.V + 31) / 32;
    p.nd = nd;
    p.lm_part = B.lm_part;
    LK(tc::lm_lowp(W.lm_lowp, W.map_lm_codes, W.map_lm_scales, B.act_map[ACT_Z16][bn_index(16)],
                   p, s));
    LK(lm_reduce(B.lm_part, D, vt, B.row_id, B.row_p1, s));
  } else if (D <= 64) {
    // Few draft rows: the vocab rows are the MMA's M (the weight stream
    // bounds the kernel), fused per-row reductions over 128-row vocab tiles.
    GemmParams p{};
    p.m_act = D;
    p.n_w = g.V;
    p.k = g.H;
    p.epi = EPI_TC_LMHEAD;
    p.wscale = W.lm_is_fp8 ? W.lm_scale : nullptr;
    p.gscale = W.lm_gscale;
    p.ws = B.ws;
    p.counters = B.counters;
    p.status = B.status;
    p.fault_ns = B.fault_ns;
    p.bitmask = bitmask;
    p.mask_words = (g.V + 31) / 32;
    p.nd = nd;
    p.lm_part = B.lm_part;
    const int bn = tc::pick_bn(D);
    LK(tc::gemm(W.map_lm, B.act_map[ACT_Z][bn_index(bn)], bn, p, s));
    LK(lm_reduce(B.lm_part, D, (g.V + 127) / 128, B.row_id, B.row_p1, s));
  } else {
    // Many draft rows: draft rows are the MMA's M, so each epilogue thread
    // reduces its own row over 256-row vocab tiles.
    LmArgs p{};
    p.m_act = D;
    p.n_w = g.V;
    p.k = g.H;
    p.bitmask = bitmask;
    p.mask_words = (g.V + 31) / 32;
    p.nd = nd;
    p.wscale = W.lm_is_fp8 ? W.lm_scale : nullptr;
    p.gscale = W.lm_gscale;
    p.out = B.lm_part;
    p.status = B.status;
    LK(tc::lmhead(B.act_map[ACT_Z][bn_index(128)], W.map_lm256, p, s));
    LK(lm_reduce(B.lm_part, D, tc::lmhead_vocab_tiles(g.V), B.row_id, B.row_p1, s));
  }
  if (B.probe_begin && B.probe_end) FK(cudaEventRecordWithFlags(B.probe_end, s, cudaEventRecordExternal));
  if (B.tap_logits) {
    GemmParams p{};
    p.m_act = D;
    p.n_w = g.V;
    p.k = g.H;
    p.epi = EPI_TC_STORE_F32;
    p.out = B.tap_logits;
    p.ldo = g.V;
    p.wscale = W.lm_is_fp8 ? W.lm_scale : nullptr;
    p.ws = B.ws;
    p.counters = B.counters;
    p.status = B.status;
    p.fault_ns = B.fault_ns;
    p.gscale = W.lm_gscale;
    if (W.lm_lowp && tc::lm_lowp_fits(D, g.H)) {
      p.tiles_m = vt;
      LK(tc::lm_lowp(W.lm_lowp, W.map_lm_codes, W.map_lm_scales,
                     B.act_map[ACT_Z16][bn_index(16)], p, s));
    } else {
      const int bn = tc::pick_bn(D);
      LK(tc::gemm(W.map_lm, B.act_map[ACT_Z][bn_index(bn)], bn, p, s));
    }
  }
  LK(finalize(B.row_id, B.row_p1, n, nd, B.status, (uint32_t *)(B.out_dev + B.off_drafts),
              (int32_t *)(B.out_dev + B.off_nout), (float *)(B.out_dev + B.off_conf),
              (int32_t *)B.out_dev, s));
  if (B.step_begin && B.step_end) FK(cudaEventRecordWithFlags(B.step_end, s, cudaEventRecordExternal));
  return DFLASH_OK;
}

cudaError_t gather_kv_rows(const Geo &g, const Weights &W, const Buffers &B, const RowMeta *rows,
                           int n, int layer, float *k_out, float *v_out, cudaStream_t s) {
  (void)B;
  return gather_kv(W.pool, g, layer, rows, n, W.kv_scale, k_out, v_out, s);
}

}  // namespace dfl

namespace dfl {

// Ctx items per SM the work split aims at: the persistent tensor-core kernel
// balances its items over its CTAs itself (three per SM keep the merge
// small); the split kernel launches one CTA per item, several resident per
// SM, where whole windows as items leave a tail wave that doubles the layer
// (measured at 128 sequences), so it gets finer items.
int attn_ctx_waves(int grid_tc) { return grid_tc > 0 ? 3 : 8; }

bool build_attn_work(const Geo &g, const std::vector<SeqMeta> &seq, int slot_cap, int grid_tc,
                     std::vector<AttnItem> *items, std::vector<AttnPair> *pairs,
                     std::vector<int32_t> *cta_off) {
  return build_attn_work_sms(g, seq, slot_cap, grid_tc, tc::num_sms(), items, pairs, cta_off);
}

bool build_attn_work_sms(const Geo &g, const std::vector<SeqMeta> &seq, int slot_cap,
                         int grid_tc, int sms, std::vector<AttnItem> *items,
                         std::vector<AttnPair> *pairs, std::vector<int32_t> *cta_off) {
  int64_t total = 0, longest = 0;
  for (const SeqMeta &m : seq) {
    total += (int64_t)(m.pos - m.ws) * g.nkv;
    longest = std::max<int64_t>(longest, (int64_t)(m.pos - m.ws) + m.ws % 64);
  }
  // About attn_ctx_waves SM waves of ctx items, at least 64 keys each so the
  // partial merge stays cheap. Chunk boundaries fall on positions that are
  // multiples of 64, so every tile but a window's first starts on a page.
  const int64_t parts = (int64_t)attn_ctx_waves(grid_tc) * sms;
  int64_t chunk = (total + parts - 1) / parts;
  chunk = std::max<int64_t>(64, (chunk + 63) / 64 * 64);
  for (;;) {
    items->clear();
    pairs->clear();
    int slots = 0;
    for (int s = 0; s < (int)seq.size(); ++s) {
      const int n_ctx = seq[s].pos - seq[s].ws;
      const int off = (int)(seq[s].ws % 64);
      const int nc = n_ctx > 0 ? (int)((n_ctx + off + chunk - 1) / chunk) : 0;
      for (int h = 0; h < g.nkv; ++h) {
        if (nc == 0) {
          items->push_back({s, h, 0, g.gamma, -1});
          continue;
        }
        pairs->push_back({s, h, slots, nc + 1});
        for (int c = 0; c < nc; ++c) {
          const int k0 = (int)std::max<int64_t>(0, c * chunk - off);
          const int k1 = (int)std::min<int64_t>(n_ctx, (c + 1) * chunk - off);
          items->push_back({s, h, k0, k1, slots++});
        }
        items->push_back({s, h, n_ctx, n_ctx + g.gamma, slots++});
      }
    }
    if (slots <= slot_cap) break;
    if (chunk >= longest) {   // one chunk per window already: the call does not fit
      items->clear();
      pairs->clear();
      cta_off->clear();
      return false;
    }
    chunk *= 2;
  }
  cta_off->clear();
  if (grid_tc <= 0) return true;
  // Longest first (a stable counting sort on the cost: key tiles + one for
  // the item's setup and output) onto the least-loaded CTA (ties: lowest
  // CTA), then the items regrouped CTA by CTA. Every buffer is reused.
  const int n = (int)items->size();
  thread_local std::vector<int> cost, order, owner, bucket;
  thread_local std::vector<int32_t> fill;
  thread_local std::vector<int64_t> heap;   // load << 16 | cta, a min-heap
  thread_local std::vector<AttnItem> regrouped;
  cost.resize(n);
  order.resize(n);
  owner.resize(n);
  int max_cost = 1;
  for (int i = 0; i < n; ++i) {
    cost[i] = attention_tc_tiles(g, seq[(*items)[i].s], (*items)[i]) + 1;
    max_cost = std::max(max_cost, cost[i]);
  }
  bucket.assign(max_cost + 2, 0);
  for (int i = 0; i < n; ++i) ++bucket[max_cost - cost[i] + 1];
  for (int c = 0; c <= max_cost; ++c) bucket[c + 1] += bucket[c];
  for (int i = 0; i < n; ++i) order[bucket[max_cost - cost[i]]++] = i;
  heap.resize(grid_tc);
  for (int b = 0; b < grid_tc; ++b) heap[b] = b;
  std::make_heap(heap.begin(), heap.end(), std::greater<int64_t>());
  cta_off->assign(grid_tc + 1, 0);
  for (int i : order) {
    std::pop_heap(heap.begin(), heap.end(), std::greater<int64_t>());
    int64_t &t = heap.back();
    const int b = (int)(t & 0xFFFF);
    owner[i] = b;
    ++(*cta_off)[b + 1];
    t += (int64_t)cost[i] << 16;
    std::push_heap(heap.begin(), heap.end(), std::greater<int64_t>());
  }
  for (int b = 0; b < grid_tc; ++b) (*cta_off)[b + 1] += (*cta_off)[b];
  regrouped.resize(n);
  fill.assign(cta_off->begin(), cta_off->end() - 1);
  for (int i : order) regrouped[fill[owner[i]]++] = (*items)[i];
  items->swap(regrouped);
  return true;
}

}  // namespace dfl
