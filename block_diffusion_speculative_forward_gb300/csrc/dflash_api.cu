// libdflash host side: the C ABI of include/dflash.h, the per-sequence state
// machine and page pool, and the orchestration of the propose forward's
// kernels on the caller's stream.
//
// Sources: [P1] "Struct BlockDiffusionDraftHead" (spark_model docs),
// [P2] "BlockDiffusionDraftHead" (metrale docs), [P3] "Trait DraftProposer".
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <string>
#include <vector>

#include "dflash.h"
#include "internal.h"
#include "forward.h"

using dfl::bf16;

namespace {
thread_local std::string g_err;

int fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

#define CK(call)                                                                     \
  do {                                                                               \
    cudaError_t e_ = (call);                                                         \
    if (e_ != cudaSuccess)                                                           \
      return fail(DFLASH_ECUDA, "%s: %s (%s:%d)", #call, cudaGetErrorString(e_),     \
                  __FILE__, __LINE__);                                               \
  } while (0)
}  // namespace

// ------------------------------------------------------------- page pool --
// Fixed pool of pages 0..n-1; a take returns the lowest free id.
struct PagePool {
  std::set<int32_t> free_ids;
  int32_t total = 0;
  void init(int32_t n) {
    total = n;
    free_ids.clear();
    for (int32_t i = 0; i < n; ++i) free_ids.insert(free_ids.end(), i);
  }
  int32_t take() {
    int32_t id = *free_ids.begin();
    free_ids.erase(free_ids.begin());
    return id;
  }
  void give(int32_t id) { free_ids.insert(id); }
  void take_id(int32_t id) { free_ids.erase(id); }
  int32_t n_free() const { return (int32_t)free_ids.size(); }
};

struct dflash_state {
  dflash_handle *owner = nullptr;
  int64_t cap = 0;                    // ctx positions the state may hold
  int64_t ctx_len = 0;                // target positions appended
  std::map<int64_t, int32_t> pages;   // logical page -> physical page
  bool pending = false;               // a propose awaits after_verify
  int64_t pend_pos = 0;
  int32_t pend_nout = 0;
  int64_t expected_next = -1;
};

struct dflash_handle {
  dflash_config cfg{};
  dfl::Geo g{};
  bool compute = false;
  dfl::Weights w{};
  dfl::Buffers b{};
  std::vector<void *> allocs;        // device allocations, freed at destroy
  std::vector<void *> host_allocs;   // pinned host allocations
  PagePool pool;
  std::mutex mu;
  std::set<dflash_state *> states;
  // pages taken out of their states (take_drafter_kv) and neither installed
  // nor freed yet: first page id -> (the bundle's pages, its ctx length)
  std::map<int32_t, std::pair<std::vector<int32_t>, int64_t>> carried;
  int R_max = 0, D_max = 0, M_ctx = 0;
  // per-call metadata staging
  char *meta_host = nullptr, *meta_dev = nullptr;
  size_t meta_cap = 0;
  cudaEvent_t meta_ev = nullptr;
  bool meta_ev_live = false;
  // fixed sections of the metadata buffer (rows follow them)
  int cap_seq = 0, cap_pages = 0, cap_items = 0, cap_pairs = 0;
  size_t off_seq = 0, off_pages = 0, off_items = 0, off_pairs = 0, off_sched = 0, off_rows = 0;
  int cap_sched = 0;
  int cap_citems = 0;
  size_t off_citems = 0;
  bool chain_ok = false;    // the head can take the chained few-row path
  int last_chained = 0;     // the last propose took it
  // captured propose graphs, keyed by the call's launch shape
  bool use_graphs = true;
  cudaStream_t cap_stream = nullptr;
  std::map<std::vector<uintptr_t>, std::pair<cudaGraphExec_t, int64_t>> graphs;
};

// ------------------------------------------------------------ helpers --
namespace {

int64_t window_start(const dflash_handle *h, int64_t end) {
  int64_t W = h->cfg.ctx_window;
  return W > 0 ? std::max<int64_t>(0, end - W) : end;
}

struct AppendPlan {
  dflash_state *st;
  int64_t old_len, new_len, lo, ws;
  std::vector<int64_t> retire, need;
  const bf16 *src;  // the caller's rows for positions old_len..new_len-1
};

// Which rows a ctx append stores and which pages it retires and takes: rows
// below new_len - ctx_window are skipped; pages wholly below the window
// start retire; a page is taken when a row first lands in it.
AppendPlan plan_append(const dflash_handle *h, dflash_state *st, int64_t n, const void *src) {
  AppendPlan p;
  p.st = st;
  p.old_len = st->ctx_len;
  p.new_len = st->ctx_len + n;
  p.ws = window_start(h, p.new_len);
  p.lo = h->cfg.ctx_window > 0 ? std::max(p.old_len, p.ws) : p.new_len;
  p.src = (const bf16 *)src;
  const int64_t B = h->cfg.kv_block;
  // the pages map is ordered by logical page: the retiring ones are a prefix
  for (auto &kv : st->pages) {
    if ((kv.first + 1) * B > p.ws) break;
    p.retire.push_back(kv.first);
  }
  if (p.lo < p.new_len)
    for (int64_t b = p.lo / B; b <= (p.new_len - 1) / B; ++b)
      if (!st->pages.count(b)) p.need.push_back(b);
  return p;
}

// All plans retire first, then take pages, in order; the caller has checked
// that the pool can cover every take.
void commit_plans(dflash_handle *h, std::vector<AppendPlan> &plans) {
  for (auto &p : plans)
    for (int64_t b : p.retire) {
      h->pool.give(p.st->pages[b]);
      p.st->pages.erase(b);
    }
  for (auto &p : plans)
    for (int64_t b : p.need) p.st->pages[b] = h->pool.take();
}

bool pool_can_cover(const dflash_handle *h, const std::vector<AppendPlan> &plans) {
  int64_t need = 0, retire = 0;
  for (auto &p : plans) {
    need += (int64_t)p.need.size();
    retire += (int64_t)p.retire.size();
  }
  return need <= h->pool.n_free() + retire;
}

void retire_below(dflash_handle *h, dflash_state *st, int64_t ws) {
  const int64_t B = h->cfg.kv_block;
  // ordered by logical page: stop at the first page that stays
  for (auto it = st->pages.begin(); it != st->pages.end() && (it->first + 1) * B <= ws;) {
    h->pool.give(it->second);
    it = st->pages.erase(it);
  }
}

// The host state of the states a call touches, taken before it commits
// anything: a call that fails after its commit (a CUDA error, or a device
// status word raised by its kernels) puts every state and the pool back.
struct Snapshot {
  struct One {
    dflash_state *st;
    int64_t ctx_len;
    std::map<int64_t, int32_t> pages;
    bool pending;
    int64_t pend_pos;
    int32_t pend_nout;
    int64_t expected_next;
  };
  std::vector<One> states;
};

Snapshot snapshot(dflash_state *const *states, int n) {
  Snapshot s;
  for (int i = 0; i < n; ++i) {
    dflash_state *st = states[i];
    s.states.push_back({st, st->ctx_len, st->pages, st->pending, st->pend_pos, st->pend_nout,
                        st->expected_next});
  }
  return s;
}

void rollback(dflash_handle *h, const Snapshot &snap) {
  std::set<int32_t> now, then;
  for (const auto &o : snap.states) {
    for (auto &kv : o.st->pages) now.insert(kv.second);
    for (auto &kv : o.pages) then.insert(kv.second);
  }
  for (int32_t id : now)
    if (!then.count(id)) h->pool.give(id);       // taken by the failed call
  for (int32_t id : then)
    if (!now.count(id)) h->pool.take_id(id);     // retired by it
  for (const auto &o : snap.states) {
    o.st->ctx_len = o.ctx_len;
    o.st->pages = o.pages;
    o.st->pending = o.pending;
    o.st->pend_pos = o.pend_pos;
    o.st->pend_nout = o.pend_nout;
    o.st->expected_next = o.expected_next;
  }
}

template <class T>
T *dev_alloc(dflash_handle *h, size_t count, cudaError_t *err) {
  void *p = nullptr;
  if (count == 0) return nullptr;
  cudaError_t e = cudaMalloc(&p, count * sizeof(T));
  if (e != cudaSuccess) {
    *err = e;
    return nullptr;
  }
  h->allocs.push_back(p);
  return (T *)p;
}

void drop_graphs(dflash_handle *h) {
  for (auto &kv : h->graphs) cudaGraphExecDestroy(kv.second.first);
  h->graphs.clear();
}

void release(dflash_handle *h) {
  drop_graphs(h);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  for (auto *st : h->states) delete st;
  h->states.clear();
  if (h->meta_ev) cudaEventDestroy(h->meta_ev);
  for (void *p : h->allocs) cudaFree(p);
  for (void *p : h->host_allocs) cudaFreeHost(p);
  h->allocs.clear();
  h->host_allocs.clear();
}

int validate_config(const dflash_config *c) {
  if (!c) return fail(DFLASH_EINVAL, "config is NULL");
  if (c->num_layers < 1 || c->hidden < 64 || c->hidden % 64 || c->hidden > 4096)
    return fail(DFLASH_EINVAL, "num_layers >= 1 and hidden a multiple of 64, at most 4096");
  if (c->intermediate < 64 || c->intermediate % 64)
    return fail(DFLASH_EINVAL, "intermediate must be a positive multiple of 64");
  if (c->head_dim != 64 && c->head_dim != 128) return fail(DFLASH_EINVAL, "head_dim must be 64 or 128");
  if (c->num_q_heads < 1 || c->num_kv_heads < 1 || c->num_q_heads % c->num_kv_heads ||
      c->num_kv_heads > 32)
    return fail(DFLASH_EINVAL, "num_q_heads must be a multiple of num_kv_heads (<= 32)");
  if ((c->num_q_heads * c->head_dim) % 128 || (c->num_kv_heads * c->head_dim) % 128)
    return fail(DFLASH_EINVAL, "num_q_heads*head_dim and num_kv_heads*head_dim must be multiples of 128");
  if (c->vocab < 2 || c->gamma < 2 || c->gamma > 64)
    return fail(DFLASH_EINVAL, "vocab >= 2 and 2 <= gamma <= 64 required");
  if (c->mask_token_id >= (uint32_t)c->vocab) return fail(DFLASH_EINVAL, "mask_token_id >= vocab");
  if (c->n_target_layers < 1 || c->target_hidden < 1)
    return fail(DFLASH_EINVAL, "n_target_layers and target_hidden must be positive");
  if ((int64_t)c->fc_in_features != (int64_t)c->n_target_layers * c->target_hidden)
    return fail(DFLASH_EINVAL,
                "fc input width %d != n_target_layers*target_hidden %lld (validate_against_target)",
                c->fc_in_features, (long long)c->n_target_layers * c->target_hidden);
  if (c->fc_in_features % 64) return fail(DFLASH_EINVAL, "fc input width must be a multiple of 64");
  if (!(c->rms_eps >= 0.f)) return fail(DFLASH_EINVAL, "rms_eps must be >= 0");
  if (c->ctx_window < 0 || c->kv_block < 1 || c->kv_block > 256 || c->prefill_chunk < 1)
    return fail(DFLASH_EINVAL, "ctx_window >= 0, 1 <= kv_block <= 256, prefill_chunk >= 1 required");
  if (c->max_batch < 1 || c->max_seq_len < 1 || c->kv_pool_blocks < 0)
    return fail(DFLASH_EINVAL, "max_batch, max_seq_len >= 1 and kv_pool_blocks >= 0 required");
  if (c->shifted_rows != 0 && c->shifted_rows != 1)
    return fail(DFLASH_EINVAL, "shifted_rows must be 0 or 1");
  if ((c->kv_dtype != 0 && c->kv_dtype != 1) || c->lm_head_dtype < 0 || c->lm_head_dtype > 2)
    return fail(DFLASH_EINVAL, "kv_dtype must be 0 or 1 and lm_head_dtype 0, 1 or 2");
  if (c->lm_head_dtype != 0 && c->hidden % 256)
    return fail(DFLASH_EINVAL, "a streamed FP8 or NVFP4 lm_head needs hidden a multiple of 256");
  if (!(c->rope_attn_factor >= 0.f && c->rope_attn_factor < 1e4f))
    return fail(DFLASH_EINVAL, "rope_attn_factor must be 0 (none) or positive");
  return DFLASH_OK;
}

int32_t pool_pages_for(const dflash_config *c) {
  if (c->kv_pool_blocks > 0) return c->kv_pool_blocks;
  if (c->ctx_window == 0) return 0;
  int64_t span = std::min<int64_t>(c->ctx_window, c->max_seq_len);
  return (int32_t)(c->max_batch * (span / c->kv_block + 2));
}

// Stage the call's metadata (seq, rows, page ids) and copy it to the device
// in one transfer. Waits first for the previous transfer out of the staging
// buffer to finish.
// Stage the call's metadata and copy it to the device in one transfer. The
// sections sit at offsets fixed per handle ([counts][seq][page ids][items]
// [pairs][rows...]), so kernels captured in a graph keep valid pointers
// across calls. Waits first for the previous transfer out of the staging
// buffer to finish.
int upload_meta(dflash_handle *h, const std::vector<dfl::SeqMeta> &seq,
                const std::vector<dfl::RowMeta> &rows, const std::vector<int32_t> &page_ids,
                cudaStream_t s, dfl::CallMeta *out,
                const std::vector<dfl::AttnItem> &items = {},
                const std::vector<dfl::AttnPair> &pairs = {},
                const std::vector<int32_t> &cta_off = {}, size_t *defer_bytes = nullptr,
                const std::vector<dfl::ChainAttnItem> &citems = {}) {
  if ((int)seq.size() > h->cap_seq || (int)page_ids.size() > h->cap_pages ||
      (int)items.size() > h->cap_items || (int)pairs.size() > h->cap_pairs ||
      (int)cta_off.size() > h->cap_sched || (int)citems.size() > h->cap_citems)
    return fail(DFLASH_EINVAL, "internal: call metadata beyond the handle's capacity");
  size_t total = h->off_rows + rows.size() * sizeof(dfl::RowMeta) + 16;
  if (h->meta_ev_live) {
    CK(cudaEventSynchronize(h->meta_ev));
    h->meta_ev_live = false;
  }
  if (total > h->meta_cap) {
    CK(cudaStreamSynchronize(s));
    size_t cap = std::max(total, h->meta_cap * 2);
    void *hp = nullptr, *dp = nullptr;
    CK(cudaMallocHost(&hp, cap));
    cudaError_t e = cudaMalloc(&dp, cap);
    if (e != cudaSuccess) {
      cudaFreeHost(hp);
      CK(e);
    }
    if (h->meta_host) {
      cudaFreeHost(h->meta_host);
      cudaFree(h->meta_dev);
      h->host_allocs.erase(std::find(h->host_allocs.begin(), h->host_allocs.end(), h->meta_host));
      h->allocs.erase(std::find(h->allocs.begin(), h->allocs.end(), h->meta_dev));
    }
    h->meta_host = (char *)hp;
    h->meta_dev = (char *)dp;
    h->host_allocs.push_back(hp);
    h->allocs.push_back(dp);
    h->meta_cap = cap;
    drop_graphs(h);   // captured kernels point into the old buffer
  }
  int32_t *counts = (int32_t *)h->meta_host;
  counts[0] = (int32_t)items.size();
  counts[1] = (int32_t)pairs.size();
  counts[2] = (int32_t)citems.size();
  if (!citems.empty())
    memcpy(h->meta_host + h->off_citems, citems.data(), citems.size() * sizeof(dfl::ChainAttnItem));
  if (!seq.empty()) memcpy(h->meta_host + h->off_seq, seq.data(), seq.size() * sizeof(dfl::SeqMeta));
  if (!page_ids.empty())
    memcpy(h->meta_host + h->off_pages, page_ids.data(), page_ids.size() * sizeof(int32_t));
  if (!items.empty())
    memcpy(h->meta_host + h->off_items, items.data(), items.size() * sizeof(dfl::AttnItem));
  if (!pairs.empty())
    memcpy(h->meta_host + h->off_pairs, pairs.data(), pairs.size() * sizeof(dfl::AttnPair));
  if (!cta_off.empty())
    memcpy(h->meta_host + h->off_sched, cta_off.data(), cta_off.size() * sizeof(int32_t));
  if (!rows.empty())
    memcpy(h->meta_host + h->off_rows, rows.data(), rows.size() * sizeof(dfl::RowMeta));
  if (defer_bytes) {
    *defer_bytes = total;   // the caller's graph (or its own copy) moves it
  } else {
    CK(cudaMemcpyAsync(h->meta_dev, h->meta_host, total, cudaMemcpyHostToDevice, s));
    CK(cudaEventRecord(h->meta_ev, s));
    h->meta_ev_live = true;
  }
  out->counts = (const int *)h->meta_dev;
  out->seq = (const dfl::SeqMeta *)(h->meta_dev + h->off_seq);
  out->rows = (const dfl::RowMeta *)(h->meta_dev + h->off_rows);
  out->page_ids = (const int32_t *)(h->meta_dev + h->off_pages);
  out->items = (const dfl::AttnItem *)(h->meta_dev + h->off_items);
  out->pairs = (const dfl::AttnPair *)(h->meta_dev + h->off_pairs);
  out->cta_off = (const int32_t *)(h->meta_dev + h->off_sched);
  out->citems = (const dfl::ChainAttnItem *)(h->meta_dev + h->off_citems);
  out->n_seq = (int)seq.size();
  out->n_rows = (int)rows.size();
  out->n_items = (int)items.size();
  out->n_pairs = (int)pairs.size();
  out->cap_items = h->cap_items;
  out->cap_pairs = h->cap_pairs;
  return DFLASH_OK;
}

// Row metadata of every stored ctx row of the plans, in plan order.
void rows_of(const dflash_handle *h, const std::vector<AppendPlan> &plans,
             std::vector<dfl::RowMeta> *rows) {
  const int64_t B = h->cfg.kv_block, S = h->g.S;
  for (size_t i = 0; i < plans.size(); ++i) {
    const AppendPlan &p = plans[i];
    for (int64_t j = p.lo; j < p.new_len; ++j) {
      dfl::RowMeta r;
      r.pos = (int32_t)j;
      auto it = p.st->pages.find(j / B);
      r.page = it == p.st->pages.end() ? -1 : it->second;  // -1 trips the kernel's page check
      r.slot = (int32_t)(j % B);
      r.seq = (int32_t)i;
      r.src = p.src + (j - p.old_len) * S;
      rows->push_back(r);
    }
  }
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

}  // namespace

// ================================================================ the ABI ==
extern "C" {

const char *dflash_last_error(void) { return g_err.c_str(); }

int dflash_create(const dflash_config *cfg, const dflash_weights *wts, dflash_handle **out) {
  if (!out) return fail(DFLASH_EINVAL, "out is NULL");
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc) return rc;
  dflash_handle *h = new dflash_handle();
  h->cfg = *cfg;
  dfl::Geo &g = h->g;
  g.L = cfg->num_layers;
  g.H = cfg->hidden;
  g.I = cfg->intermediate;
  g.nq = cfg->num_q_heads;
  g.nkv = cfg->num_kv_heads;
  g.d = cfg->head_dim;
  g.V = cfg->vocab;
  g.gamma = cfg->gamma;
  g.B = cfg->kv_block;
  g.S = cfg->fc_in_features;
  g.kv = g.nkv * g.d;
  g.qkv_w = g.nq * g.d + 2 * g.kv;
  g.kv_fp8 = cfg->kv_dtype;
  g.eps = cfg->rms_eps;
  g.draft0 = cfg->shifted_rows ? 0 : 1;
  g.pages = pool_pages_for(cfg);
  h->pool.init(g.pages);
  h->R_max = cfg->max_batch * g.gamma;
  h->D_max = cfg->max_batch * (g.gamma - 1);
  h->M_ctx = std::max(cfg->prefill_chunk, h->R_max);
  h->compute = wts != nullptr;
  {
    // fixed metadata sections: sequences, window page ids, attention work
    const int64_t span = cfg->ctx_window > 0 ? std::min<int64_t>(cfg->ctx_window, cfg->max_seq_len) : 0;
    h->cap_seq = cfg->max_batch;
    h->cap_pages = (int)(cfg->max_batch * (span / cfg->kv_block + 2));
    h->cap_pairs = cfg->max_batch * g.nkv;
    auto al = [](size_t x) { return (x + 15) & ~(size_t)15; };
    h->off_seq = 16;
    h->off_pages = al(h->off_seq + sizeof(dfl::SeqMeta) * h->cap_seq);
    h->off_items = al(h->off_pages + sizeof(int32_t) * h->cap_pages);
  }
  if (!h->compute) {
    *out = h;
    return DFLASH_OK;
  }
  rc = dfl::build_device_side(h->cfg, h->g, wts, h->R_max, h->D_max, h->M_ctx, &h->w, &h->b,
                              &h->allocs, &h->host_allocs);
  if (rc == DFLASH_OK) {
    cudaError_t e = cudaEventCreateWithFlags(&h->meta_ev, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) rc = fail(DFLASH_ECUDA, "cudaEventCreate: %s", cudaGetErrorString(e));
  } else {
    g_err = dfl::last_build_error();
  }
  if (rc != DFLASH_OK) {
    release(h);
    delete h;
    return rc;
  }
  h->chain_ok = h->b.use_chain;
  // the chained launch is opt-in: at the shipped drafter geometry it ran
  // slower than the kernel-per-step path (its cross-CTA hand-offs between
  // phases are L2 round trips taken while every other SM streams weights)
  h->b.use_chain = false;
  h->cap_items = h->b.attn_slots + h->cap_pairs;
  h->off_pairs = (h->off_items + sizeof(dfl::AttnItem) * h->cap_items + 15) & ~(size_t)15;
  h->cap_sched = h->b.attn_grid_tc + 1;
  h->off_sched = (h->off_pairs + sizeof(dfl::AttnPair) * h->cap_pairs + 15) & ~(size_t)15;
  h->cap_citems = dfl::chain_attn_capacity(h->g);
  h->off_citems = (h->off_sched + sizeof(int32_t) * h->cap_sched + 15) & ~(size_t)15;
  h->off_rows = (h->off_citems + sizeof(dfl::ChainAttnItem) * h->cap_citems + 15) & ~(size_t)15;
  *out = h;
  return DFLASH_OK;
}

void dflash_destroy(dflash_handle *h) {
  if (!h) return;
  if (h->compute) cudaDeviceSynchronize();
  release(h);
  delete h;
}

int dflash_propose_batch_max(const dflash_handle *h) { return h ? h->cfg.max_batch : DFLASH_EINVAL; }
int dflash_block_gamma(const dflash_handle *h) { return h ? h->cfg.gamma : DFLASH_EINVAL; }

int dflash_alloc_state(dflash_handle *h, int64_t budget_tokens, dflash_state **out) {
  if (!h || !out) return fail(DFLASH_EINVAL, "NULL argument");
  if (budget_tokens <= 0) return fail(DFLASH_EINVAL, "budget_tokens must be positive");
  std::lock_guard<std::mutex> lk(h->mu);
  dflash_state *st = new dflash_state();
  st->owner = h;
  st->cap = std::min<int64_t>(budget_tokens, h->cfg.max_seq_len);
  h->states.insert(st);
  *out = st;
  return DFLASH_OK;
}

int dflash_free_state(dflash_handle *h, dflash_state *st) {
  if (!h || !st) return fail(DFLASH_EINVAL, "NULL argument");
  std::lock_guard<std::mutex> lk(h->mu);
  if (!h->states.count(st)) return fail(DFLASH_EINVAL, "state does not belong to this handle");
  for (auto &kv : st->pages) h->pool.give(kv.second);
  h->states.erase(st);
  delete st;
  return DFLASH_OK;
}

int dflash_prefill(dflash_handle *h, dflash_state *st, const void *stack, int32_t n_rows,
                   void *stream) {
  if (!h || !st) return fail(DFLASH_EINVAL, "NULL argument");
  cudaStream_t s = (cudaStream_t)stream;
  std::lock_guard<std::mutex> lk(h->mu);
  if (!h->states.count(st)) return fail(DFLASH_EINVAL, "state does not belong to this handle");
  if (n_rows < 0) return fail(DFLASH_EINVAL, "n_rows < 0");
  if (st->pending) return fail(DFLASH_ESTATE, "prefill while a propose awaits after_verify");
  if (st->ctx_len + n_rows > st->cap) return fail(DFLASH_EINVAL, "ctx beyond the state's budget");
  if (h->compute && n_rows > 0 && (!stack || !aligned16(stack)))
    return fail(DFLASH_EINVAL, "stack must be a 16-byte aligned device pointer");
  std::vector<AppendPlan> plans{plan_append(h, st, n_rows, stack)};
  if (!pool_can_cover(h, plans)) return fail(DFLASH_ENOMEM, "KV pool exhausted");
  const Snapshot snap = snapshot(&st, 1);
  commit_plans(h, plans);
  st->ctx_len = plans[0].new_len;
  if (!h->compute) return DFLASH_BOOKKEEPING_ONLY;
  std::vector<dfl::RowMeta> rows;
  rows_of(h, plans, &rows);
  for (size_t a = 0; a < rows.size(); a += (size_t)h->cfg.prefill_chunk) {
    size_t nb = std::min(rows.size() - a, (size_t)h->cfg.prefill_chunk);
    std::vector<dfl::RowMeta> chunk(rows.begin() + a, rows.begin() + a + nb);
    dfl::CallMeta cm;
    int rc = upload_meta(h, {}, chunk, {}, s, &cm);
    if (rc == DFLASH_OK) {
      rc = dfl::ctx_append(h->g, h->w, h->b, cm.rows, cm.n_rows, h->M_ctx, s);
      if (rc) fail(rc, "%s", dfl::last_build_error());
    }
    if (rc) {
      rollback(h, snap);   // no state claims rows that were never written
      return rc;
    }
  }
  return DFLASH_OK;
}

int dflash_propose_batch(dflash_handle *h, int32_t n, dflash_state *const *states,
                         const uint32_t *last_tokens, const int64_t *positions,
                         const void *const *new_rows, const int32_t *n_new, int32_t num_drafts,
                         const int32_t *bitmask, uint32_t *drafts, int32_t *n_out, float *conf,
                         void *stream);

int dflash_propose(dflash_handle *h, dflash_state *st, uint32_t last_token, int64_t position,
                   const void *new_rows, int32_t n_new, int32_t num_drafts, const int32_t *bitmask,
                   uint32_t *drafts, int32_t *n_out, float *conf, void *stream) {
  return dfl::propose_impl(h, 1, &st, &last_token, &position, &new_rows, &n_new, num_drafts,
                           bitmask, drafts, n_out, conf, stream);
}

int dflash_propose_batch(dflash_handle *h, int32_t n, dflash_state *const *states,
                         const uint32_t *last_tokens, const int64_t *positions,
                         const void *const *new_rows, const int32_t *n_new, int32_t num_drafts,
                         const int32_t *bitmask, uint32_t *drafts, int32_t *n_out, float *conf,
                         void *stream) {
  if (!h) return fail(DFLASH_EINVAL, "NULL handle");
  if (n < 2 || n > h->cfg.max_batch) return DFLASH_DECLINED;
  return dfl::propose_impl(h, n, states, last_tokens, positions, new_rows, n_new, num_drafts,
                           bitmask, drafts, n_out, conf, stream);
}

int dflash_after_verify(dflash_handle *h, dflash_state *st, int32_t num_accepted) {
  if (!h || !st) return fail(DFLASH_EINVAL, "NULL argument");
  std::lock_guard<std::mutex> lk(h->mu);
  if (!h->states.count(st)) return fail(DFLASH_EINVAL, "state does not belong to this handle");
  if (!st->pending) return fail(DFLASH_ESTATE, "after_verify without a propose");
  if (num_accepted < 0 || num_accepted > st->pend_nout)
    return fail(DFLASH_EINVAL, "num_accepted %d outside 0..%d", num_accepted, st->pend_nout);
  st->expected_next = st->pend_pos + num_accepted + 1;
  st->pending = false;
  retire_below(h, st, window_start(h, st->expected_next));
  return DFLASH_OK;
}

int dflash_after_verify_batch(dflash_handle *h, int32_t n, dflash_state *const *states,
                              const int32_t *num_accepted) {
  if (!h || n < 0 || (n > 0 && (!states || !num_accepted)))
    return fail(DFLASH_EINVAL, "NULL argument");
  std::lock_guard<std::mutex> lk(h->mu);
  std::set<dflash_state *> seen;
  for (int i = 0; i < n; ++i) {
    dflash_state *st = states[i];
    if (!st || !h->states.count(st)) return fail(DFLASH_EINVAL, "state %d unknown", i);
    if (!seen.insert(st).second) return fail(DFLASH_EINVAL, "state %d repeated", i);
    if (!st->pending) return fail(DFLASH_ESTATE, "state %d: after_verify without a propose", i);
    if (num_accepted[i] < 0 || num_accepted[i] > st->pend_nout)
      return fail(DFLASH_EINVAL, "state %d: num_accepted %d outside 0..%d", i, num_accepted[i],
                  st->pend_nout);
  }
  for (int i = 0; i < n; ++i) {
    dflash_state *st = states[i];
    st->expected_next = st->pend_pos + num_accepted[i] + 1;
    st->pending = false;
    retire_below(h, st, window_start(h, st->expected_next));
  }
  return DFLASH_OK;
}

int dflash_catchup_batch(dflash_handle *h, int32_t n, dflash_state *const *states,
                         const uint32_t *const *tokens, const void *const *rows,
                         const int32_t *n_rows, const int64_t *first_pos, int64_t *written,
                         void *stream) {
  if (written) *written = 0;
  if (!h || n < 0 || (n > 0 && (!states || !rows || !n_rows || !first_pos)))
    return fail(DFLASH_EINVAL, "NULL argument");
  cudaStream_t s = (cudaStream_t)stream;
  std::lock_guard<std::mutex> lk(h->mu);
  std::set<dflash_state *> seen;
  int64_t total = 0;
  for (int i = 0; i < n; ++i) {
    dflash_state *st = states[i];
    const int32_t m = n_rows[i];
    if (!st || !h->states.count(st)) return fail(DFLASH_EINVAL, "state %d unknown", i);
    if (!seen.insert(st).second) return fail(DFLASH_EINVAL, "state %d repeated", i);
    if (m < 0) return fail(DFLASH_EINVAL, "state %d: n_rows < 0", i);
    if (st->pending) return fail(DFLASH_ESTATE, "state %d: catch-up while a propose awaits after_verify", i);
    if (tokens && tokens[i])
      for (int32_t r = 0; r < m; ++r)
        if (tokens[i][r] >= (uint32_t)h->cfg.vocab)
          return fail(DFLASH_EINVAL, "state %d: token %d outside the vocab", i, r);
    if (first_pos[i] != st->ctx_len)
      return fail(DFLASH_EPOSITION, "state %d: first position %lld != its append point %lld", i,
                  (long long)first_pos[i], (long long)st->ctx_len);
    if (st->expected_next >= 0 && st->ctx_len + m > st->expected_next)
      return fail(DFLASH_EPOSITION, "state %d: rows past the position after_verify set (%lld)", i,
                  (long long)st->expected_next);
    if (st->ctx_len + m > st->cap) return fail(DFLASH_EINVAL, "state %d: ctx beyond its budget", i);
    if (h->compute && m > 0 && (!rows[i] || !aligned16(rows[i])))
      return fail(DFLASH_EINVAL, "state %d: rows must be a 16-byte aligned device pointer", i);
    total += m;
  }
  std::vector<AppendPlan> plans;
  for (int i = 0; i < n; ++i) plans.push_back(plan_append(h, states[i], n_rows[i], rows[i]));
  if (!pool_can_cover(h, plans)) return fail(DFLASH_ENOMEM, "KV pool exhausted");
  const Snapshot snap = snapshot(states, n);
  commit_plans(h, plans);
  for (auto &p : plans) p.st->ctx_len = p.new_len;
  if (written) *written = total;
  if (!h->compute) return DFLASH_BOOKKEEPING_ONLY;
  // the rows sit at their states' append points, so the row metadata of an
  // append (position j at slot j) carries the explicit positions as they are
  std::vector<dfl::RowMeta> meta;
  rows_of(h, plans, &meta);
  for (size_t a = 0; a < meta.size(); a += (size_t)h->cfg.prefill_chunk) {
    size_t nb = std::min(meta.size() - a, (size_t)h->cfg.prefill_chunk);
    std::vector<dfl::RowMeta> chunk(meta.begin() + a, meta.begin() + a + nb);
    dfl::CallMeta cm;
    int rc = upload_meta(h, {}, chunk, {}, s, &cm);
    if (rc == DFLASH_OK) {
      rc = dfl::ctx_append(h->g, h->w, h->b, cm.rows, cm.n_rows, h->M_ctx, s);
      if (rc) fail(rc, "%s", dfl::last_build_error());
    }
    if (rc) {
      rollback(h, snap);
      if (written) *written = 0;
      return rc;
    }
  }
  return DFLASH_OK;
}

int dflash_yarn_inv_freq(double theta, int32_t head_dim, double factor, double beta_fast,
                         double beta_slow, int32_t original_max_pos, float *inv_freq,
                         float *attn_factor) {
  if (!inv_freq || !(theta > 1.0) || head_dim < 2 || head_dim % 2 || !(factor >= 1.0) ||
      !(beta_slow > 0.0) || !(beta_fast > beta_slow) || original_max_pos < 1)
    return fail(DFLASH_EINVAL, "bad YaRN parameters");
  const int half = head_dim / 2;
  const double two_pi = 6.283185307179586476925286766559;
  // the real pair index whose frequency turns r times over the original context
  auto pair_turning = [&](double r) {
    return head_dim * std::log(original_max_pos / (r * two_pi)) / (2.0 * std::log(theta));
  };
  const double lo = std::max(std::floor(pair_turning(beta_fast)), 0.0);
  const double hi = std::min(std::ceil(pair_turning(beta_slow)), (double)(half - 1));
  for (int i = 0; i < half; ++i) {
    const double base = std::pow(theta, -2.0 * i / head_dim);
    const double ramp = std::min(std::max((i - lo) / std::max(hi - lo, 1e-3), 0.0), 1.0);
    inv_freq[i] = (float)(base * (1.0 - ramp) + (base / factor) * ramp);
  }
  if (attn_factor) *attn_factor = factor <= 1.0 ? 1.f : (float)(0.1 * std::log(factor) + 1.0);
  return DFLASH_OK;
}

int dflash_take_drafter_kv(dflash_handle *h, dflash_state *st, int32_t *blocks, int32_t cap,
                           int32_t *n_blocks, int64_t *rows) {
  if (!h || !st || !n_blocks || !rows || cap < 0 || (cap > 0 && !blocks))
    return fail(DFLASH_EINVAL, "NULL argument");
  std::lock_guard<std::mutex> lk(h->mu);
  if (!h->states.count(st)) return fail(DFLASH_EINVAL, "state does not belong to this handle");
  if (st->pending) return fail(DFLASH_ESTATE, "take_drafter_kv while a propose awaits after_verify");
  if (st->pages.empty()) return DFLASH_DECLINED;
  if ((int64_t)st->pages.size() > cap)
    return fail(DFLASH_EINVAL, "%zu pages to carry, room for %d", st->pages.size(), cap);
  // the live pages are consecutive logical pages: retirement removes from below
  if (st->pages.rbegin()->first - st->pages.begin()->first + 1 != (int64_t)st->pages.size())
    return fail(DFLASH_ESTATE, "internal: live pages are not consecutive");
  std::vector<int32_t> ids;
  for (auto &kv : st->pages) ids.push_back(kv.second);
  std::copy(ids.begin(), ids.end(), blocks);
  *n_blocks = (int32_t)ids.size();
  *rows = st->ctx_len;
  h->carried[ids.front()] = std::make_pair(ids, st->ctx_len);
  st->pages.clear();
  st->ctx_len = 0;
  st->pending = false;
  st->expected_next = -1;
  return DFLASH_OK;
}

int dflash_install_drafter_kv(dflash_handle *h, dflash_state *st, const int32_t *blocks,
                              int32_t n_blocks, int64_t rows) {
  if (!h || !st || !blocks || n_blocks < 1) return fail(DFLASH_EINVAL, "NULL argument");
  std::lock_guard<std::mutex> lk(h->mu);
  if (!h->states.count(st)) return fail(DFLASH_EINVAL, "state does not belong to this handle");
  auto it = h->carried.find(blocks[0]);
  if (it == h->carried.end() || it->second.second != rows ||
      it->second.first != std::vector<int32_t>(blocks, blocks + n_blocks))
    return fail(DFLASH_EINVAL, "pages and rows are not a bundle taken by take_drafter_kv");
  if (st->ctx_len != 0 || !st->pages.empty() || st->pending || st->expected_next >= 0)
    return fail(DFLASH_EINVAL, "install_drafter_kv into a state that is not fresh");
  if (rows > st->cap) return fail(DFLASH_EINVAL, "rows %lld beyond the state's budget", (long long)rows);
  const int64_t B = h->cfg.kv_block;
  const int64_t b0 = (rows + B - 1) / B - n_blocks;
  for (int32_t i = 0; i < n_blocks; ++i) st->pages[b0 + i] = blocks[i];
  st->ctx_len = rows;
  h->carried.erase(it);
  return DFLASH_OK;
}

int dflash_free_drafter_kv(dflash_handle *h, const int32_t *blocks, int32_t n_blocks) {
  if (!h || !blocks || n_blocks < 1) return fail(DFLASH_EINVAL, "NULL argument");
  std::lock_guard<std::mutex> lk(h->mu);
  auto it = h->carried.find(blocks[0]);
  if (it == h->carried.end() || it->second.first != std::vector<int32_t>(blocks, blocks + n_blocks))
    return fail(DFLASH_EINVAL, "pages are not a bundle taken by take_drafter_kv");
  for (int32_t p : it->second.first) h->pool.give(p);
  h->carried.erase(it);
  return DFLASH_OK;
}

int dflash_debug_state(const dflash_state *st, int64_t *ctx_len, int32_t *first_block,
                       int32_t *table, int32_t cap) {
  if (!st) return fail(DFLASH_EINVAL, "NULL state");
  if (ctx_len) *ctx_len = st->ctx_len;
  if (st->pages.empty()) {
    if (first_block) *first_block = -1;
    return 0;
  }
  int64_t lo = st->pages.begin()->first, hi = st->pages.rbegin()->first;
  if (first_block) *first_block = (int32_t)lo;
  int32_t n = (int32_t)(hi - lo + 1);
  for (int64_t b = lo; b <= hi && table && b - lo < cap; ++b) {
    auto it = st->pages.find(b);
    table[b - lo] = it == st->pages.end() ? -1 : it->second;
  }
  return n;
}

int dflash_debug_pool(const dflash_handle *h, int32_t *in_use, int32_t *total) {
  if (!h) return fail(DFLASH_EINVAL, "NULL handle");
  if (in_use) *in_use = h->pool.total - h->pool.n_free();
  if (total) *total = h->pool.total;
  return DFLASH_OK;
}

int dflash_debug_gather_kv(dflash_handle *h, const dflash_state *st, int32_t layer, int64_t pos0,
                           int32_t n, float *k_out, float *v_out, void *stream) {
  if (!h || !st || !h->compute) return fail(DFLASH_EINVAL, "NULL argument or no device side");
  if (layer < 0 || layer >= h->g.L || n < 0) return fail(DFLASH_EINVAL, "bad layer or count");
  std::lock_guard<std::mutex> lk(h->mu);
  std::vector<dfl::RowMeta> rows;
  for (int64_t j = pos0; j < pos0 + n; ++j) {
    auto it = st->pages.find(j / h->cfg.kv_block);
    if (j < 0 || j >= st->ctx_len || it == st->pages.end())
      return fail(DFLASH_EINVAL, "position %lld is not stored", (long long)j);
    dfl::RowMeta r{};
    r.pos = (int32_t)j;
    r.page = it->second;
    r.slot = (int32_t)(j % h->cfg.kv_block);
    rows.push_back(r);
  }
  cudaStream_t s = (cudaStream_t)stream;
  dfl::CallMeta cm;
  int rc = upload_meta(h, {}, rows, {}, s, &cm);
  if (rc) return rc;
  CK(dfl::gather_kv_rows(h->g, h->w, h->b, cm.rows, n, layer, k_out, v_out, s));
  return DFLASH_OK;
}

int dflash_debug_set_graphs(dflash_handle *h, int32_t enable) {
  if (!h) return fail(DFLASH_EINVAL, "NULL handle");
  h->use_graphs = enable != 0;
  if (!h->use_graphs) drop_graphs(h);
  return DFLASH_OK;
}

int dflash_debug_set_probe(dflash_handle *h, void *ev_begin, void *ev_end) {
  if (!h) return fail(DFLASH_EINVAL, "NULL handle");
  h->b.probe_begin = (cudaEvent_t)ev_begin;
  h->b.probe_end = (cudaEvent_t)ev_end;
  return DFLASH_OK;
}

int dflash_debug_set_step_probe(dflash_handle *h, void *ev_begin, void *ev_end) {
  if (!h) return fail(DFLASH_EINVAL, "NULL handle");
  h->b.step_begin = (cudaEvent_t)ev_begin;
  h->b.step_end = (cudaEvent_t)ev_end;
  return DFLASH_OK;
}

int64_t dflash_debug_launch_count(void) { return dfl::launch_count(); }

int dflash_debug_set_chain(dflash_handle *h, int32_t enable) {
  if (!h) return fail(DFLASH_EINVAL, "NULL handle");
  if (!h->compute) return DFLASH_OK;
  h->b.use_chain = enable != 0 && h->chain_ok;
  drop_graphs(h);
  return DFLASH_OK;
}

int dflash_debug_last_path(const dflash_handle *h) {
  if (!h) return fail(DFLASH_EINVAL, "NULL handle");
  return h->last_chained;
}

int dflash_debug_set_fault(dflash_handle *h, int64_t wait_ns) {
  if (!h || wait_ns < 0 || wait_ns > 2000000000ll)
    return fail(DFLASH_EINVAL, "NULL handle or wait outside 0..2e9 ns");
  h->b.fault_ns = wait_ns;
  return DFLASH_OK;
}

int dflash_debug_rows(dflash_handle *h, int32_t n_rows, int32_t *ids, float *p1, void *stream) {
  if (!h || !h->compute || n_rows < 0 || n_rows > h->D_max || (n_rows > 0 && (!ids || !p1)))
    return fail(DFLASH_EINVAL, "NULL argument, no device side, or rows outside 0..%d", h ? h->D_max : 0);
  cudaStream_t s = (cudaStream_t)stream;
  CK(cudaMemcpyAsync(ids, h->b.row_id, sizeof(int32_t) * (size_t)n_rows, cudaMemcpyDeviceToHost, s));
  CK(cudaMemcpyAsync(p1, h->b.row_p1, sizeof(float) * (size_t)n_rows, cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  return DFLASH_OK;
}

int dflash_debug_gemm(const void *w, const void *x, float *y, int32_t m, int32_t n_w, int32_t k,
                      int32_t grid_cap, void *stream) {
  if (!w || !x || !y || m <= 0 || n_w <= 0 || k <= 0 || k % 64)
    return fail(DFLASH_EINVAL, "bad GEMM arguments");
  cudaStream_t s = (cudaStream_t)stream;
  const int bn = dfl::tc::pick_bn(m);
  CUtensorMap mw, mx;
  if (!dfl::tc::make_map_2d(&mw, w, false, n_w, k, 128) ||
      !dfl::tc::make_map_2d(&mx, x, false, m, k, bn))
    return fail(DFLASH_ECUDA, "cuTensorMapEncodeTiled failed");
  dfl::GemmParams p{};
  p.m_act = m;
  p.n_w = n_w;
  p.k = k;
  p.epi = dfl::EPI_TC_STORE_F32;
  p.out = y;
  p.ldo = n_w;
  p.grid_cap = grid_cap;
  const int tiles = ((n_w + 127) / 128) * ((m + bn - 1) / bn);
  void *ws = nullptr, *cnt = nullptr, *status = nullptr;
  CK(cudaMalloc(&ws, dfl::tc::ws_floats(dfl::tc::num_sms()) * sizeof(float)));
  CK(cudaMalloc(&cnt, sizeof(int) * (size_t)tiles + 16));
  CK(cudaMalloc(&status, 16));
  CK(cudaMemsetAsync(cnt, 0, sizeof(int) * (size_t)tiles + 16, s));
  CK(cudaMemsetAsync(status, 0, 16, s));
  p.ws = (float *)ws;
  p.counters = (int *)cnt;
  p.status = (int *)status;
  cudaError_t e = dfl::tc::gemm(mw, mx, bn, p, s);
  int st = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&st, status, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  cudaFree(ws);
  cudaFree(cnt);
  cudaFree(status);
  CK(e);
  if (st) return fail(DFLASH_EDEVICE, "GEMM status %d", st);
  return DFLASH_OK;
}

int dflash_debug_lmhead(const void *w, const void *x, void *partials, int32_t m, int32_t n_w,
                        int32_t k, void *stream) {
  if (!w || !x || !partials || m <= 0 || n_w <= 0 || k <= 0 || k % 64)
    return fail(DFLASH_EINVAL, "bad lm_head arguments");
  cudaStream_t s = (cudaStream_t)stream;
  CUtensorMap mx, mw;
  if (!dfl::tc::make_map_2d(&mx, x, false, m, k, 128) ||
      !dfl::tc::make_map_2d(&mw, w, false, n_w, k, 256))
    return fail(DFLASH_ECUDA, "cuTensorMapEncodeTiled failed");
  void *status = nullptr;
  CK(cudaMalloc(&status, 16));
  CK(cudaMemsetAsync(status, 0, 16, s));
  dfl::LmArgs p{};
  p.m_act = m;
  p.n_w = n_w;
  p.k = k;
  p.nd = m;
  p.mask_words = (n_w + 31) / 32;
  p.out = (dfl::LmPartial *)partials;
  p.status = (int *)status;
  cudaError_t e = dfl::tc::lmhead(mx, mw, p, s);
  int st = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&st, status, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  cudaFree(status);
  CK(e);
  if (st) return fail(DFLASH_EDEVICE, "lm_head status %d", st);
  return DFLASH_OK;
}

int dflash_debug_set_taps(dflash_handle *h, float *x_taps, void *z, float *logits) {
  if (!h) return fail(DFLASH_EINVAL, "NULL handle");
  if (((uintptr_t)x_taps | (uintptr_t)z | (uintptr_t)logits) & 15)
    return fail(DFLASH_EINVAL, "tap buffers must be 16-byte aligned");
  h->b.tap_x = x_taps;
  h->b.tap_z = (bf16 *)z;
  h->b.tap_logits = logits;
  return DFLASH_OK;
}

int32_t dflash_debug_attn_work(int32_t n_seq, const int32_t *pos, const int32_t *ws,
                               int32_t num_kv_heads, int32_t gamma, int32_t slot_cap,
                               int32_t grid, int32_t sms, int32_t *items, int32_t cap_items,
                               int32_t *cta_off, int32_t *n_pairs) {
  if (n_seq < 0 || (n_seq > 0 && (!pos || !ws)) || num_kv_heads < 1 || gamma < 1 ||
      slot_cap < 1 || grid < 0 || sms < 1 || cap_items < 0 || (cap_items > 0 && !items) ||
      (grid > 0 && !cta_off))
    return fail(DFLASH_EINVAL, "bad attention work arguments");
  std::vector<dfl::SeqMeta> seq(n_seq);
  for (int i = 0; i < n_seq; ++i) {
    if (ws[i] < 0 || ws[i] > pos[i]) return fail(DFLASH_EINVAL, "window start outside 0..pos");
    seq[i].pos = pos[i];
    seq[i].ws = ws[i];
  }
  dfl::Geo g{};
  g.nkv = num_kv_heads;
  g.gamma = gamma;
  std::vector<dfl::AttnItem> it;
  std::vector<dfl::AttnPair> pr;
  std::vector<int32_t> off;
  if (!dfl::build_attn_work_sms(g, seq, slot_cap, grid, sms, &it, &pr, &off))
    return fail(DFLASH_EINVAL, "slot_cap %d cannot hold one chunk per window", slot_cap);
  if ((int64_t)it.size() > cap_items) return fail(DFLASH_EINVAL, "items beyond cap_items");
  for (size_t i = 0; i < it.size(); ++i) {
    int32_t *o = items + 5 * i;
    o[0] = it[i].s;
    o[1] = it[i].g;
    o[2] = it[i].k0;
    o[3] = it[i].k1;
    o[4] = it[i].slot;
  }
  if (grid > 0) memcpy(cta_off, off.data(), sizeof(int32_t) * (size_t)(grid + 1));
  if (n_pairs) *n_pairs = (int32_t)pr.size();
  return (int32_t)it.size();
}

}  // extern "C"

// ====================================================== propose driver ==
namespace dfl {

// Runs the forward of a call: replays the graph captured for the call's launch
// shape (capturing it on first use), or launches the kernels directly when
// graphs are off or the capture fails.
// The call's metadata upload (meta_bytes from the pinned staging buffer) and
// the results' download are part of the same graph, so a replay is one
// launch and one synchronisation.
int run_forward(dflash_handle *h, const CallMeta &cm, int nd, const int32_t *bitmask,
                size_t meta_bytes, cudaStream_t s) {
  auto body = [&](cudaStream_t st) -> int {
    if (cudaMemcpyAsync(h->meta_dev, h->meta_host, meta_bytes, cudaMemcpyHostToDevice, st) !=
        cudaSuccess)
      return DFLASH_ECUDA;
    int rc = forward(h->g, h->cfg, h->w, h->b, cm, nd, bitmask, h->M_ctx, st);
    if (rc) return rc;
    if (cudaMemcpyAsync(h->b.out_host, h->b.out_dev, h->b.out_bytes, cudaMemcpyDeviceToHost, st) !=
        cudaSuccess)
      return DFLASH_ECUDA;
    return DFLASH_OK;
  };
  if (h->use_graphs) {
    const std::vector<uintptr_t> key = {
        (uintptr_t)meta_bytes,
        (uintptr_t)cm.n_seq, (uintptr_t)cm.n_rows, (uintptr_t)nd, (uintptr_t)bitmask,
        (uintptr_t)h->b.tap_x, (uintptr_t)h->b.tap_z, (uintptr_t)h->b.tap_logits,
        (uintptr_t)h->b.probe_begin, (uintptr_t)h->b.probe_end,
        (uintptr_t)h->b.step_begin,  (uintptr_t)h->b.step_end, (uintptr_t)h->b.fault_ns};
    auto it = h->graphs.find(key);
    if (it == h->graphs.end()) {
      const int64_t l0 = launch_count();
      cudaGraph_t graph = nullptr;
      cudaGraphExec_t exec = nullptr;
      bool ok = cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeRelaxed) == cudaSuccess;
      int rc = ok ? body(h->cap_stream) : DFLASH_ECUDA;
      if (ok) ok = cudaStreamEndCapture(h->cap_stream, &graph) == cudaSuccess && rc == DFLASH_OK;
      if (ok) ok = cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess;
      if (graph) cudaGraphDestroy(graph);
      const int64_t launches = launch_count() - l0;
      count_launches((int)-launches);   // counted when the graph runs
      cudaGetLastError();
      if (ok) {
        if (h->graphs.size() >= 64) drop_graphs(h);
        it = h->graphs.emplace(key, std::make_pair(exec, launches)).first;
      } else {
        h->use_graphs = false;   // capture is not available here: launch directly from now on
      }
    }
    if (it != h->graphs.end()) {
      CK(cudaGraphLaunch(it->second.first, s));
      count_launches((int)it->second.second);
      return DFLASH_OK;
    }
  }
  const int rc = body(s);
  if (rc) return fail(rc, "%s", rc == DFLASH_ECUDA ? "cudaMemcpyAsync failed" : last_build_error());
  return DFLASH_OK;
}

int propose_impl(dflash_handle *h, int n, dflash_state *const *states,
                 const uint32_t *last_tokens, const int64_t *positions,
                 const void *const *new_rows, const int32_t *n_new, int num_drafts,
                 const int32_t *bitmask, uint32_t *drafts, int32_t *n_out, float *conf,
                 void *stream) {
  if (!h) return fail(DFLASH_EINVAL, "NULL handle");
  if (!states || !last_tokens || !positions || !n_new || !drafts || !n_out)
    return fail(DFLASH_EINVAL, "NULL argument");
  cudaStream_t s = (cudaStream_t)stream;
  std::lock_guard<std::mutex> lk(h->mu);
  const dflash_config &c = h->cfg;
  if (num_drafts < 1 || num_drafts > c.gamma - 1)
    return fail(DFLASH_EINVAL, "num_drafts %d outside 1..%d", num_drafts, c.gamma - 1);
  std::set<dflash_state *> seen;
  for (int i = 0; i < n; ++i) {
    dflash_state *st = states[i];
    if (!st || !h->states.count(st)) return fail(DFLASH_EINVAL, "state %d unknown", i);
    if (!seen.insert(st).second) return fail(DFLASH_EINVAL, "state %d repeated", i);
    if (last_tokens[i] >= (uint32_t)c.vocab) return fail(DFLASH_EINVAL, "token %u >= vocab", last_tokens[i]);
    if (st->pending) return fail(DFLASH_ESTATE, "sequence %d: propose before after_verify", i);
    if (n_new[i] < 0) return fail(DFLASH_EINVAL, "n_new < 0");
    if (positions[i] != st->ctx_len + n_new[i])
      return fail(DFLASH_EPOSITION, "sequence %d: position %lld != ctx_len %lld + n_new %d", i,
                  (long long)positions[i], (long long)st->ctx_len, n_new[i]);
    if (st->expected_next >= 0 && positions[i] != st->expected_next)
      return fail(DFLASH_EPOSITION, "sequence %d: position %lld != %lld set by after_verify", i,
                  (long long)positions[i], (long long)st->expected_next);
    if (positions[i] > st->cap) return fail(DFLASH_EINVAL, "sequence %d: beyond its budget", i);
    if (c.ctx_window > 0 && !st->pages.empty() &&
        window_start(h, positions[i]) < st->pages.begin()->first * (int64_t)c.kv_block)
      // only an installed carry can get here: rows below its first page are gone
      return fail(DFLASH_EPOSITION,
                  "sequence %d: the window of position %lld reaches below the installed pages",
                  i, (long long)positions[i]);
    if (h->compute && n_new[i] > 0 &&
        (!new_rows || !new_rows[i] || !aligned16(new_rows[i])))
      return fail(DFLASH_EINVAL, "sequence %d: new rows must be a 16-byte aligned device pointer", i);
  }
  std::vector<AppendPlan> plans;
  for (int i = 0; i < n; ++i)
    plans.push_back(plan_append(h, states[i], n_new[i], new_rows ? new_rows[i] : nullptr));
  if (!pool_can_cover(h, plans)) return fail(DFLASH_ENOMEM, "KV pool exhausted");
  const Snapshot snap = snapshot(states, n);
  commit_plans(h, plans);
  for (auto &p : plans) p.st->ctx_len = p.new_len;
  if (!h->compute) {
    for (int i = 0; i < n; ++i) {
      states[i]->pending = true;
      states[i]->pend_pos = positions[i];
      states[i]->pend_nout = num_drafts;
      states[i]->expected_next = -1;
      n_out[i] = num_drafts;
      for (int t = 0; t < num_drafts; ++t) drafts[i * num_drafts + t] = 0;
      if (conf) conf[i] = 0.f;
    }
    return DFLASH_BOOKKEEPING_ONLY;
  }
  // Metadata: sequences, stored ctx rows, live page ids of each window.
  std::vector<SeqMeta> seq(n);
  std::vector<RowMeta> rows;
  std::vector<int32_t> page_ids;
  rows_of(h, plans, &rows);
  // Calls whose new-row totals differ share a graph: above 16 rows the list
  // is padded to a multiple of 32 with rows (seq -1) that are packed as
  // zeros, carried through the projections and never stored.
  if (rows.size() > 16) {
    RowMeta pad{};
    pad.page = -1;
    pad.seq = -1;
    pad.src = nullptr;
    rows.resize((rows.size() + 31) / 32 * 32, pad);
  }
  for (int i = 0; i < n; ++i) {
    dflash_state *st = states[i];
    SeqMeta &m = seq[i];
    m.pos = (int32_t)positions[i];
    m.ws = (int32_t)window_start(h, positions[i]);
    m.token = (int32_t)last_tokens[i];
    m.page_base = (int32_t)page_ids.size();
    if (m.ws < m.pos) {
      // the window's pages are consecutive keys of the ordered page map
      auto it = st->pages.lower_bound(m.ws / c.kv_block);
      for (int64_t b = m.ws / c.kv_block; b <= (m.pos - 1) / c.kv_block; ++b, ++it) {
        if (it == st->pages.end() || it->first != b) {
          rollback(h, snap);
          return fail(DFLASH_ESTATE, "internal: window page %lld of sequence %d missing",
                      (long long)b, i);
        }
        page_ids.push_back(it->second);
      }
    }
  }
  std::vector<AttnItem> items;
  std::vector<AttnPair> pairs;
  std::vector<int32_t> cta_off;
  thread_local std::vector<ChainAttnItem> citems;
  citems.clear();
  const bool chained = chain_applies(h->g, h->b, (int)rows.size(), n * h->g.gamma);
  if (chained) {
    // the chained path runs the attention inside its launches
    build_chain_attn_items(h->g, seq, tc::num_sms(), &citems);
    if ((int)citems.size() > h->cap_citems) {
      rollback(h, snap);
      return fail(DFLASH_EINVAL, "internal: chained attention items beyond the capacity");
    }
  } else if (!build_attn_work(h->g, seq, h->b.attn_slots, h->b.attn_grid_tc, &items, &pairs,
                              &cta_off)) {
    rollback(h, snap);
    return fail(DFLASH_EINVAL, "internal: attention work beyond the slot capacity");
  }
  CallMeta cm;
  size_t meta_bytes = 0;
  int rc = upload_meta(h, seq, rows, page_ids, s, &cm, items, pairs, cta_off, &meta_bytes, citems);
  if (rc == DFLASH_OK) rc = run_forward(h, cm, num_drafts, bitmask, meta_bytes, s);
  h->last_chained = chained ? 1 : 0;
  if (rc == DFLASH_OK) {
    // Results are on the host after one synchronisation.
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess)
      rc = fail(DFLASH_ECUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  }
  if (rc) {
    rollback(h, snap);
    return rc;
  }
  size_t nd = (size_t)num_drafts;
  const int32_t *status = (const int32_t *)h->b.out_host;
  const uint32_t *dr = (const uint32_t *)(h->b.out_host + h->b.off_drafts);
  const int32_t *no = (const int32_t *)(h->b.out_host + h->b.off_nout);
  const float *cf = (const float *)(h->b.out_host + h->b.off_conf);
  if (*status) {
    // The device abandoned or rejected part of the call's work: nothing of it
    // is returned and every state goes back to where it was. The status word
    // and the stream-K tile counters (an aborted CTA may have left a tile's
    // count behind) start from zero again.
    int st_bits = *status;
    rollback(h, snap);
    CK(cudaMemsetAsync(h->b.status, 0, sizeof(int), s));
    CK(cudaMemsetAsync(h->b.counters, 0, sizeof(int) * (size_t)h->b.n_counters, s));
    CK(cudaStreamSynchronize(s));
    return fail(DFLASH_EDEVICE, "device status %d (%s)", st_bits,
                (st_bits & dfl::ST_TIMEOUT) ? "a bounded wait ran out" : "a bounds check tripped");
  }
  for (int i = 0; i < n; ++i) {
    n_out[i] = no[i];
    memcpy(drafts + i * nd, dr + i * nd, nd * sizeof(uint32_t));
    if (conf) conf[i] = cf[i];
    states[i]->pending = true;
    states[i]->pend_pos = positions[i];
    states[i]->pend_nout = no[i];
    states[i]->expected_next = -1;
  }
  return DFLASH_OK;
}

}  // namespace dfl
