/*
 * dflash.h — C ABI of libdflash: the propose forward of a block-diffusion
 * (DFlash-style) speculative-decoding draft head on one sm_103a GPU.
 *
 * Sources (API pages of the head this library implements):
 *   [P1] "Struct BlockDiffusionDraftHead"  (spark_model::layers::dflash_head)
 *   [P2] "BlockDiffusionDraftHead"         (metrale_model_arch::dflash_head)
 *   [P3] "Trait DraftProposer"             (spark_model::speculative)
 *
 * Conventions for every call:
 *   - Every call returns a status (DFLASH_OK or a code below). On any error
 *     the handle and every state are unchanged: a call checks all arguments
 *     and the KV pool's capacity before it mutates anything, and a call that
 *     fails after that point (a CUDA error, or DFLASH_EDEVICE: a kernel's
 *     bounds check or bounded wait gave up) puts every state it touched and
 *     the pool back as they were. After DFLASH_EDEVICE the call's outputs
 *     are not written and the device work it started has been abandoned:
 *     K/V slots past a restored ctx_len may hold partial writes (the next
 *     append of those positions overwrites them), and a page that the call
 *     retired and took again may have lost rows below the window, which no
 *     later propose of that state attends. The handle stays usable.
 *   - dflash_last_error() returns a message for the last failing call on the
 *     calling thread.
 *   - "dev" marks a device pointer, "host" a host pointer. Device work runs on
 *     the caller's stream (a cudaStream_t passed as void*, NULL = the legacy
 *     default stream).
 *   - Ownership: the caller owns the weights, the input stacks and the
 *     bitmasks, and keeps them alive for the handle's life (weights) or until
 *     the call's stream work has finished (inputs). The library owns the
 *     stitched K/V and QKV weights it builds, the paged KV pool, its scratch
 *     and the states.
 *   - One handle is driven by one host thread at a time; the KV pool inside a
 *     handle is guarded by a lock (the Mutex around kv_cache in [P1]).
 *
 * Tensor layouts (row-major, bf16 unless noted; a "[out, in]" matrix is a
 * linear layer's weight, y = x W^T):
 *   embed, lm_head [vocab, hidden]      shared with the target ([P1] fields
 *                                        embed_tokens_shared, lm_head_shared)
 *   fc             [hidden, n_target_layers*target_hidden]   ([P1] field fc)
 *   hidden_norm, norm [hidden]          RMSNorm gains ([P1] fields)
 *   inv_freq       [head_dim/2] f32     RoPE table ([P1] field yarn_inv_freq)
 *   per layer l, 11 pointers in this order:
 *     in_norm [hidden], q [nq*d, hidden], k [nkv*d, hidden], v [nkv*d, hidden],
 *     q_norm [d], k_norm [d], o [hidden, nq*d], post_norm [hidden],
 *     gate [inter, hidden], up [inter, hidden], down [hidden, inter]
 *   lm_head_fp8    [vocab, hidden] FP8 E4M3 codes, lm_head_scale [vocab] f32
 *                  ([P1] field lm_head_shared_fp8; logit = scale_v * <z, codes_v>)
 *   kv_scale       [num_layers][num_kv_heads][2] f32 (K, V) for the FP8 cache
 *   target stack rows [rows, n_target_layers*target_hidden] bf16, the target's
 *                  hiddens captured at target_layer_ids, shallow to deep
 *                  ([P3] propose argument target_hidden_stack)
 *   bitmask        [ceil(vocab/32)] int32 words per sequence; token t allowed
 *                  iff bit (t & 31) of word (t >> 5) is set ([P3] propose
 *                  argument grammar_bitmask)
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dflash_handle dflash_handle;
typedef struct dflash_state dflash_state;

enum {
    DFLASH_OK = 0,
    DFLASH_DECLINED = 1,          /* propose_batch declined: loop dflash_propose ([P3] propose_batch, Ok(None)) */
    DFLASH_BOOKKEEPING_ONLY = 2,  /* handle built without weights: state updated, nothing computed */
    DFLASH_EINVAL = -1,           /* bad argument or geometry */
    DFLASH_ENOMEM = -2,           /* KV pool or device memory exhausted */
    DFLASH_ESTATE = -3,           /* call out of order (propose twice, after_verify without propose) */
    DFLASH_EPOSITION = -4,        /* position != ctx_len + n_new, or != the position after_verify set */
    DFLASH_ECUDA = -5,            /* a CUDA call failed */
    DFLASH_EDEVICE = -6           /* a kernel's bounds check or bounded wait gave up (device status word) */
};

typedef struct {
    int32_t num_layers, hidden, intermediate, num_q_heads, num_kv_heads, head_dim;
    int32_t vocab;
    int32_t gamma;               /* block rows per sequence ([P1] field gamma) */
    uint32_t mask_token_id;      /* rows 1..gamma-1 of a block embed this id */
    int32_t n_target_layers;     /* len(target_layer_ids) */
    int32_t target_hidden;
    int32_t fc_in_features;      /* the fc weight's input width; must equal n_target_layers*target_hidden
                                    ([P1] validate_against_target: a mismatch is a hard error) */
    float rms_eps;               /* 1e-6 ([P1] field rms_norm_eps) */
    int32_t ctx_window;          /* most past positions attended; 0 = no ctx ([P1]/[P2] field ctx_window) */
    int32_t kv_block;            /* positions per KV page */
    int32_t prefill_chunk;       /* ctx rows per fused K/V GEMM pass in prefill */
    int32_t max_batch;           /* widest propose_batch ([P1] propose_batch_max) */
    int32_t max_seq_len;         /* per-state position ceiling ([P1] field max_seq_len) */
    int32_t kv_pool_blocks;      /* pages in the pool; 0 = max_batch * (min(ctx_window, max_seq_len)/kv_block + 2) */
    int32_t kv_dtype;            /* 0 = bf16 cache ([P2] kv_cache), 1 = FP8 E4M3 with kv_scale ([P1] kv_cache) */
    int32_t lm_head_dtype;       /* 0 = bf16 lm_head; 1 = FP8 E4M3 codes + per-row scales; 2 =
                                    NVFP4: E2M1 codes + E4M3 scales per 16 elements + a global
                                    scale. 1 and 2 stream the codes (no 16-bit copy of the table
                                    is made) and need hidden a multiple of 256 */
    float rope_attn_factor;      /* YaRN attention temperature: the rotated q and k (ctx keys
                                    included) are scaled by it; 0 = none (1). For rope_scaling
                                    factor s, dflash_yarn_inv_freq returns 0.1 ln(s) + 1 */
    int32_t shifted_rows;        /* [P1]/[P2] field shifted_rows (the DSpark convention): 1 = block
                                    row j predicts the token at position+j+1, so drafts 1..n come
                                    from block rows 0..n-1 (the all-rows argmax vector rotated
                                    right by one); 0 = drafts from rows 1..n */
} dflash_config;

typedef struct {
    const void *embed, *lm_head;                       /* dev, borrowed; lm_head may be NULL when
                                                          lm_head_dtype != 0 */
    const void *lm_head_fp8; const float *lm_head_scale;/* dev, used when lm_head_dtype == 1 */
    const void *fc, *hidden_norm, *norm;               /* dev */
    const float *inv_freq;                             /* dev [head_dim/2] */
    const float *kv_scale;                             /* dev, used when kv_dtype == 1 */
    const void *const *layers;                         /* HOST array of num_layers*11 dev pointers */
    /* used when lm_head_dtype == 2 ([P1]/[P2] field lm_head_nvfp4, "packed + scales"):
     * codes [vocab, hidden/2] u8, element 2j in the low nibble; scales
     * [vocab, hidden/16] E4M3 bytes, one per 16 consecutive elements of a row;
     * value = e2m1 * e4m3(scale) * global */
    const void *lm_head_nvfp4; const void *lm_head_nvfp4_scale;
    float lm_head_nvfp4_global;
} dflash_weights;

/* Build a head ([P1] from_weights). Validates the geometry, stitches the fused
 * ctx K/V weight [L*2*kv_dim, hidden] with rows [K0; V0; K1; V1; ...]
 * ([P1]/[P2] field fused_kv_weight) and per-layer QKV / gate-up weights,
 * builds the RoPE cos/sin table from inv_freq, and allocates the KV pool and
 * the scratch. weights == NULL builds a bookkeeping-only handle (no device
 * memory, no kernels) whose prefill/propose only run the page bookkeeping and
 * return DFLASH_BOOKKEEPING_ONLY; it exists for host-side tests.
 * Errors: EINVAL (geometry, fc width), ENOMEM, ECUDA. */
DFLASH_API int dflash_create(const dflash_config *cfg, const dflash_weights *weights, dflash_handle **out);
DFLASH_API void dflash_destroy(dflash_handle *h);   /* frees every state still alive, then the handle */

/* [P1]/[P3] propose_batch_max: the widest batch one forward carries (max_batch). */
DFLASH_API int dflash_propose_batch_max(const dflash_handle *h);
/* [P1]/[P3] block_gamma: the trained block size gamma. */
DFLASH_API int dflash_block_gamma(const dflash_handle *h);

/* [P3] alloc_state / alloc_state_for. budget_tokens bounds the positions the
 * state will hold (prompt + max new tokens); INT64_MAX means unknown and
 * falls back to max_seq_len. Allocates no device memory (pages come from the
 * shared pool as rows land). Errors: EINVAL. */
DFLASH_API int dflash_alloc_state(dflash_handle *h, int64_t budget_tokens, dflash_state **out);
/* [P3] free_state: returns every page the state holds to the pool and frees
 * the state. Errors: EINVAL (unknown state). */
DFLASH_API int dflash_free_state(dflash_handle *h, dflash_state *st);

/* Append n_rows ctx rows (target stack rows of positions ctx_len ..
 * ctx_len+n_rows-1): fc, hidden_norm, fused K/V GEMM, k_norm, RoPE and paged
 * write ([P1] fields fc, hidden_norm, fused_kv_weight, kv_cache). Rows below
 * ctx_len+n_rows-ctx_window are neither computed nor stored; the rest run in
 * chunks of prefill_chunk rows. Asynchronous on the stream.
 * stack: dev [n_rows, n_target_layers*target_hidden] bf16, rows 16-byte aligned.
 * Errors: EINVAL, ESTATE (a propose awaits after_verify), ENOMEM (pool). */
DFLASH_API int dflash_prefill(dflash_handle *h, dflash_state *st, const void *stack, int32_t n_rows,
                   void *stream);

/* [P3] propose: append the n_new target stack rows of positions
 * ctx_len..position-1 (as dflash_prefill), then run the gamma-row block
 * (last_token at `position`, mask_token_id at position+1..position+gamma-1)
 * through the layers, the final norm and the lm_head, and return the argmax
 * of block rows 1..num_drafts (rows 0..num_drafts-1 with shifted_rows).
 * position must equal ctx_len + n_new, and,
 * after dflash_after_verify(k), the previous position + k + 1.
 *   new_rows: dev [n_new, stack width] bf16 or NULL when n_new == 0
 *   num_drafts: 1 .. gamma-1
 *   bitmask: dev [ceil(vocab/32)] int32 or NULL (unconstrained)
 *   drafts: host [num_drafts] u32; n_out: host, drafts produced (0 when the
 *     bitmask allows no token); conf: host f32 or NULL — chain confidence, the
 *     minimum over drafts of the top-1 softmax probability ([P1]/[P3]
 *     last_confidence), 0 when n_out == 0.
 * Synchronises the stream once (the drafts are returned on the host).
 * Errors: EINVAL, ESTATE, EPOSITION, ENOMEM, ECUDA, EDEVICE. */
DFLASH_API int dflash_propose(dflash_handle *h, dflash_state *st, uint32_t last_token, int64_t position,
                   const void *new_rows, int32_t n_new, int32_t num_drafts,
                   const int32_t *bitmask, uint32_t *drafts, int32_t *n_out, float *conf,
                   void *stream);

/* [P1]/[P2]/[P3] propose_batch: the same as n dflash_propose calls, with one
 * forward over n*gamma rows. Row i of every array belongs to sequence i.
 * Returns DFLASH_DECLINED (nothing changed) for n < 2 or n > max_batch.
 *   states: host [n]; last_tokens: host [n]; positions: host [n];
 *   new_rows: host [n] array of dev pointers (NULL where n_new[i] == 0);
 *   n_new: host [n]; bitmask: dev [n][ceil(vocab/32)] int32 or NULL;
 *   drafts: host [n][num_drafts]; n_out: host [n]; conf: host [n] or NULL.
 * Pages: all sequences retire first, then take pages, in sequence order.
 * Errors: as dflash_propose; EINVAL also for a repeated state. */
DFLASH_API int dflash_propose_batch(dflash_handle *h, int32_t n, dflash_state *const *states,
                         const uint32_t *last_tokens, const int64_t *positions,
                         const void *const *new_rows, const int32_t *n_new, int32_t num_drafts,
                         const int32_t *bitmask, uint32_t *drafts, int32_t *n_out, float *conf,
                         void *stream);

/* [P3] after_verify: the target accepted num_accepted (0..n_out) drafts of
 * the last propose. The next propose sits at position + num_accepted + 1 and
 * brings the num_accepted + 1 target rows of positions position ..
 * position + num_accepted. Pages below that propose's window return to the
 * pool now. Host-only. Errors: EINVAL, ESTATE. */
DFLASH_API int dflash_after_verify(dflash_handle *h, dflash_state *st, int32_t num_accepted);
/* [P3] take_drafter_kv: move the sequence's KV pages out of st so that
 * dflash_free_state releases none of them and the caller can carry them to
 * the sequence's next turn; st then behaves as freshly allocated (ctx_len 0,
 * no pages, no propose pending, no expected position). On DFLASH_OK the
 * physical ids of the live pages, in logical order, are in
 * blocks[0..*n_blocks) (host array of cap entries) and the ctx length in
 * *rows: the bundle now belongs to the caller, who installs it with
 * dflash_install_drafter_kv or releases it with dflash_free_drafter_kv. The
 * page contents are those the state's earlier calls wrote on their streams.
 * The row space is positions, so the trait's last_pair_key has no
 * counterpart (None). Returns DFLASH_DECLINED, changing nothing, when st
 * holds no pages (nothing to carry). Host-only. Errors (nothing changes):
 * EINVAL (unknown state, cap too small), ESTATE (a propose awaits
 * after_verify). */
DFLASH_API int dflash_take_drafter_kv(dflash_handle *h, dflash_state *st, int32_t *blocks,
                                      int32_t cap, int32_t *n_blocks, int64_t *rows);
/* [P3] install_drafter_kv: install a bundle exactly as dflash_take_drafter_kv
 * returned it (blocks[0..n_blocks), rows) into st, which must be fresh
 * (nothing appended since dflash_alloc_state, or taken since). st then holds
 * ctx_len = rows with the bundle as its live pages (logical pages
 * ceil(rows/kv_block) - n_blocks onwards); its next propose brings the rows
 * of positions rows..position-1, and a propose whose window would start
 * below the first installed page fails with EPOSITION. Host-only. Errors
 * (nothing changes, the caller still owns the bundle): EINVAL (not a carried
 * bundle, rows differ, st not fresh or unknown, rows beyond st's budget). */
DFLASH_API int dflash_install_drafter_kv(dflash_handle *h, dflash_state *st,
                                         const int32_t *blocks, int32_t n_blocks, int64_t rows);
/* [P3] free_drafter_kv: return a carried bundle that no state owns to the
 * pool. Host-only. Errors: EINVAL (not a carried bundle); nothing changes. */
DFLASH_API int dflash_free_drafter_kv(dflash_handle *h, const int32_t *blocks, int32_t n_blocks);
/* The YaRN-corrected RoPE inverse-frequency table of a drafter config's
 * rope_scaling ([P1] field yarn_inv_freq: the shipped drafter has factor 64,
 * beta_fast 32, beta_slow 1, original_max_position_embeddings 4096), by the
 * published YaRN "NTK-by-parts" method: pair i of the base table
 * theta^(-2i/head_dim) turns original_max_pos / (2 pi) * base_i times over
 * the original context; pairs from ceil(i_slow) on are divided by factor,
 * pairs up to floor(i_fast) are kept, and those between blend the two
 * linearly in the pair index (i_r: the real pair index that turns r times,
 * clamped to the table). Evaluated in double, written as f32 to the HOST
 * array inv_freq[head_dim/2]; *attn_factor (may be NULL) receives the
 * matching temperature 0.1 ln(factor) + 1 (1 when factor <= 1), to be set
 * as dflash_config.rope_attn_factor. factor 1 gives the plain table.
 * Host-only. Errors: EINVAL (theta <= 1, head_dim not even and positive,
 * factor < 1, beta_slow <= 0, beta_fast <= beta_slow, original_max_pos < 1,
 * NULL inv_freq). */
DFLASH_API int dflash_yarn_inv_freq(double theta, int32_t head_dim, double factor,
                                    double beta_fast, double beta_slow, int32_t original_max_pos,
                                    float *inv_freq, float *attn_factor);
/* [P2] catchup_batch / [P3] catchup_drafter: append, for each of n states,
 * n_rows[i] ctx rows (the target hiddens paired with the tokens the last
 * verify settled) at RoPE positions first_pos[i] .. first_pos[i]+n_rows[i]-1,
 * exactly as dflash_prefill computes and stores them (rows below the window
 * are neither computed nor stored). This head keeps one ctx row per target
 * position, so a state's KV slot and the RoPE position of its next row
 * coincide: first_pos[i] must equal the state's ctx_len. After
 * dflash_after_verify(k) the rows of positions position..position+k (the
 * last verified token's and the accepted drafts') may come here, all or a
 * first part of them, and the next propose then brings only the rest as
 * new_rows (none when all came here).
 *   states: host [n], distinct; tokens: host [n] array of host [n_rows[i]]
 *     u32 arrays (or NULL, or NULL entries): checked < vocab only, the ctx
 *     rows depend on the hiddens alone;
 *   rows: host [n] array of dev [n_rows[i], stack width] bf16 (16-byte
 *     aligned; NULL where n_rows[i] == 0); n_rows, first_pos: host [n];
 *   written: host, may be NULL: rows appended (their sum), 0 on an error.
 * Pages: all states retire first, then take pages, in state order; on an
 * error nothing changes and the message names the state's index. Asynchronous
 * on the stream. Errors: EINVAL (unknown or repeated state, negative count,
 * token outside the vocab, budget, pointer), ESTATE (a propose awaits
 * after_verify), EPOSITION (first_pos != ctx_len, or rows past the position
 * after_verify set), ENOMEM (pool), ECUDA. */
DFLASH_API int dflash_catchup_batch(dflash_handle *h, int32_t n, dflash_state *const *states,
                                    const uint32_t *const *tokens, const void *const *rows,
                                    const int32_t *n_rows, const int64_t *first_pos,
                                    int64_t *written, void *stream);
/* dflash_after_verify for the n states of one propose_batch in one call:
 * num_accepted[i] (0..n_out of state i) applies to states[i]. Every state is
 * checked first (known, not repeated, awaiting after_verify, count in range);
 * on an error nothing changes and the message names the state's index.
 * Host-only. Errors: EINVAL, ESTATE. */
DFLASH_API int dflash_after_verify_batch(dflash_handle *h, int32_t n, dflash_state *const *states,
                                         const int32_t *num_accepted);

/* Message of the last failing call on this thread ("" if none). */
DFLASH_API const char *dflash_last_error(void);

/* ---- inspection, for tests ---------------------------------------------- */
/* ctx_len, the first live logical page (-1 if none) and the physical ids of
 * the live logical pages first..last (table, host, capacity cap). Returns the
 * number of live pages, or a negative status. */
DFLASH_API int dflash_debug_state(const dflash_state *st, int64_t *ctx_len, int32_t *first_block,
                       int32_t *table, int32_t cap);
/* Pages in use / in the pool. */
DFLASH_API int dflash_debug_pool(const dflash_handle *h, int32_t *in_use, int32_t *total);
/* Stored K and V of one layer at positions pos0..pos0+n-1 (all live),
 * dequantised to f32: k_out, v_out dev [n, num_kv_heads, head_dim]. */
DFLASH_API int dflash_debug_gather_kv(dflash_handle *h, const dflash_state *st, int32_t layer, int64_t pos0,
                           int32_t n, float *k_out, float *v_out, void *stream);
/* Taps filled by every later propose* (NULL disables each; 16-byte aligned):
 * x_taps dev f32 [num_layers+1][rows][hidden] (the residual entering each
 * layer and leaving the last); z dev bf16 [rows][hidden] (final norm);
 * logits dev f32 [n*num_drafts][vocab] (draft rows, sequence-major).
 * rows = n*gamma of the call. The logits tap adds a separate GEMM. */
/* Timing probe: when both events are non-NULL, every later propose* records
 * ev_begin before and ev_end after its lm_head stage (the GEMM over the vocab
 * and the per-row argmax/confidence reduction), on the call's stream. Events
 * are the caller's cudaEvent_t. NULL, NULL disables it. */
DFLASH_API int dflash_debug_set_probe(dflash_handle *h, void *ev_begin, void *ev_end);
/* The same around the whole device part of a propose* (from its first
 * kernel to its last), separating device time from host time. */
DFLASH_API int dflash_debug_set_step_probe(dflash_handle *h, void *ev_begin, void *ev_end);
/* Propose calls replay a CUDA graph captured per launch shape (sequences,
 * new ctx rows, drafts, bitmask and tap/probe pointers); enable = 0 launches
 * the kernels one by one instead (same results). On by default. */
DFLASH_API int dflash_debug_set_graphs(dflash_handle *h, int32_t enable);
/* enable = 1 makes few-row proposes (one sequence of 16 block rows, at most
 * 16 new ctx rows, hidden at most 2048, bf16 KV) run as one persistent
 * launch that walks every layer's phases with cross-CTA dependency counters;
 * enable = 0 (the default) keeps them on the kernel-per-step path that every
 * other propose takes (same results within rounding). A shape the chained
 * launch does not take stays on the kernel-per-step path. Errors: EINVAL. */
DFLASH_API int dflash_debug_set_chain(dflash_handle *h, int32_t enable);
/* 1 when the last propose* call took the chained few-row path, else 0. */
DFLASH_API int dflash_debug_last_path(const dflash_handle *h);
/* Test hook of the bounded-wait abort path: with wait_ns > 0, every
 * tensor-core GEMM of later propose* calls has one thread of each CTA wait up
 * to wait_ns (<= 2e9) on a barrier that nothing arrives on; the wait runs
 * out, the CTA raises the device status word, drains its own copies and
 * MMAs, frees its TMEM and exits, and the call returns DFLASH_EDEVICE with
 * its states put back. 0 turns it off. Errors: EINVAL. */
DFLASH_API int dflash_debug_set_fault(dflash_handle *h, int64_t wait_ns);
/* Per draft row of the last propose* call, sequence-major (n*num_drafts
 * rows): the argmax token id (-1 when the bitmask allows nothing) and the
 * top-1 softmax probability 1 / sum_v exp(l_v - max l), as the chain
 * confidence takes its minimum over them. ids, p1: host [n_rows].
 * Synchronises the stream. Errors: EINVAL, ECUDA. */
DFLASH_API int dflash_debug_rows(dflash_handle *h, int32_t n_rows, int32_t *ids, float *p1,
                                 void *stream);
/* Kernels this library has launched since it was loaded (all handles). */
DFLASH_API int64_t dflash_debug_launch_count(void);
/* One tensor-core GEMM in isolation, for kernel tests: y[m, n_w] = x[m, k] *
 * w[n_w, k]^T (bf16 in, f32 out, k % 64 == 0), all dev pointers 16-byte
 * aligned. grid_cap > 0 caps the persistent grid (to force split k-ranges).
 * Synchronises the stream; allocates its own workspace. */
DFLASH_API int dflash_debug_gemm(const void *w, const void *x, float *y, int32_t m, int32_t n_w,
                                 int32_t k, int32_t grid_cap, void *stream);
/* The tensor-core GEMM y[m, n_w] = x[m, k] * w[n_w, k]^T (bf16 in, f32 out),
 * for callers that may not allocate device memory while they run, e.g. an
 * engine that has already handed the whole GPU to its own arena, or a
 * latency-critical loop that cannot afford the device-wide synchronisation
 * of cudaMalloc/cudaFree. It allocates nothing: its scratch (stream-K
 * partials, tile counters, a status word; 2.6 MB) is a fixed array inside
 * the library that every GPU loading the library holds until exit. The API
 * pages have no counterpart of this call.
 * Limits: 1 <= m <= 16, k % 64 == 0, n_w <= 524288 (4096 tiles of 128 rows);
 * w and x 16-byte aligned dev pointers, y a dev pointer. Larger sizes return
 * DFLASH_EINVAL. The first call on each device looks up the array's device
 * address with that device current and keeps it for later calls; make that
 * first call before any stream capture. The kept address belongs to the
 * device's current context: after cudaDeviceReset (or any other end of that
 * context) do not call this entry point again in the same process, since
 * the kept address would no longer be valid. All calls share the array, so calls that overlap on the GPU race:
 * order them. Synchronises the stream; returns DFLASH_OK, DFLASH_EINVAL,
 * DFLASH_ECUDA or DFLASH_EDEVICE (dflash_last_error is not updated). */
DFLASH_API int dflash_gemm_noalloc(const void *w, const void *x, float *y, int32_t m, int32_t n_w,
                                   int32_t k, void *stream);
/* The many-row lm_head kernel in isolation, for kernel tests: for each of the
 * m rows of x [m, k] and each 256-row tile of w [n_w, k] (bf16), the tile's
 * max logit, lowest argmax and sum exp(logit - max), no mask, written to
 * partials dev [m][ceil(n_w/256)] of 16-byte (f32 max, i32 id, f32 sum, pad)
 * records. Synchronises the stream. */
DFLASH_API int dflash_debug_lmhead(const void *w, const void *x, void *partials, int32_t m,
                                   int32_t n_w, int32_t k, void *stream);
DFLASH_API int dflash_debug_set_taps(dflash_handle *h, float *x_taps, void *z, float *logits);
/* Host-only inspection of the split of a call's attention into work items
 * (needs no GPU): for n_seq sequences whose blocks sit at positions pos[i]
 * and whose windows start at ws[i] (0 <= ws[i] <= pos[i]), each of the
 * num_kv_heads key ranges (ctx keys ws..pos-1, then the gamma block keys) is
 * cut into ctx chunks plus one block item, at most slot_cap partial slots in
 * all; with grid > 0 the items are then balanced over grid persistent CTAs
 * for a GPU of sms SMs, exactly as a propose* call does. Writes the items
 * in the order the kernel reads them, 5 int32 each (sequence, kv head, first
 * key, end key, partial slot; the slot is -1 for the block item of a
 * sequence without ctx keys, which is then its only item)
 * into items[cap_items][5], the CTA offsets into cta_off[grid + 1] (CTA b
 * runs items cta_off[b] .. cta_off[b+1]-1) and the number of split pairs into
 * *n_pairs (may be NULL). Keys count from the window start. Returns the item
 * count, or DFLASH_EINVAL (nothing written) for a bad argument or more items
 * than cap_items. Host pointers only. */
DFLASH_API int32_t dflash_debug_attn_work(int32_t n_seq, const int32_t *pos, const int32_t *ws,
                                          int32_t num_kv_heads, int32_t gamma, int32_t slot_cap,
                                          int32_t grid, int32_t sms, int32_t *items,
                                          int32_t cap_items, int32_t *cta_off, int32_t *n_pairs);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
