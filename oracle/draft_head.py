"""CPU oracle for the block-diffusion (DFlash-style) draft head propose forward.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or runs
this module; only the test suite, the package's smoke check and the bench's
CPU-baseline leg do. It shares no code with the CUDA library: it reads plain
CPU tensors (bf16 weights, bf16 target stacks) and computes every step with
torch CPU ops in float64, rounding to bf16 (or FP8 E4M3) exactly where the
method stores a tensor in that format.

Sources (API pages of the same head):
  [P1] "Struct BlockDiffusionDraftHead" (spark_model::layers::dflash_head docs)
  [P2] "BlockDiffusionDraftHead" (metrale_model_arch::dflash_head docs)
  [P3] "Trait DraftProposer" (spark_model::speculative docs)

Where the pages leave a step open, the reading taken is named inline as
"reading: ..." and listed with the others in the design notes.

Precision points (reading: a bf16 model runs bf16 GEMMs, so every GEMM
operand is bf16 and every GEMM accumulates in wide precision):
  * the residual stream x is kept wide (fp32 on the GPU, float64 here);
  * GEMM inputs h, o, u, z, the ctx rows c, the block q/k/v and the cached
    ctx K/V are rounded to bf16 (the cached K/V to E4M3 codes on the FP8 path);
  * norms, RoPE, softmax, SiLU and the logit reductions are wide.

Parity status: every function here is pinned by the CPU tests (closed forms,
brute force on tiny inputs, invariants). Whole-model parity with a real trained
DFlash drafter is unpinned: the pages print no values and no checkpoint exists.
"""
from __future__ import annotations

import heapq
import math
from dataclasses import dataclass, field

import torch

F64 = torch.float64
E4M3_MAX = 448.0


# ----------------------------------------------------------------- formats --
def round_bf16(x: torch.Tensor) -> torch.Tensor:
    """Round to bf16 (round to nearest even) and back to float64.

    The value is first rounded to fp32, as a GPU register holds it, then to
    bf16 by torch's conversion."""
    return x.to(torch.float32).to(torch.bfloat16).to(F64)


def e4m3_codes(x32: torch.Tensor) -> torch.Tensor:
    """fp32 -> FP8 E4M3 value (as float64), round to nearest even, saturating
    at +-448 (OCP 8-bit floating point, E4M3 'satfinite')."""
    x32 = x32.to(torch.float32)
    return x32.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).to(F64)


def e2m1_value(code: int) -> float:
    """OCP MX FP4 E2M1 code -> value: sign bit 3, exponent bits 2..1 (bias
    1), mantissa bit 0; exponent 0 is subnormal (m * 0.5). Magnitudes 0, 0.5,
    1, 1.5, 2, 3, 4, 6."""
    sign = -1.0 if code & 8 else 1.0
    e, m = (code >> 1) & 3, code & 1
    return sign * (0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m))


def e4m3_value(code: int) -> float:
    """OCP FP8 E4M3 byte -> value: sign bit 7, exponent bits 6..3 (bias 7),
    mantissa bits 2..0; exponent 0 is subnormal (m * 2^-9); S.1111.111 is
    NaN (no infinities)."""
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return math.nan
    return sign * (m * 2.0 ** -9 if e == 0 else 2.0 ** (e - 7) * (1.0 + m / 8.0))


def nvfp4_dequant(packed: torch.Tensor, scales: torch.Tensor, global_scale: float) -> torch.Tensor:
    """NVFP4 table -> float64 values ([P1] field lm_head_nvfp4: the target's
    NVFP4 lm_head, 'packed + scales'). reading: the NVFP4 format: E2M1 codes
    two per byte (element 2j in the low nibble, 2j+1 in the high one) in
    packed [rows, k/2] uint8, one E4M3 scale per 16 consecutive elements of a
    row in scales [rows, k/16] uint8, and one f32 global scale: value =
    e2m1 * e4m3(scale) * global."""
    lut4 = torch.tensor([e2m1_value(c) for c in range(16)], dtype=F64)
    lut8 = torch.tensor([e4m3_value(c) for c in range(256)], dtype=F64)
    p = packed.to(torch.int64)
    q = torch.stack([lut4[p & 15], lut4[p >> 4]], dim=-1).reshape(packed.shape[0], -1)
    sc = lut8[scales.to(torch.int64)].repeat_interleave(16, dim=1)
    return q * sc * float(global_scale)


# --------------------------------------------------------------- the math --
def rms_norm(x: torch.Tensor, g: torch.Tensor, eps: float) -> torch.Tensor:
    """RMSNorm over the last axis: g * x / sqrt(mean(x^2) + eps).

    [P1] field ``rms_norm_eps`` (Qwen3 default 1e-6), ``hidden_norm``, ``norm``."""
    x = x.to(F64)
    return g.to(F64) * x / torch.sqrt((x * x).mean(dim=-1, keepdim=True) + eps)


def rope(x: torch.Tensor, pos: torch.Tensor, inv_freq: torch.Tensor) -> torch.Tensor:
    """Rotary embedding over the whole head ([P1] field ``rotary_dim``: full
    rotation, rotary_dim = head_dim), angle pos * inv_freq[i] from the table
    ([P1] field ``yarn_inv_freq``).

    reading: rotate-half pairing (i, i + d/2), the Qwen/NeoX convention.
    x: [..., rows, d]; pos: [rows] integer positions."""
    d = x.shape[-1]
    half = d // 2
    ang = pos.to(F64)[:, None] * inv_freq.to(F64)[None, :]          # [rows, d/2]
    c, s = torch.cos(ang), torch.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=-1)


def yarn_inv_freq(theta: float, d: int, factor: float, beta_fast: float, beta_slow: float,
                  original_max_pos: int) -> torch.Tensor:
    """YaRN inverse frequencies ([P1] field yarn_inv_freq: the drafter's
    rope_scaling factor 64, beta_fast 32, beta_slow 1,
    original_max_position_embeddings 4096), from the published YaRN method
    ("NTK-by-parts"): pair i of the base table theta^(-2i/d) turns
    original_max_pos / (2 pi theta^(2i/d)) times over the original context.
    Pairs turning more than beta_fast times keep their frequency, pairs turning
    fewer than beta_slow times are interpolated (frequency / factor), and the
    pairs between blend the two along a linear ramp over the pair index.

    reading: the ramp runs from floor(i_fast) to ceil(i_slow), i_r being the
    (real) pair index that turns r times, clamped to the table, as config
    files' rope_scaling is read; evaluated in double, stored f32."""
    half = d // 2

    def pair_turning(r):
        return d * math.log(original_max_pos / (r * 2.0 * math.pi)) / (2.0 * math.log(theta))

    lo = max(math.floor(pair_turning(beta_fast)), 0)
    hi = min(math.ceil(pair_turning(beta_slow)), half - 1)
    out = []
    for i in range(half):
        base = theta ** (-2.0 * i / d)
        ramp = min(max((i - lo) / max(hi - lo, 1e-3), 0.0), 1.0)   # 0: keep, 1: interpolate
        out.append(base * (1.0 - ramp) + (base / factor) * ramp)
    return torch.tensor(out, dtype=F64).to(torch.float32)


def yarn_attention_factor(factor: float) -> float:
    """YaRN's attention temperature (the published 0.1 ln(s) + 1), applied by
    scaling the rotated q and k, so the logits scale by its square."""
    return 1.0 if factor <= 1.0 else 0.1 * math.log(factor) + 1.0


def silu(a: torch.Tensor) -> torch.Tensor:
    return a / (1.0 + torch.exp(-a))


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> torch.Tensor:
    """softmax(q k^T / sqrt(d)) v for every query head, no mask.

    q: [rows, nq, d]; k, v: [keys, nkv, d]. reading: query head j reads kv
    head floor(j * nkv / nq) (contiguous GQA groups), scale 1/sqrt(d)."""
    rows, nq, d = q.shape
    nkv = k.shape[1]
    out = torch.empty((rows, nq, d), dtype=F64)
    for j in range(nq):
        g = (j * nkv) // nq
        s = q[:, j, :] @ k[:, g, :].T / math.sqrt(d)                 # [rows, keys]
        s = s - s.max(dim=1, keepdim=True).values
        p = torch.exp(s)
        p = p / p.sum(dim=1, keepdim=True)
        out[:, j, :] = p @ v[:, g, :]
    return out


def bitmask_allowed(bitmask_row: torch.Tensor, vocab: int) -> torch.Tensor:
    """Bool [vocab] from ceil(vocab/32) int32 words: token t is allowed iff bit
    (t & 31) of word (t >> 5) is set ([P3] ``propose`` argument
    ``grammar_bitmask``: 'bit tok set => allowed'; reading: LSB-first)."""
    words = bitmask_row.to(torch.int64) & 0xFFFFFFFF
    t = torch.arange(vocab, dtype=torch.int64)
    return ((words[t >> 5] >> (t & 31)) & 1).bool()


def select_drafts(logits: torch.Tensor, allowed: torch.Tensor | None):
    """Per-row argmax and top-1 softmax probability, then the chain.

    [P1] field ``lm_head_shared`` (per-position argmax over the block's
    logits), [P1]/[P3] ``last_confidence`` (min over drafts of the top-1
    softmax probability). reading: ties go to the lowest token id; masked
    tokens are excluded from the softmax; a row with no allowed token ends the
    chain before it. Returns (drafts, n_out, conf, p1 per produced row)."""
    drafts, p1s = [], []
    for i in range(logits.shape[0]):
        row = logits[i].to(F64)
        if allowed is not None:
            if not bool(allowed.any()):
                break
            row = torch.where(allowed, row, torch.full_like(row, -math.inf))
        m = row.max()
        idx = int(torch.nonzero(row == m)[0, 0])          # lowest id among maxima
        p1 = 1.0 / float(torch.exp(row - m).sum())
        drafts.append(idx)
        p1s.append(p1)
    conf = min(p1s) if p1s else 0.0
    return drafts, len(drafts), conf, p1s


# ------------------------------------------------------- page bookkeeping --
class PagePool:
    """Fixed pool of KV pages with ids 0..n-1; a take returns the lowest free
    id (reading: the pages leave the allocation order open)."""

    def __init__(self, n_pages: int):
        self.free = list(range(n_pages))
        heapq.heapify(self.free)
        self.n_pages = n_pages

    def take(self) -> int:
        return heapq.heappop(self.free)

    def give(self, page: int) -> None:
        heapq.heappush(self.free, page)

    def n_free(self) -> int:
        return len(self.free)


class OracleError(Exception):
    def __init__(self, code: str, msg: str):
        super().__init__(f"{code}: {msg}")
        self.code = code


@dataclass
class SeqState:
    cap: int                                   # ctx positions this state may hold
    ctx_len: int = 0                           # target positions appended
    pages: dict = field(default_factory=dict)  # logical page -> physical id
    rows: dict = field(default_factory=dict)   # position -> (K [L,nkv,d], V [L,nkv,d])
    pending: tuple | None = None               # (position, drafts returned)
    expected_next: int | None = None


# ------------------------------------------------------------------ model --
class DraftHeadOracle:
    """The draft head: construction, per-sequence state, prefill, propose,
    propose_batch and after_verify.

    cfg keys: num_layers hidden intermediate num_q_heads num_kv_heads head_dim
    vocab gamma mask_token_id n_target_layers target_hidden rms_eps ctx_window
    kv_block prefill_chunk max_batch max_seq_len kv_pool_blocks kv_dtype
    (0 bf16, 1 fp8) lm_head_dtype (0 bf16, 1 fp8, 2 nvfp4) shifted_rows (0/1,
    optional)."""

    def __init__(self, cfg: dict, w: dict):
        self.cfg = dict(cfg)
        c = self.cfg
        self.L, self.H = c["num_layers"], c["hidden"]
        self.nq, self.nkv, self.d = c["num_q_heads"], c["num_kv_heads"], c["head_dim"]
        self.kv = self.nkv * self.d
        self.V, self.gamma = c["vocab"], c["gamma"]
        self.eps, self.W, self.B = c["rms_eps"], c["ctx_window"], c["kv_block"]
        if c.get("fc_in_features", c["n_target_layers"] * c["target_hidden"]) != \
                c["n_target_layers"] * c["target_hidden"]:
            # [P1] validate_against_target: a width mismatch is a hard error.
            raise OracleError("EINVAL", "fc input width != n_target_layers*target_hidden")
        f = lambda t: t.to(F64)
        self.embed = w["embed"]                              # gathered per row
        self.lm_head_bf16 = w["lm_head"]
        self.fc = f(w["fc"])
        self.hidden_norm, self.norm = f(w["hidden_norm"]), f(w["norm"])
        self.inv_freq = w["inv_freq"].to(torch.float32)
        # reading: the rotated q and k are scaled by the attention factor
        # (YaRN's temperature; 0 or absent means none)
        self.rope_scale = float(c.get("rope_attn_factor", 0.0) or 1.0)
        self.layers = [{k: f(v) for k, v in lay.items()} for lay in w["layers"]]
        # [P1]/[P2] field fused_kv_weight: rows [K0; V0; K1; V1; ...].
        self.w_kv = torch.cat([torch.cat([lay["k"], lay["v"]], 0) for lay in self.layers], 0)
        self.kv_fp8 = c.get("kv_dtype", 0) == 1
        self.lm_fp8 = c.get("lm_head_dtype", 0) == 1
        # reading: the NVFP4 head is weight-only like the FP8 one (the
        # final-normed z is not quantised), with the block and global scales
        # folded into the dequantised table
        self.lm_nvfp4 = c.get("lm_head_dtype", 0) == 2
        if self.kv_fp8:
            self.kv_scale = w["kv_scale"].to(torch.float32)   # [L, nkv, 2]
        if self.lm_fp8:
            self.lm_codes = w["lm_head_fp8"]
            self.lm_scale = w["lm_head_scale"].to(F64)
        if self.lm_nvfp4:
            self.lm_nv = (w["lm_head_nvfp4"], w["lm_head_nvfp4_scale"],
                          float(w["lm_head_nvfp4_global"]))
        # [P1]/[P2] field shifted_rows (the DSpark convention): block row j's
        # logits give the token at position p + j + 1, so the draft vector is
        # the full-row argmax vector rotated right by one; the verify indexing
        # then reads drafts 1..nd from block rows 0..nd-1. Otherwise row i
        # gives draft i (rows 1..nd).
        self.draft0 = 0 if c.get("shifted_rows", 0) else 1
        self._lm = None
        self.pool = PagePool(self.n_pool_pages())
        self.states: list[SeqState] = []
        # pages moved out of their states by take_drafter_kv and not yet
        # installed or freed: tuple(page ids) -> (ctx_len, stored rows)
        self.carried: dict[tuple, tuple] = {}

    # -- sizes ----------------------------------------------------------------
    def pages_per_seq(self) -> int:
        c = self.cfg
        span = min(self.W, c["max_seq_len"]) if self.W > 0 else 0
        return 0 if span == 0 else span // self.B + 2

    def n_pool_pages(self) -> int:
        c = self.cfg
        if c.get("kv_pool_blocks", 0) > 0:
            return c["kv_pool_blocks"]
        return max(1, c["max_batch"]) * self.pages_per_seq()

    def lm_head(self) -> torch.Tensor:
        """Float64 lm_head rows, built once: bf16 table, the FP8 codes
        (weight-only; the per-row scale is applied to the logits) or the
        dequantised NVFP4 table."""
        if self._lm is None:
            if self.lm_nvfp4:
                self._lm = nvfp4_dequant(*self.lm_nv)
            else:
                src = self.lm_codes if self.lm_fp8 else self.lm_head_bf16
                self._lm = src.to(F64)
        return self._lm

    # -- state ----------------------------------------------------------------
    def alloc_state(self, budget_tokens: int | None = None) -> SeqState:
        """[P3] alloc_state / alloc_state_for: a None budget means 'unknown,
        use the ceiling' (max_seq_len)."""
        cap = self.cfg["max_seq_len"]
        if budget_tokens is not None:
            if budget_tokens <= 0:
                raise OracleError("EINVAL", "budget must be positive")
            cap = min(cap, budget_tokens)
        st = SeqState(cap=cap)
        self.states.append(st)
        return st

    def free_state(self, st: SeqState) -> None:
        """[P3] free_state: release every KV page the state holds."""
        for b in sorted(st.pages):
            self.pool.give(st.pages[b])
        st.pages.clear()
        st.rows.clear()
        self.states.remove(st)

    # -- ctx append: fc, hidden_norm, fused K/V, k_norm, RoPE, paged write ----
    def _plan_append(self, st: SeqState, n: int):
        """Which rows are stored and which pages retire / are taken.

        reading: rows below new_len - ctx_window are neither computed nor
        stored ([P1]/[P2] field ctx_window); pages entirely below the window
        start retire; a page is taken when a row first lands in it."""
        new_len = st.ctx_len + n
        lo = max(st.ctx_len, new_len - self.W) if self.W > 0 else new_len
        ws = max(0, new_len - self.W) if self.W > 0 else new_len
        retire = sorted(b for b in st.pages if (b + 1) * self.B <= ws)
        need = sorted({j // self.B for j in range(lo, new_len)} - set(st.pages))
        return new_len, lo, retire, need

    def _store_rows(self, st: SeqState, stack: torch.Tensor, positions: range) -> None:
        """Compute and store the ctx K/V of the given positions.

        [P1] field fc: c = fc(stack) maps the captured hidden stack into the
        drafter; field hidden_norm: RMSNorm of the projected ctx;
        field fused_kv_weight: one GEMM of c against [L*2*kv_dim, h] gives every
        layer's ctx K and V; the keys then take the layer's k_norm and RoPE at
        their position. reading: values are not normalised; the same c feeds
        every layer (one fused GEMM needs one shared input)."""
        if len(positions) == 0:
            return
        x = stack.to(F64)                                         # bf16 values
        cvec = round_bf16(rms_norm(x @ self.fc.T, self.hidden_norm, self.eps))
        kv = cvec @ self.w_kv.T                                   # [m, L*2*kv]
        pos = torch.tensor(list(positions), dtype=torch.int64)
        for l, lay in enumerate(self.layers):
            base = l * 2 * self.kv
            k = kv[:, base:base + self.kv].reshape(-1, self.nkv, self.d)
            v = kv[:, base + self.kv:base + 2 * self.kv].reshape(-1, self.nkv, self.d)
            k = rope(rms_norm(k, lay["k_norm"], self.eps).transpose(0, 1), pos,
                     self.inv_freq).transpose(0, 1) * self.rope_scale
            k_st, v_st = self._quant_kv(l, k), self._quant_kv(l, v, is_v=True)
            for r, j in enumerate(positions):
                if j not in st.rows:
                    st.rows[j] = (torch.empty(self.L, self.nkv, self.d, dtype=F64),
                                  torch.empty(self.L, self.nkv, self.d, dtype=F64))
                st.rows[j][0][l] = k_st[r]
                st.rows[j][1][l] = v_st[r]

    def _quant_kv(self, l: int, t: torch.Tensor, is_v: bool = False) -> torch.Tensor:
        """Cache storage format: bf16 ([P2] field kv_cache), or FP8 E4M3 codes
        with a static per-(layer, kv head, K|V) scale ([P1] field kv_cache,
        'paged FP8'): code = e4m3(x / s) taken in fp32, read back as code * s."""
        if not self.kv_fp8:
            return round_bf16(t)
        s = self.kv_scale[l, :, 1 if is_v else 0]                  # [nkv] f32
        codes = e4m3_codes(t.to(torch.float32) / s[None, :, None])
        return codes * s.to(F64)[None, :, None]

    def _commit_pages(self, st, retire, need):
        for b in retire:
            self.pool.give(st.pages.pop(b))
        for b in need:
            st.pages[b] = self.pool.take()

    def _drop_retired_rows(self, st, ws):
        for j in [j for j in st.rows if j < (ws // self.B) * self.B]:
            del st.rows[j]

    def prefill(self, st: SeqState, stack: torch.Tensor) -> None:
        """Append n ctx rows (target hiddens of positions ctx_len..ctx_len+n-1).

        reading: the stored rows are computed in chunks of prefill_chunk rows;
        the chunking does not change the values."""
        n = stack.shape[0]
        if st not in self.states:
            raise OracleError("EINVAL", "unknown state")
        if st.pending is not None:
            raise OracleError("ESTATE", "prefill before after_verify")
        new_len, lo, retire, need = self._plan_append(st, n)
        if new_len > st.cap:
            raise OracleError("EINVAL", "ctx beyond state capacity")
        if len(need) > self.pool.n_free() + len(retire):
            raise OracleError("ENOMEM", "KV pool exhausted")
        self._commit_pages(st, retire, need)
        self._drop_retired_rows(st, max(0, new_len - self.W) if self.W > 0 else new_len)
        ch = self.cfg.get("prefill_chunk", 512)
        for a in range(lo, new_len, ch):
            b = min(new_len, a + ch)
            self._store_rows(st, stack[a - st.ctx_len:b - st.ctx_len], range(a, b))
        st.ctx_len = new_len

    # -- the block forward ----------------------------------------------------
    def block_forward(self, st: SeqState, last_token: int, p: int, num_drafts: int,
                      allowed: torch.Tensor | None, taps: dict | None = None):
        """One non-causal block of gamma rows at positions p..p+gamma-1.

        [P1] fields gamma/mask_token_id (block = the last verified token plus
        gamma-1 mask rows), embed_tokens_shared (shared embed table), layers
        (Qwen3-style layer stack), norm (final RMSNorm), lm_head_shared (argmax
        over the block's logits). reading: rows 1..num_drafts give drafts
        1..num_drafts (rows 0..num_drafts-1 with shifted_rows); queries see the
        windowed ctx and every block key."""
        g = self.gamma
        toks = [last_token] + [self.cfg["mask_token_id"]] * (g - 1)
        x = self.embed[torch.tensor(toks)].to(F64)                # [g, H]
        if taps is not None:
            taps["x"] = [x.clone()]
        for l in range(self.L):
            x = self.layer_forward(st, l, x, p)
            if taps is not None:
                taps["x"].append(x.clone())
        z = round_bf16(rms_norm(x, self.norm, self.eps))
        logits = self.draft_logits(z, num_drafts)
        if taps is not None:
            taps["z"] = z
            taps["logits"] = logits
        return select_drafts(logits, allowed)

    def layer_forward(self, st: SeqState, l: int, x: torch.Tensor, p: int) -> torch.Tensor:
        """One Qwen3-style drafter layer over the gamma block rows x [gamma, H]
        at positions p..p+gamma-1, attending to the window's stored ctx rows of
        layer l and the block's own keys ([P1] field layers; the
        mask-free block attention). Returns the new residual."""
        lay = self.layers[l]
        g = x.shape[0]
        pos = torch.arange(p, p + g, dtype=torch.int64)
        ws = max(0, p - self.W) if self.W > 0 else p
        ctx_pos = list(range(ws, p))
        h = round_bf16(rms_norm(x, lay["in_norm"], self.eps))
        q = (h @ lay["q"].T).reshape(g, self.nq, self.d)
        k = (h @ lay["k"].T).reshape(g, self.nkv, self.d)
        v = (h @ lay["v"].T).reshape(g, self.nkv, self.d)
        q = rope(rms_norm(q, lay["q_norm"], self.eps).transpose(0, 1), pos,
                 self.inv_freq).transpose(0, 1) * self.rope_scale
        k = rope(rms_norm(k, lay["k_norm"], self.eps).transpose(0, 1), pos,
                 self.inv_freq).transpose(0, 1) * self.rope_scale
        q, k, v = round_bf16(q), round_bf16(k), round_bf16(v)
        if ctx_pos:
            kc = torch.stack([st.rows[j][0][l] for j in ctx_pos])
            vc = torch.stack([st.rows[j][1][l] for j in ctx_pos])
            keys, vals = torch.cat([kc, k], 0), torch.cat([vc, v], 0)
        else:
            keys, vals = k, v
        o = round_bf16(attention(q, keys, vals).reshape(g, self.nq * self.d))
        x = x + o @ lay["o"].T
        h2 = round_bf16(rms_norm(x, lay["post_norm"], self.eps))
        u = round_bf16(silu(h2 @ lay["gate"].T) * (h2 @ lay["up"].T))
        return x + u @ lay["down"].T

    def draft_logits(self, z: torch.Tensor, num_drafts: int) -> torch.Tensor:
        """lm_head logits of the draft rows of the final-normed z: block rows
        1..num_drafts, or 0..num_drafts-1 with shifted_rows ([P1] field
        lm_head_shared; FP8 mirror: scale_v * <z, codes_v>)."""
        logits = z[self.draft0:self.draft0 + num_drafts] @ self.lm_head().T
        if self.lm_fp8:
            logits = logits * self.lm_scale[None, :]
        return logits

    # -- trait calls ----------------------------------------------------------
    def propose(self, st, last_token, position, new_rows, num_drafts, bitmask=None,
                taps=None):
        """[P3] propose: append the new ctx rows, run the block, return drafts.

        reading: position == ctx_len + n_new (the new rows are the target
        hiddens of positions ctx_len..position-1); after an after_verify(k) the
        next position is p + k + 1."""
        r = self.propose_batch([st], [last_token], [position], [new_rows], num_drafts,
                               None if bitmask is None else bitmask[None, :], taps=taps,
                               _single=True)
        return r[0]

    def _check(self, st, last_token, position, new_rows, num_drafts):
        n_new = 0 if new_rows is None else new_rows.shape[0]
        if st not in self.states:
            raise OracleError("EINVAL", "unknown state")
        if not (1 <= num_drafts <= self.gamma - 1):
            raise OracleError("EINVAL", "num_drafts out of range")
        if not (0 <= last_token < self.V):
            raise OracleError("EINVAL", "token out of range")
        if st.pending is not None:
            raise OracleError("ESTATE", "propose before after_verify")
        if position != st.ctx_len + n_new:
            raise OracleError("EPOSITION", "position != ctx_len + n_new")
        if st.expected_next is not None and position != st.expected_next:
            raise OracleError("EPOSITION", "position != expected next")
        if position > st.cap:
            raise OracleError("EINVAL", "ctx beyond state capacity")
        if self.W > 0 and st.pages and max(0, position - self.W) < min(st.pages) * self.B:
            # only an installed carry can get here: its window would reach
            # below the first page it brought (rows retired before the take)
            raise OracleError("EPOSITION", "window reaches below the installed pages")
        return n_new

    def propose_batch(self, states, last_tokens, positions, new_rows, num_drafts,
                      bitmask=None, taps=None, _single=False):
        """[P1]/[P2]/[P3] propose_batch: per-sequence prep, then one forward for
        every sequence (row i of every slice belongs to sequence i). Declines
        (returns None) for fewer than 2 or more than max_batch sequences.

        reading: all sequences retire first, then take pages, in sequence order;
        a batch that cannot get its pages changes nothing."""
        n = len(states)
        if not _single and (n < 2 or n > self.cfg["max_batch"]):
            return None
        if len(set(map(id, states))) != n:
            raise OracleError("EINVAL", "duplicate state")
        n_news = [self._check(st, t, p, r, num_drafts)
                  for st, t, p, r in zip(states, last_tokens, positions, new_rows)]
        plans = [self._plan_append(st, nn) for st, nn in zip(states, n_news)]
        need = sum(len(pl[3]) for pl in plans)
        retire = sum(len(pl[2]) for pl in plans)
        if need > self.pool.n_free() + retire:
            raise OracleError("ENOMEM", "KV pool exhausted")
        for st, pl in zip(states, plans):
            for b in pl[2]:
                self.pool.give(st.pages.pop(b))
        for st, pl in zip(states, plans):
            for b in pl[3]:
                st.pages[b] = self.pool.take()
        for st, rows, nn, pl in zip(states, new_rows, n_news, plans):
            new_len, lo = pl[0], pl[1]
            self._drop_retired_rows(st, max(0, new_len - self.W) if self.W > 0 else new_len)
            if nn:
                self._store_rows(st, rows[lo - st.ctx_len:], range(lo, new_len))
            st.ctx_len = new_len
        out = []
        for i, (st, t, p) in enumerate(zip(states, last_tokens, positions)):
            allowed = None if bitmask is None else bitmask_allowed(bitmask[i], self.V)
            tp = None
            if taps is not None:
                tp = {}
                taps.setdefault("seq", []).append(tp)
            drafts, n_out, conf, _ = self.block_forward(st, t, p, num_drafts, allowed, tp)
            st.pending = (p, n_out)
            st.expected_next = None
            out.append((drafts, n_out, conf))
        return out

    def after_verify(self, st: SeqState, num_accepted: int) -> None:
        """[P3] after_verify: trim the state to the accepted count.

        reading: the next propose sits at p + k + 1 and brings the k + 1 target
        hiddens of positions p..p+k; pages below that propose's window retire
        now."""
        if st.pending is None:
            raise OracleError("ESTATE", "after_verify without propose")
        p, n_out = st.pending
        if not (0 <= num_accepted <= n_out):
            raise OracleError("EINVAL", "num_accepted out of range")
        st.expected_next = p + num_accepted + 1
        st.pending = None
        ws = max(0, st.expected_next - self.W) if self.W > 0 else st.expected_next
        for b in sorted(b for b in st.pages if (b + 1) * self.B <= ws):
            self.pool.give(st.pages.pop(b))
        self._drop_retired_rows(st, ws)

    def catchup_batch(self, states, rows, first_pos, tokens=None) -> int:
        """[P2]/[P3] catchup_batch (catchup_drafter for one state): append,
        for each state, the ctx rows of target hiddens paired with tokens
        accepted by the last verify, at explicit RoPE positions first_pos[i],
        first_pos[i] + 1, ... Returns the rows appended (their sum).

        reading: this head keeps one ctx row per target position (the row
        space is positions, never compacted), so a state's append slot and
        the RoPE position of its next row coincide: first_pos[i] must equal
        the state's ctx_len. The rows are the ones the next propose would
        otherwise bring as new rows (the last verified token's and those of
        the accepted drafts), so after after_verify(k) at most k + 1 rows fit
        before the expected position. The ctx rows depend on the hiddens
        alone; tokens (when given) are only range-checked. Pages: all states
        retire first, then take pages, in state order; a batch that cannot
        get its pages changes nothing."""
        n = len(states)
        if len(rows) != n or len(first_pos) != n or (tokens is not None and len(tokens) != n):
            raise OracleError("EINVAL", "array lengths differ")
        if len(set(map(id, states))) != n:
            raise OracleError("EINVAL", "duplicate state")
        counts = []
        for i, st in enumerate(states):
            m = 0 if rows[i] is None else rows[i].shape[0]
            if st not in self.states:
                raise OracleError("EINVAL", "unknown state")
            if st.pending is not None:
                raise OracleError("ESTATE", "catch-up before after_verify")
            if tokens is not None and (len(tokens[i]) != m or
                                       any(not (0 <= t < self.V) for t in tokens[i])):
                raise OracleError("EINVAL", "tokens do not pair with the rows")
            if first_pos[i] != st.ctx_len:
                raise OracleError("EPOSITION", "first position != the state's append point")
            if st.expected_next is not None and st.ctx_len + m > st.expected_next:
                raise OracleError("EPOSITION", "rows past the position after_verify set")
            if st.ctx_len + m > st.cap:
                raise OracleError("EINVAL", "ctx beyond state capacity")
            counts.append(m)
        plans = [self._plan_append(st, m) for st, m in zip(states, counts)]
        need = sum(len(pl[3]) for pl in plans)
        retire = sum(len(pl[2]) for pl in plans)
        if need > self.pool.n_free() + retire:
            raise OracleError("ENOMEM", "KV pool exhausted")
        for st, pl in zip(states, plans):
            for b in pl[2]:
                self.pool.give(st.pages.pop(b))
        for st, pl in zip(states, plans):
            for b in pl[3]:
                st.pages[b] = self.pool.take()
        for st, r, m, f, pl in zip(states, rows, counts, first_pos, plans):
            new_len, lo = pl[0], pl[1]
            self._drop_retired_rows(st, max(0, new_len - self.W) if self.W > 0 else new_len)
            if m:
                # explicit positions: row r of the feed sits at first_pos + r
                self._store_rows(st, r[lo - st.ctx_len:], range(f + (lo - st.ctx_len), f + m))
            st.ctx_len = new_len
        return sum(counts)

    # -- drafter-KV carry across turns ----------------------------------------
    def take_drafter_kv(self, st: SeqState):
        """[P3] take_drafter_kv: move the sequence's KV pages out of its state,
        so free_state releases none of them and the caller can carry them to
        the next turn; the state then behaves as freshly allocated. Returns
        (blocks, rows, last_pair_key), or None when there is nothing to carry.

        reading: blocks = physical ids of the live pages in logical order,
        rows = ctx_len (the first live logical page is ceil(rows/B) -
        len(blocks)); the row space is positions, not compacted, so no pair
        key is tracked (None); a propose awaiting after_verify cannot be
        carried (ESTATE)."""
        if st not in self.states:
            raise OracleError("EINVAL", "unknown state")
        if st.pending is not None:
            raise OracleError("ESTATE", "take before after_verify")
        if not st.pages:
            return None
        lo, hi = min(st.pages), max(st.pages)
        blocks = [st.pages[b] for b in range(lo, hi + 1)]
        self.carried[tuple(blocks)] = (st.ctx_len, st.rows)
        st.ctx_len, st.pages, st.rows = 0, {}, {}
        st.pending, st.expected_next = None, None
        return blocks, self.carried[tuple(blocks)][0], None

    def install_drafter_kv(self, st: SeqState, blocks, rows: int, last_pair_key=None) -> bool:
        """[P3] install_drafter_kv: the inverse of take_drafter_kv, into a
        fresh state. reading: the state then holds ctx_len = rows with the
        carried pages as its live window; the next propose brings the rows of
        positions rows..position-1 and may not place its window below the
        first carried page. A bad bundle or a state that is not fresh is an
        error that changes nothing (the caller still owns the pages)."""
        key = tuple(int(b) for b in blocks)
        if st not in self.states:
            raise OracleError("EINVAL", "unknown state")
        if key not in self.carried or self.carried[key][0] != rows:
            raise OracleError("EINVAL", "pages not carried with these rows")
        if st.ctx_len or st.pages or st.pending is not None or st.expected_next is not None:
            raise OracleError("EINVAL", "state is not fresh")
        if rows > st.cap:
            raise OracleError("EINVAL", "rows beyond state capacity")
        _, kv = self.carried.pop(key)
        b0 = -(-rows // self.B) - len(key)
        st.pages = {b0 + i: p for i, p in enumerate(key)}
        st.rows, st.ctx_len = kv, rows
        return True

    def free_drafter_kv(self, blocks) -> None:
        """[P3] free_drafter_kv: release carried pages that no state owns."""
        key = tuple(int(b) for b in blocks)
        if key not in self.carried:
            raise OracleError("EINVAL", "pages not carried")
        del self.carried[key]
        for p in key:
            self.pool.give(p)

    # -- views for parity checks ---------------------------------------------
    def block_table(self, st: SeqState):
        """(ctx_len, first live logical page, physical ids of the live pages)."""
        if not st.pages:
            return st.ctx_len, -1, []
        lo, hi = min(st.pages), max(st.pages)
        return st.ctx_len, lo, [st.pages.get(b, -1) for b in range(lo, hi + 1)]

    def gather_kv(self, st: SeqState, layer: int, positions):
        """Stored K, V of one layer at the given positions: [n, nkv, d] each."""
        k = torch.stack([st.rows[j][0][layer] for j in positions])
        v = torch.stack([st.rows[j][1][layer] for j in positions])
        return k, v
