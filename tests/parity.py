"""Shared helpers of the GPU parity tests: build the oracle and the library
head from the same seeded CPU weights, and compare results with the
tolerances of the parity gate:
  * block tables, ctx_len, first page: bit-exact;
  * residual taps, final z, gathered ctx K/V: max-abs 3e-2;
  * logits: per row max|diff| / max|ref| <= 2e-2 (5e-2 on FP8 paths);
  * draft ids: exact wherever the oracle's masked top-1 - top-2 gap > 1e-2;
  * confidence: |diff| <= 1e-2 end to end; and, teacher-forced (the
    oracle's logits from the GPU's own final-normed rows), every draft row's
    top-1 probability and the chain minimum within 1e-2 relative.
Deep stacks are compared layer by layer (teacher-forced), see E2E_* below."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from block_diffusion_speculative_forward_gb300 import binding as B
from block_diffusion_speculative_forward_gb300 import synthetic as syn

HIDDEN_TOL = 3e-2
LOGIT_TOL = 2e-2
LOGIT_TOL_FP8 = 5e-2
GAP = 1e-2
CONF_TOL = 1e-2
# Teacher-forced top-1 probabilities (oracle logits from the GPU's own z):
# relative, so that probabilities of 1e-3 .. 1e-6 (random weights, full
# vocab) are checked as strictly as probabilities near one.
CONF_REL = 1e-2
P1_FLOOR = 1e-12
# End to end over many layers, an fp32 evaluation of the method drifts from the
# fp64 oracle (measured: the oracle in fp32 vs fp64 at the shipped geometry,
# 8 layers: max residual diff 0.09, logits ~1.3% of max|l|). End-to-end
# logits get this envelope; drafts are compared where the gap exceeds it.
E2E_LOGIT_TOL = 5e-2
E2E_GAP = 0.25


def cfg_for(geom, **kw):
    c = dict(num_layers=geom.num_layers, hidden=geom.hidden, intermediate=geom.intermediate,
             num_q_heads=geom.num_q_heads, num_kv_heads=geom.num_kv_heads,
             head_dim=geom.head_dim, vocab=geom.vocab, gamma=geom.gamma,
             mask_token_id=geom.mask_token_id, n_target_layers=geom.n_target_layers,
             target_hidden=geom.target_hidden, rms_eps=geom.rms_eps,
             ctx_window=geom.ctx_window, kv_block=geom.kv_block,
             prefill_chunk=geom.prefill_chunk, max_batch=4, max_seq_len=9216,
             kv_pool_blocks=0, kv_dtype=0, lm_head_dtype=0)
    c.update(kw)
    return c


class Pair:
    """Oracle and library heads over the same weights."""

    def __init__(self, geom, seed, cfg_kw=None, lm_fp8=False, kv_fp8=False, taps=True,
                 max_rows=None, lm_nvfp4=False):
        self.geom = geom
        self.cfg = cfg_for(geom, **(cfg_kw or {}), kv_dtype=int(kv_fp8),
                           lm_head_dtype=2 if lm_nvfp4 else int(lm_fp8))
        self.w = syn.make_weights(geom, seed, lm_head_fp8=lm_fp8, kv_fp8=kv_fp8,
                                  lm_head_nvfp4=lm_nvfp4)
        self.ora = oracle.DraftHeadOracle(self.cfg, self.w)
        self.wd = B.weights_to_device(self.w)
        self.lib = B.DraftHead(self.cfg, self.wd)
        self.fp8 = lm_fp8 or kv_fp8
        if taps:
            rows = max_rows or self.cfg["max_batch"] * geom.gamma
            self.tx = torch.zeros((geom.num_layers + 1, rows, geom.hidden), device="cuda")
            self.tz = torch.zeros((rows, geom.hidden), dtype=torch.bfloat16, device="cuda")
            self.tl = torch.zeros((rows, geom.vocab), device="cuda")
            self.lib.set_taps(self.tx, self.tz, self.tl)


def gaps(logits: torch.Tensor, allowed) -> torch.Tensor:
    lg = logits.to(torch.float64)
    if allowed is not None:
        lg = torch.where(allowed[None, :], lg, torch.full_like(lg, -math.inf))
    top = torch.topk(lg, 2, dim=1).values
    return top[:, 0] - top[:, 1]


def check_drafts(ref_drafts, got_drafts, ref_logits, allowed):
    g = gaps(ref_logits, allowed)
    n_checked = 0
    for i, (a, b) in enumerate(zip(ref_drafts, got_drafts)):
        if g[i] > GAP:
            assert a == b, f"draft {i}: oracle {a} gpu {b} (gap {float(g[i]):.4f})"
            n_checked += 1
    return n_checked


def check_logits(ref: torch.Tensor, got: torch.Tensor, tol: float):
    ref = ref.to(torch.float64).cpu()
    got = got.to(torch.float64).cpu()
    for i in range(ref.shape[0]):
        rel = float((ref[i] - got[i]).abs().max() / ref[i].abs().max())
        assert rel <= tol, f"logit row {i}: rel err {rel:.3e} > {tol}"


def check_abs(ref, got, tol, what):
    ref = torch.as_tensor(ref).to(torch.float64).cpu()
    got = torch.as_tensor(got).to(torch.float64).cpu()
    err = float((ref - got).abs().max())
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol}"
    return err


def check_rows(lg_ref, allowed, ids, p1, got_out=None):
    """The lm_head stage row by row, teacher-forced: lg_ref are the oracle's
    logits of the draft rows computed from the GPU's own final-normed rows, so
    the only difference left is the stage's own arithmetic (the GEMM's fp32
    accumulation and the per-tile max / argmax / sum-exp merge). Every row's
    id matches where the top-1/top-2 gap exceeds GAP (elsewhere the GPU's id
    must be within GAP of the max); every row's top-1 probability and the
    chain confidence match within CONF_REL relative. Returns the p1 values."""
    d_ref, n_ref, c_ref, p1_ref = oracle.select_drafts(lg_ref, allowed)
    lg = lg_ref.to(torch.float64)
    if allowed is not None:
        lg = torch.where(allowed[None, :], lg, torch.full_like(lg, -math.inf))
    g = gaps(lg_ref, allowed)
    for i in range(n_ref):
        if g[i] > GAP:
            assert ids[i] == d_ref[i], f"row {i}: id {ids[i]} vs oracle {d_ref[i]} (gap {float(g[i]):.4f})"
        else:
            assert 0 <= ids[i] < lg.shape[1] and float(lg[i].max() - lg[i, ids[i]]) <= GAP, \
                f"row {i}: id {ids[i]} is not within {GAP} of the row's max"
        rel = abs(p1[i] - p1_ref[i]) / max(p1_ref[i], P1_FLOOR)
        assert rel <= CONF_REL, f"row {i}: p1 {p1[i]:.6e} vs oracle {p1_ref[i]:.6e} (rel {rel:.2e})"
    for i in range(n_ref, len(ids)):
        assert ids[i] == -1 and p1[i] == 0.0, f"row {i} after the chain ended: {ids[i]}, {p1[i]}"
    if got_out is not None:
        got_d, got_n, got_c = got_out
        assert got_n == n_ref, (got_n, n_ref)
        if got_c is not None:
            ref_c = min(p1_ref[:n_ref]) if n_ref else 0.0
            assert abs(got_c - ref_c) <= CONF_REL * max(ref_c, P1_FLOOR), (got_c, ref_c)
    return p1_ref


def check_seq(pair: Pair, ref_tap: dict, ref_out, got_out, seq_idx: int, n_seq: int,
              nd: int, allowed=None, hidden=True):
    """Compare one sequence of a propose call: taps, logits, drafts, conf."""
    g = pair.geom.gamma
    torch.cuda.synchronize()
    if hidden:
        R, H, L = n_seq * g, pair.geom.hidden, pair.geom.num_layers
        tx = pair.tx.reshape(-1)[:(L + 1) * R * H].reshape(L + 1, R, H)
        for l, xr in enumerate(ref_tap["x"]):
            check_abs(xr, tx[l, seq_idx * g:(seq_idx + 1) * g], HIDDEN_TOL, f"x tap {l}")
        check_abs(ref_tap["z"], pair.tz[seq_idx * g:(seq_idx + 1) * g].float(), HIDDEN_TOL, "z")
    got_logits = pair.tl[seq_idx * nd:(seq_idx + 1) * nd]
    check_logits(ref_tap["logits"], got_logits, LOGIT_TOL_FP8 if pair.fp8 else LOGIT_TOL)
    ref_d, ref_n, ref_c = ref_out
    got_d, got_n, got_c = got_out
    assert ref_n == got_n
    n = check_drafts(ref_d[:ref_n], got_d[:got_n], ref_tap["logits"], allowed)
    if got_c is not None:
        assert abs(ref_c - got_c) <= CONF_TOL, (ref_c, got_c)
    # the lm_head stage teacher-forced from the GPU's own final-normed rows
    g = pair.geom.gamma
    ids, p1 = pair.lib.debug_rows(n_seq * nd)
    z_got = pair.tz[seq_idx * g:(seq_idx + 1) * g].double().cpu()
    check_rows(pair.ora.draft_logits(z_got, nd), allowed, ids[seq_idx * nd:(seq_idx + 1) * nd],
               p1[seq_idx * nd:(seq_idx + 1) * nd], got_out)
    return n


def check_kv(pair: Pair, so, sl, positions):
    """Gathered ctx K/V of every layer at the given positions (any order);
    the library gathers contiguous runs."""
    positions = sorted(positions)
    runs, start = [], 0
    for i in range(1, len(positions) + 1):
        if i == len(positions) or positions[i] != positions[i - 1] + 1:
            runs.append(positions[start:i])
            start = i
    for run in runs:
        _check_kv_run(pair, so, sl, run)


def _check_kv_run(pair: Pair, so, sl, positions):
    for l in range(pair.geom.num_layers):
        k, v = pair.lib.gather_kv(sl, l, positions[0], len(positions))
        kr, vr = pair.ora.gather_kv(so, l, positions)
        if pair.cfg["kv_dtype"] == 1:
            check_fp8_kv(pair, l, kr, k, 0)
            check_fp8_kv(pair, l, vr, v, 1)
        else:
            check_abs(kr, k, HIDDEN_TOL, f"ctx K layer {l}")
            check_abs(vr, v, HIDDEN_TOL, f"ctx V layer {l}")


def e4m3_step(x: torch.Tensor) -> torch.Tensor:
    """Spacing of E4M3 codes just below |x| and at |x| (3 mantissa bits,
    subnormal spacing 2^-9 below 2^-6): the larger of the two."""
    a = x.abs().clamp(min=2.0 ** -6)
    e = torch.floor(torch.log2(a))
    at = torch.pow(2.0, e - 3)
    below = torch.where(a == torch.pow(2.0, e), torch.pow(2.0, e - 4), at)
    return torch.maximum(torch.maximum(at, below), torch.full_like(at, 2.0 ** -9))


def check_fp8_kv(pair, l, ref, got, kind, max_frac=5e-3):
    """FP8 cache: each dequantised value within the FP8-path tolerance
    (max-abs 5e-2), or its code exactly one E4M3 step from the oracle's (a
    rounding decision on either side of a midpoint: the two sides' fp32
    inputs differ by summation order and by bf16 flips of the ctx rows, about
    1e-4 absolute). Measured at the shipped geometry: ~1e-3 of the codes
    differ."""
    s = pair.w["kv_scale"][l, :, kind].to(torch.float64)[None, :, None]
    ref = ref.to(torch.float64).cpu()
    got = got.to(torch.float64).cpu()
    rc, gc = ref / s, got / s
    diff = (rc - gc).abs()
    bad = diff > 1e-5 * rc.abs().clamp(min=1.0)     # beyond the fp32 dequant rounding
    frac = float(bad.double().mean())
    step = torch.maximum(e4m3_step(rc), e4m3_step(gc))
    far = (diff > step * (1 + 1e-5)) & ((ref - got).abs() > LOGIT_TOL_FP8)
    if bool(far.any()):
        i = tuple(torch.nonzero(far)[0].tolist())
        raise AssertionError(f"FP8 KV layer {l} kind {kind}: codes {float(rc[i])} vs "
                             f"{float(gc[i])} differ by more than one step and 5e-2 at {i}")
    assert frac <= max_frac, f"FP8 KV: {frac:.2e} of codes differ"


def assert_tables(pair, so, sl):
    assert pair.lib.debug_state(sl) == pair.ora.block_table(so)
