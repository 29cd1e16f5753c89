"""GPU parity of the low-precision lm_heads ([P1] fields lm_head_shared_fp8
and lm_head_nvfp4): FP8 E4M3 codes with per-row scales and NVFP4 (E2M1
codes, E4M3 scales per 16 elements, a global scale). Up to 16 draft rows the
codes stream and are dequantised on chip into tensor memory; wider proposes
multiply by the table widened to bf16 once. The oracle multiplies by the
dequantised table in float64.

Both dequantisations are exact (every E4M3 value and every E2M1 x E4M3
product is a bf16 and an f16 value), so the logits match the oracle's to the
fp32 accumulation of a 16-bit GEMM: the bf16 tolerance applies, not the FP8
one. Covered: one sequence (the streamed kernel), 24 / 72 / 144 draft rows
(the widened table on the few-row GEMM and on the many-row kernel, with
bitmasks), the debug logit tap, and the shipped geometry with sharpened
logits (top-1 probabilities across 1e-3 .. 1), teacher-forced from the GPU's
own final-normed rows."""
import pytest
import torch

import oracle
from block_diffusion_speculative_forward_gb300 import binding as B
from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.parity import LOGIT_TOL, Pair, cfg_for, check_logits, check_rows, check_seq
from tests.test_gpu_confidence import SHARP, _check_lm_stage

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_diffusion_speculative_forward_gb300 import build
    build.build()


def _pair(fmt, seed, **kw):
    return Pair(syn.TINY, seed, lm_fp8=fmt == "fp8", lm_nvfp4=fmt == "nvfp4", **kw)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_tiny_single_sequence(fmt):
    pair = _pair(fmt, 1301)
    so, sl = pair.ora.alloc_state(), pair.lib.alloc_state()
    stack = syn.make_stack(syn.TINY, 50, 1301)
    pair.ora.prefill(so, stack)
    pair.lib.prefill(sl, stack.cuda())
    taps = {}
    ref = pair.ora.propose(so, 3, 50, None, 3, taps=taps)
    got = pair.lib.propose(sl, 3, 50, None, 3)
    torch.cuda.synchronize()
    # exact dequantisation: the bf16 bar, not the FP8 one
    check_logits(taps["seq"][0]["logits"], pair.tl[:3], LOGIT_TOL)
    check_seq(pair, taps["seq"][0], ref, got, 0, 1, 3)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("n", [8, 24, 48])
def test_tiny_many_rows(fmt, n):
    """n sequences x 3 drafts: 24, 72 or 144 draft rows over the widened
    table, with a bitmask per sequence."""
    pair = _pair(fmt, 1303 + n, cfg_kw=dict(max_batch=n))
    ctx = syn.uniform_ints(5, 30, n, 1303, 1)
    so, sl = [], []
    for i, c in enumerate(ctx):
        a, b = pair.ora.alloc_state(), pair.lib.alloc_state()
        st = syn.make_stack(syn.TINY, c, 1303, idx=i)
        pair.ora.prefill(a, st)
        pair.lib.prefill(b, st.cuda())
        so.append(a)
        sl.append(b)
    toks = syn.uniform_ints(0, syn.TINY.vocab - 1, n, 1303, 2)
    masks = syn.make_bitmask(syn.TINY.vocab, n, 1303)
    taps = {}
    ref = pair.ora.propose_batch(so, toks, ctx, [None] * n, 3, bitmask=masks, taps=taps)
    got = pair.lib.propose_batch(sl, toks, ctx, [None] * n, 3, bitmask=masks.cuda())
    for i in sorted({0, 7, n - 1}):
        allowed = oracle.bitmask_allowed(masks[i], syn.TINY.vocab)
        check_seq(pair, taps["seq"][i], ref[i], got[i], i, n, 3, allowed=allowed)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("masked", [False, True])
def test_full_geometry_sharp(fmt, masked):
    """The shipped geometry, batch 1, 15 drafts, codes quantised from a
    sharpened table: drafts and per-row probabilities teacher-forced."""
    geom, seed, nd = syn.FULL, 1311, 15
    cfg = cfg_for(geom, max_batch=1, max_seq_len=256,
                  lm_head_dtype=1 if fmt == "fp8" else 2)
    w = syn.make_weights(geom, seed, lm_head_fp8=fmt == "fp8", lm_head_nvfp4=fmt == "nvfp4")
    w["norm"] = (w["norm"].to(torch.float32) * SHARP).to(torch.bfloat16)
    ora = oracle.DraftHeadOracle(cfg, w)
    # the streamed head needs no bf16 table: none is passed
    wd = B.weights_to_device({k: v for k, v in w.items() if k != "lm_head"} |
                             {"lm_head": torch.empty(0, dtype=torch.bfloat16)})
    head = B.DraftHead(cfg, wd)
    g = geom.gamma
    tz = torch.zeros((g, geom.hidden), dtype=torch.bfloat16, device="cuda")
    tl = torch.zeros((nd, geom.vocab), device="cuda")
    head.set_taps(None, tz, tl)
    st = head.alloc_state()
    head.prefill(st, syn.make_stack(geom, 40, seed).cuda())
    masks = syn.make_bitmask(geom.vocab, 1, seed) if masked else None
    got = head.propose(st, 4244, 41, syn.make_stack(geom, 1, seed, idx=1).cuda(), nd,
                       bitmask=None if masks is None else masks[0].cuda())
    torch.cuda.synchronize()
    _check_lm_stage(head, ora, tz, tl, [0], 1, nd, masks, g, [got])
    head.close()
