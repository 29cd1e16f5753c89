"""GPU parity of the DSpark conventions ([P1]/[P2] field shifted_rows; [P2]
catchup_batch, [P3] catchup_drafter) through the C ABI against the oracle.

Shifted rows change which block rows reach the lm_head (0..nd-1 instead of
1..nd): covered on the kernel-per-step path, inside the chained launch, on the
many-row lm_head kernel (more than 64 draft rows) and at the shipped geometry
with sharpened logits. Catch-up appends ctx rows between a verify and the next
propose: rounds with every split of the k + 1 rows between the catch-up feed
and the propose's new rows, one and several states per call."""
from dataclasses import replace

import pytest
import torch

import oracle
from block_diffusion_speculative_forward_gb300 import binding as B
from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.parity import Pair, assert_tables, cfg_for, check_kv, check_seq
from tests.test_gpu_confidence import _check_lm_stage, _sharp_weights
from tests.test_oracle_pins import MICRO

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_diffusion_speculative_forward_gb300 import build
    build.build()


def _prefill(pair, n_rows, seed, idx=0):
    so, sl = pair.ora.alloc_state(), pair.lib.alloc_state()
    stack = syn.make_stack(pair.geom, n_rows, seed, idx)
    pair.ora.prefill(so, stack)
    pair.lib.prefill(sl, stack.cuda())
    return so, sl


def _propose(pair, so, sl, tok, pos, rows, nd):
    taps = {}
    ref = pair.ora.propose(so, tok, pos, rows, nd, taps=taps)
    got = pair.lib.propose(sl, tok, pos, None if rows is None else rows.cuda(), nd)
    return taps["seq"][0], ref, got


@pytest.mark.parametrize("chained", [False, True])
def test_shifted_rows_rounds(chained):
    pair = Pair(syn.TINY, 1201, cfg_kw=dict(shifted_rows=1))
    pair.lib.set_chain(chained)
    so, sl = _prefill(pair, 45, 1201)
    rows = syn.make_stack(syn.TINY, 20, 1201, idx=4)
    p, n_new, used = 45, 0, 0
    for k in [2, 0, 3, 1]:
        r = rows[used:used + n_new] if n_new else None
        used += n_new
        tap, ref, got = _propose(pair, so, sl, (11 * p) % syn.TINY.vocab, p, r, 3)
        assert pair.lib.last_path_chained() == chained
        check_seq(pair, tap, ref, got, 0, 1, 3)
        pair.ora.after_verify(so, k)
        pair.lib.after_verify(sl, k)
        p, n_new = p + k + 1, k + 1
    assert_tables(pair, so, sl)


def test_shifted_rows_many_row_lm_head():
    """24 sequences x 3 drafts = 72 draft rows: the many-row lm_head kernel."""
    n = 24
    pair = Pair(syn.TINY, 1203, cfg_kw=dict(shifted_rows=1, max_batch=n))
    ctx = syn.uniform_ints(5, 40, n, 1203, 1)
    so, sl = [], []
    for i, c in enumerate(ctx):
        a, b = _prefill(pair, c, 1203, idx=i)
        so.append(a)
        sl.append(b)
    toks = syn.uniform_ints(0, syn.TINY.vocab - 1, n, 1203, 2)
    taps = {}
    ref = pair.ora.propose_batch(so, toks, ctx, [None] * n, 3, taps=taps)
    got = pair.lib.propose_batch(sl, toks, ctx, [None] * n, 3)
    for i in (0, 5, 17, 23):
        check_seq(pair, taps["seq"][i], ref[i], got[i], i, n, 3)


@pytest.mark.parametrize("chained", [False, True])
def test_shifted_rows_full_geometry(chained):
    """The shipped geometry, batch 1, sharpened logits (top-1 probabilities
    spread over 1e-3 .. 1): drafts and probabilities of block rows 0..14."""
    geom, seed, nd = syn.FULL, 1205, 15
    cfg = cfg_for(geom, max_batch=1, max_seq_len=256, shifted_rows=1)
    w = _sharp_weights(geom, seed)
    ora = oracle.DraftHeadOracle(cfg, w)
    head = B.DraftHead(cfg, B.weights_to_device(w))
    head.set_chain(chained)
    g = geom.gamma
    tz = torch.zeros((g, geom.hidden), dtype=torch.bfloat16, device="cuda")
    tl = torch.zeros((nd, geom.vocab), device="cuda")
    head.set_taps(None, tz, tl)
    st = head.alloc_state()
    head.prefill(st, syn.make_stack(geom, 40, seed).cuda())
    got = head.propose(st, 4243, 41, syn.make_stack(geom, 1, seed, idx=1).cuda(), nd)
    torch.cuda.synchronize()
    assert head.last_path_chained() == chained
    _check_lm_stage(head, ora, tz, tl, [0], 1, nd, None, g, [got])
    head.close()


@pytest.mark.parametrize("window", [24, 0])
def test_catchup_rounds(window):
    """Rounds on one state: propose, verify accepts k, the first j of the
    k + 1 rows through the catch-up feed, the rest as new rows."""
    geom = replace(MICRO, ctx_window=window)
    pair = Pair(geom, 1207)
    so, sl = _prefill(pair, 37, 1207)
    rows = syn.make_stack(geom, 200, 1207, idx=1)
    p, pend, used = 37, 0, 0
    for k, j in [(3, 4), (0, 1), (2, 0), (3, 2), (1, 2), (2, 3), (0, 0)]:
        r = rows[used:used + pend] if pend else None
        used += pend
        tap, ref, got = _propose(pair, so, sl, (5 * p) % geom.vocab, p, r, 3)
        check_seq(pair, tap, ref, got, 0, 1, 3)
        pair.ora.after_verify(so, k)
        pair.lib.after_verify(sl, k)
        j = min(j, k + 1)
        feed = rows[used:used + j] if j else None
        used += j
        first = so.ctx_len
        assert pair.ora.catchup_batch([so], [feed], [first]) == j
        assert pair.lib.catchup_batch([sl], [None if feed is None else feed.cuda()], [first],
                                      tokens=[[1] * j]) == j
        assert_tables(pair, so, sl)
        p, pend = p + k + 1, k + 1 - j
    live = [q for q in range(so.ctx_len) if q in so.rows]
    check_kv(pair, so, sl, live)


def test_catchup_batch_three_states():
    geom = replace(MICRO, ctx_window=24)
    pair = Pair(geom, 1209, cfg_kw=dict(max_batch=4))
    ctx = [9, 30, 17]
    so, sl = [], []
    for i, c in enumerate(ctx):
        a, b = _prefill(pair, c, 1209, idx=i)
        so.append(a)
        sl.append(b)
    for rnd, counts in enumerate([[2, 0, 5], [1, 9, 3]]):
        feeds = [syn.make_stack(geom, m, 1209, idx=50 + 3 * rnd + i) if m else None
                 for i, m in enumerate(counts)]
        first = [s.ctx_len for s in so]
        assert pair.ora.catchup_batch(so, feeds, first) == sum(counts)
        assert pair.lib.catchup_batch(sl, [None if f is None else f.cuda() for f in feeds],
                                      first) == sum(counts)
        for a, b in zip(so, sl):
            assert_tables(pair, a, b)
    for a, b in zip(so, sl):
        check_kv(pair, a, b, [q for q in range(a.ctx_len) if q in a.rows])
    taps = {}
    pos = [s.ctx_len for s in so]
    ref = pair.ora.propose_batch(so, [3, 4, 5], pos, [None] * 3, 3, taps=taps)
    got = pair.lib.propose_batch(sl, [3, 4, 5], pos, [None] * 3, 3)
    for i in range(3):
        check_seq(pair, taps["seq"][i], ref[i], got[i], i, 3, 3)
