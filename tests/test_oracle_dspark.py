"""Pins of the oracle's DSpark conventions ([P1]/[P2] field shifted_rows;
[P2] catchup_batch, [P3] catchup_drafter) against facts that do not come from
the code under test.

Shifted rows: the block forward is unchanged, and the draft vector is the
argmax vector of all gamma block rows rotated right by one, read from index
1 on. The argmax vector here is recomputed from the oracle's final-normed rows
by a plain numpy product with the lm_head table and a first-maximum scan, so a
wrong row offset, a left rotation or a dropped row fails.

Catch-up: rows appended at explicit RoPE positions equal a prefill of the
same rows on a fresh state, and in a round they equal the rows the next
propose would otherwise bring; the page ids follow the position-by-position
simulator (written separately from the oracle's planner)."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.test_oracle_pins import MICRO, cfg_of
from tests.test_oracle_state import PositionSim

G = MICRO.gamma


def heads(seed, **kw):
    w = syn.make_weights(MICRO, seed)
    return (oracle.DraftHeadOracle(cfg_of(MICRO, **kw), w),
            oracle.DraftHeadOracle(cfg_of(MICRO, shifted_rows=1, **kw), w), w)


def all_rows_argmax(z, w, allowed=None):
    """Argmax (first maximum) and top-1 probability of every block row."""
    lg = z.double().numpy() @ w["lm_head"].double().numpy().T
    if allowed is not None:
        lg = np.where(allowed.numpy()[None, :], lg, -np.inf)
    ids = lg.argmax(1)
    srt = np.sort(lg, 1)
    gap = srt[:, -1] - srt[:, -2]
    m = lg.max(1, keepdims=True)
    p1 = 1.0 / np.exp(lg - m).sum(1)
    return [int(i) for i in ids], p1, gap


def run(h, seed, P, nd, bitmask=None):
    st = h.alloc_state()
    h.prefill(st, syn.make_stack(MICRO, P, seed))
    t = {}
    r = h.propose(st, 17, P, None, nd, bitmask=bitmask, taps=t)
    return r, t["seq"][0]


@pytest.mark.parametrize("seed,P", [(31, 20), (32, 9), (33, 41)])
def test_shifted_drafts_are_the_argmax_vector_rotated_right(seed, P):
    h0, h1, w = heads(seed)
    (d0, n0, c0), t0 = run(h0, seed, P, G - 1)
    (d1, n1, c1), t1 = run(h1, seed, P, G - 1)
    # the convention changes which rows are read, not the block forward
    assert torch.equal(t0["z"], t1["z"])
    for a, b in zip(t0["x"], t1["x"]):
        assert torch.equal(a, b)
    a, p1, gap = all_rows_argmax(t0["z"], w)
    assert np.all(gap > 1e-9)              # the first-maximum scan is unambiguous
    rot = a[-1:] + a[:-1]                  # rotate right by one
    assert d1 == rot[1:] == a[:G - 1] and n1 == G - 1
    assert d0 == a[1:] and n0 == G - 1
    assert d1[1:] == d0[:-1]               # same forward: shifted by one row
    assert abs(c1 - min(p1[:G - 1])) <= 1e-12 * max(1.0, c1)
    assert abs(c0 - min(p1[1:])) <= 1e-12 * max(1.0, c0)


def test_shifted_prefix_and_masks():
    h0, h1, w = heads(34)
    # fewer drafts: the first rows of the rotated vector
    (d, n, _), t = run(h1, 34, 15, 2)
    a, _, _ = all_rows_argmax(t["z"], w)
    assert n == 2 and d == a[:2]
    # a random bitmask: the masked argmax of rows 0..nd-1
    mask = syn.make_bitmask(MICRO.vocab, 1, 34)[0]
    allowed = oracle.bitmask_allowed(mask, MICRO.vocab)
    (d, n, c), t = run(h1, 34, 15, G - 1, bitmask=mask)
    a, p1, _ = all_rows_argmax(t["z"], w, allowed)
    assert n == G - 1 and d == a[:G - 1]
    assert abs(c - min(p1[:G - 1])) <= 1e-12
    # one allowed token: every draft is that token with probability one
    one = torch.zeros_like(mask)
    one[77 >> 5] = 1 << (77 & 31)
    (d, n, c), _ = run(h1, 34, 15, G - 1, bitmask=one)
    assert d == [77] * (G - 1) and n == G - 1 and c == 1.0


def same_kv(h1, s1, h2, s2, positions):
    for l in range(MICRO.num_layers):
        a, b = h1.gather_kv(s1, l, positions), h2.gather_kv(s2, l, positions)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("n", [1, 7, 8, 23, 37])
def test_catchup_on_a_fresh_state_is_a_prefill(n):
    """Rows at positions 0..n-1 through the catch-up feed equal a prefill of
    them: block table, stored K/V (the window's rows only, n = 37 > W = 24)
    and the next propose."""
    w = syn.make_weights(MICRO, 35)
    ha = oracle.DraftHeadOracle(cfg_of(MICRO), w)
    hb = oracle.DraftHeadOracle(cfg_of(MICRO), w)
    rows = syn.make_stack(MICRO, n, 35)
    sa, sb = ha.alloc_state(), hb.alloc_state()
    assert ha.catchup_batch([sa], [rows], [0], tokens=[list(range(n))]) == n
    hb.prefill(sb, rows)
    assert ha.block_table(sa) == hb.block_table(sb)
    ws = max(0, n - MICRO.ctx_window)
    same_kv(ha, sa, hb, sb, range(ws, n))
    ta, tb = {}, {}
    assert ha.propose(sa, 3, n, None, G - 1, taps=ta) == hb.propose(sb, 3, n, None, G - 1, taps=tb)
    assert torch.equal(ta["seq"][0]["logits"], tb["seq"][0]["logits"])


@pytest.mark.parametrize("P", [15, 16, 22, 30])
@pytest.mark.parametrize("k", list(range(G)))
def test_catchup_then_propose_equals_propose_with_rows(P, k):
    """A round: propose at P, the verify accepts k drafts, then the k + 1
    rows of positions P..P+k come through the catch-up feed (all of them, or
    the first j with the rest as the propose's new rows) instead of as the
    next propose's new rows. Every result is the same; page boundaries at 8,
    16, 24 are crossed by some of the cases."""
    w = syn.make_weights(MICRO, 36)
    stack = syn.make_stack(MICRO, P + k + 1, 36)
    for j in range(0, k + 2):
        ha = oracle.DraftHeadOracle(cfg_of(MICRO), w)
        hb = oracle.DraftHeadOracle(cfg_of(MICRO), w)
        sa, sb = ha.alloc_state(), hb.alloc_state()
        for h, s in ((ha, sa), (hb, sb)):
            h.prefill(s, stack[:P])
            h.propose(s, 5, P, None, G - 1)
            h.after_verify(s, k)
        got = ha.catchup_batch([sa], [stack[P:P + j]], [P])
        assert got == j
        rest = stack[P + j:P + k + 1] if j < k + 1 else None
        ta, tb = {}, {}
        ra = ha.propose(sa, 9, P + k + 1, rest, G - 1, taps=ta)
        rb = hb.propose(sb, 9, P + k + 1, stack[P:P + k + 1], G - 1, taps=tb)
        assert ra == rb
        assert torch.equal(ta["seq"][0]["logits"], tb["seq"][0]["logits"])
        assert ha.block_table(sa) == hb.block_table(sb)
        ws = max(0, P + k + 1 - MICRO.ctx_window)
        same_kv(ha, sa, hb, sb, range(ws, P + k + 1))


def test_catchup_batch_pages_follow_the_simulator():
    """Several states in one call, counts including zero: pages retire for
    every state first, then new pages go to the states in order, lowest free
    id first (the position-by-position simulator's rule)."""
    geom = replace(MICRO, ctx_window=40, kv_block=8)
    w = syn.make_weights(geom, 37)
    h = oracle.DraftHeadOracle(cfg_of(geom, max_batch=4), w)
    sim = PositionSim(h.pool.n_pages, 8, 40)
    ctx = [13, 40, 7, 29]
    sts = []
    for i, c in enumerate(ctx):
        st = h.alloc_state()
        h.prefill(st, syn.make_stack(geom, c, 37, idx=i))
        sim.new(i)
        sim.step([i], [c])
        sts.append(st)
    for rnd, counts in enumerate([[3, 0, 9, 1], [8, 5, 0, 16], [1, 1, 1, 1]]):
        rows = [syn.make_stack(geom, m, 37, idx=100 + 4 * rnd + i) if m else None
                for i, m in enumerate(counts)]
        assert h.catchup_batch(sts, rows, [s.ctx_len for s in sts]) == sum(counts)
        sim.step(list(range(4)), counts)
        for i, st in enumerate(sts):
            assert h.block_table(st) == sim.table(i)


def expect(code, fn):
    with pytest.raises(oracle.OracleError) as e:
        fn()
    assert e.value.code == code


def test_catchup_errors_change_nothing():
    w = syn.make_weights(MICRO, 38)
    h = oracle.DraftHeadOracle(cfg_of(MICRO, kv_pool_blocks=6), w)
    s1, s2 = h.alloc_state(), h.alloc_state()
    rows = syn.make_stack(MICRO, 20, 38)
    h.prefill(s1, rows[:18])
    before = (h.block_table(s1), h.block_table(s2), h.pool.n_free())
    expect("EPOSITION", lambda: h.catchup_batch([s1], [rows[:2]], [19]))
    expect("EPOSITION", lambda: h.catchup_batch([s1], [rows[:2]], [17]))
    expect("EINVAL", lambda: h.catchup_batch([s1, s1], [rows[:1], rows[:1]], [18, 18]))
    expect("EINVAL", lambda: h.catchup_batch([s1], [rows[:2]], [18], tokens=[[1]]))
    expect("EINVAL", lambda: h.catchup_batch([s1], [rows[:2]], [18], tokens=[[1, 256]]))
    # the pool holds 6 pages of 8: s1 has 3, s2's window of 24 rows needs 4
    expect("ENOMEM", lambda: h.catchup_batch([s1, s2], [rows[:1], torch.cat([rows, rows])[:33]],
                                             [18, 0]))
    assert (h.block_table(s1), h.block_table(s2), h.pool.n_free()) == before
    h.propose(s1, 4, 18, None, G - 1)
    expect("ESTATE", lambda: h.catchup_batch([s1], [rows[:1]], [18]))
    h.after_verify(s1, 1)
    # after accepting 1 draft, at most 2 rows fit before the expected position 20
    expect("EPOSITION", lambda: h.catchup_batch([s1], [rows[:3]], [18]))
    assert h.catchup_batch([s1], [rows[:2]], [18]) == 2
    assert h.block_table(s1)[0] == 20
