"""Pins of the oracle's drafter-KV carry across turns ([P3] "Trait
DraftProposer": take_drafter_kv, install_drafter_kv, free_drafter_kv)
against facts that do not come from the carry code: a take followed by an
install is the identity on every result a propose computes; a taken state
behaves exactly as a freshly allocated one (the trait's wording); freeing the
carried pages returns the pool to its starting count; page ids follow the
position-by-position simulator extended with the three calls."""
import pytest
import torch

import oracle
from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.test_oracle_pins import MICRO, cfg_of
from tests.test_oracle_state import PositionSim

NU = 3   # drafts per propose (gamma 4)


def pair_of_heads(seed):
    w = syn.make_weights(MICRO, seed)
    return oracle.DraftHeadOracle(cfg_of(MICRO), w), oracle.DraftHeadOracle(cfg_of(MICRO), w)


def same_result(a, b, ta, tb):
    assert a == b
    assert torch.equal(ta["seq"][0]["logits"], tb["seq"][0]["logits"])
    for xa, xb in zip(ta["seq"][0]["x"], tb["seq"][0]["x"]):
        assert torch.equal(xa, xb)


@pytest.mark.parametrize("P,k", [(29, 0), (29, 3), (44, 3), (7, 1)])
def test_take_then_install_is_identity(P, k):
    """One head carries the sequence through take + install into another
    state between two turns; the other never carries. Every later result,
    the block table and the stored K/V are identical."""
    h1, h2 = pair_of_heads(21)
    stack = syn.make_stack(MICRO, P + k + 1, 21)
    s1, s2 = h1.alloc_state(), h2.alloc_state()
    for h, s in ((h1, s1), (h2, s2)):
        h.prefill(s, stack[:P])
        h.propose(s, 4, P, None, NU)
        h.after_verify(s, k)
    blocks, rows, key = h1.take_drafter_kv(s1)
    assert rows == P and key is None and blocks == h2.block_table(s2)[2]
    s1b = h1.alloc_state()
    assert h1.install_drafter_kv(s1b, blocks, rows, key)
    assert h1.block_table(s1b) == h2.block_table(s2)
    t1, t2 = {}, {}
    r1 = h1.propose(s1b, 77, P + k + 1, stack[P:P + k + 1], NU, taps=t1)
    r2 = h2.propose(s2, 77, P + k + 1, stack[P:P + k + 1], NU, taps=t2)
    same_result(r1, r2, t1, t2)
    assert h1.block_table(s1b) == h2.block_table(s2)
    ws = max(0, P + k + 1 - MICRO.ctx_window)
    for l in range(MICRO.num_layers):
        a, b = h1.gather_kv(s1b, l, range(ws, P + k + 1)), h2.gather_kv(s2, l, range(ws, P + k + 1))
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_taken_state_behaves_fresh():
    """After a take the state equals a new one: same block table, and a new
    prefill + propose on it gives what a brand-new state gives while the
    carried pages stay out of the pool."""
    h1, h2 = pair_of_heads(22)
    first = syn.make_stack(MICRO, 40, 22)
    second = syn.make_stack(MICRO, 33, 22, idx=1)
    s1, s2 = h1.alloc_state(), h2.alloc_state()
    for h, s in ((h1, s1), (h2, s2)):
        h.prefill(s, first)
        h.propose(s, 9, 40, None, NU)
        h.after_verify(s, 2)
    blocks, rows, _ = h1.take_drafter_kv(s1)
    assert h1.block_table(s1) == (0, -1, [])
    s3 = h2.alloc_state()       # h2 keeps its pages in s2: same free set as h1
    t1, t2 = {}, {}
    for h, s, t in ((h1, s1, t1), (h2, s3, t2)):
        h.prefill(s, second[:30])
        t["r"] = h.propose(s, 5, 33, second[30:33], NU, taps=t)
    same_result(t1["r"], t2["r"], t1, t2)
    assert h1.block_table(s1) == h2.block_table(s3)
    assert h1.pool.n_free() == h2.pool.n_free()
    # free_state of the taken-then-reused state releases only its own pages
    h1.free_state(s1)
    h1.free_drafter_kv(blocks)
    assert h1.pool.n_free() == h1.pool.n_pages


def test_page_ids_follow_the_simulator():
    """A scripted mix of turns: pages of live states, carried bundles and the
    free set always partition the pool, and every table matches the
    position-by-position simulator extended with take / install / free."""
    h, _ = pair_of_heads(23)
    sim = PositionSim(h.pool.n_pages, MICRO.kv_block, MICRO.ctx_window)
    B = MICRO.kv_block
    states, pos = {}, {}
    script = [("new", 0, 30), ("new", 1, 12), ("turn", 0, 2), ("turn", 1, 0), ("take", 0, None),
              ("new", 2, 20), ("install", 3, 0), ("turn", 3, 1), ("take", 1, None),
              ("turn", 2, 3), ("free", 1, None), ("turn", 3, 3), ("take", 3, None),
              ("install", 4, 3), ("turn", 4, 0)]
    carried = {}
    stack = syn.make_stack(MICRO, 64, 23)
    for op, sid, arg in script:
        if op == "new":
            states[sid] = h.alloc_state()
            sim.new(sid)
            h.prefill(states[sid], stack[:arg])
            sim.step([sid], [arg])
            pos[sid] = arg
        elif op == "turn":
            st, p = states[sid], pos[sid]
            n_new = p - st.ctx_len
            h.propose(st, 3, p, stack[:n_new] if n_new else None, NU)
            sim.step([sid], [n_new])
            h.after_verify(st, arg)
            sim.verify(sid, p, arg)
            pos[sid] = p + arg + 1
        elif op == "take":
            blocks, rows, _ = h.take_drafter_kv(states[sid])
            t = sim.tab[sid]
            assert blocks == [t[b] for b in sorted(t)] and rows == sim.len[sid]
            carried[sid] = (blocks, rows, pos[sid])   # the turn's next position
            sim.new(sid)
        elif op == "install":
            blocks, rows, nxt = carried.pop(arg)
            states[sid] = h.alloc_state()
            sim.new(sid)
            assert h.install_drafter_kv(states[sid], blocks, rows)
            b0 = -(-rows // B) - len(blocks)
            sim.tab[sid] = {b0 + i: p for i, p in enumerate(blocks)}
            sim.len[sid] = rows
            pos[sid] = nxt
        elif op == "free":
            blocks, _, _ = carried.pop(sid)
            h.free_drafter_kv(blocks)
            sim.free.update(blocks)
        for s_id, st in states.items():
            assert h.block_table(st) == sim.table(s_id)
        in_states = [p for st in states.values() for p in st.pages.values()]
        in_carry = [p for bl, _, _ in carried.values() for p in bl]
        assert sorted(in_states + in_carry + sorted(h.pool.free)) == list(range(h.pool.n_pages))
        assert set(h.pool.free) == sim.free


def test_carry_errors_change_nothing():
    h, _ = pair_of_heads(24)
    stack = syn.make_stack(MICRO, 60, 24)
    s = h.alloc_state()
    h.prefill(s, stack[:44])
    assert h.take_drafter_kv(h.alloc_state()) is None          # nothing to carry
    h.propose(s, 1, 44, None, NU)
    with pytest.raises(oracle.OracleError, match="ESTATE"):    # a propose awaits verify
        h.take_drafter_kv(s)
    h.after_verify(s, 3)          # next propose at 48: pages below 24 retire
    blocks, rows, _ = h.take_drafter_kv(s)
    assert blocks and rows == 44
    busy = h.alloc_state()
    h.prefill(busy, stack[:5])
    with pytest.raises(oracle.OracleError, match="EINVAL"):    # not a fresh state
        h.install_drafter_kv(busy, blocks, rows)
    t = h.alloc_state()
    with pytest.raises(oracle.OracleError, match="EINVAL"):    # rows do not match
        h.install_drafter_kv(t, blocks, rows + 1)
    with pytest.raises(oracle.OracleError, match="EINVAL"):    # not carried
        h.free_drafter_kv([blocks[0]])
    assert h.block_table(t) == (0, -1, [])
    assert h.install_drafter_kv(t, blocks, rows)
    with pytest.raises(oracle.OracleError, match="EINVAL"):    # installed already
        h.free_drafter_kv(blocks)
    # the window of a propose at 44 would start at 20, below the first
    # carried page (positions 24..): rejected; at 48 it starts at 24
    with pytest.raises(oracle.OracleError, match="EPOSITION"):
        h.propose(t, 1, 44, None, NU)
    h.propose(t, 1, 48, stack[44:48], NU)
