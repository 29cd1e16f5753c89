"""Pins of the oracle's page bookkeeping (window retirement, trim, page ids)
against a second simulator written position by position, on scripted call
sequences shaped like the windowed single-sequence workload and the batched
FP8 workload (scaled down). Also checks the invariants: no page is shared,
pages in use equal the sum of live pages, every page is free after free."""
from dataclasses import replace

import pytest
import torch

import oracle
from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.test_oracle_pins import MICRO, cfg_of


class PositionSim:
    """Marks pages per stored position; retires a page once every one of its
    positions lies below the window start; new pages get min(free set)."""

    def __init__(self, n_pages, B, W):
        self.free, self.B, self.W = set(range(n_pages)), B, W
        self.tab, self.len = {}, {}

    def new(self, sid):
        self.tab[sid], self.len[sid] = {}, 0

    def _retire(self, sid, ws):
        for b in list(self.tab[sid]):
            if all(j < ws for j in range(b * self.B, (b + 1) * self.B)):
                self.free.add(self.tab[sid].pop(b))

    def step(self, sids, n_news):
        starts = {}
        for sid, n in zip(sids, n_news):
            end = self.len[sid] + n
            ws = max(0, end - self.W) if self.W else end
            starts[sid] = (max(self.len[sid], ws), end)
            self._retire(sid, ws)
        for sid in sids:
            lo, end = starts[sid]
            for j in range(lo, end):
                if j // self.B not in self.tab[sid]:
                    pid = min(self.free)
                    self.free.remove(pid)
                    self.tab[sid][j // self.B] = pid
            self.len[sid] = end

    def verify(self, sid, p, k):
        nxt = p + k + 1
        self._retire(sid, max(0, nxt - self.W) if self.W else nxt)

    def table(self, sid):
        t = self.tab[sid]
        if not t:
            return self.len[sid], -1, []
        lo, hi = min(t), max(t)
        return self.len[sid], lo, [t.get(b, -1) for b in range(lo, hi + 1)]


def _check_invariants(head, states):
    used = [pid for st in states for pid in st.pages.values()]
    assert len(used) == len(set(used))
    assert len(used) + head.pool.n_free() == head.pool.n_pages


def test_windowed_single_sequence_script():
    geom = replace(MICRO, gamma=16, ctx_window=100, kv_block=16, prefill_chunk=64)
    w = syn.make_weights(geom, 3)
    head = oracle.DraftHeadOracle(cfg_of(geom, max_seq_len=4096), w)
    sim = PositionSim(head.pool.n_pages, 16, 100)
    st = head.alloc_state()
    sim.new(0)
    prompt = 300
    head.prefill(st, syn.make_stack(geom, prompt, 3))
    sim.step([0], [prompt])
    assert head.block_table(st) == sim.table(0)
    p, n_new = prompt, 0
    ks = syn.uniform_ints(0, 15, 64, 3, 0)
    rows = syn.make_stack(geom, 64 * 16 + 1, 3, idx=1)
    used = 0
    for k in ks:
        nr = rows[used:used + n_new] if n_new else None
        used += n_new
        head.propose(st, 5, p, nr, 15)
        sim.step([0], [n_new])
        assert head.block_table(st) == sim.table(0)
        head.after_verify(st, k)
        sim.verify(0, p, k)
        assert head.block_table(st) == sim.table(0)
        _check_invariants(head, [st])
        p, n_new = p + k + 1, k + 1
    head.free_state(st)
    assert head.pool.n_free() == head.pool.n_pages


def test_batched_script_with_ragged_ctx():
    geom = replace(MICRO, gamma=8, ctx_window=64, kv_block=16, prefill_chunk=64)
    w = syn.make_weights(geom, 4)
    n = 5
    head = oracle.DraftHeadOracle(cfg_of(geom, max_batch=n, max_seq_len=2048), w)
    sim = PositionSim(head.pool.n_pages, 16, 64)
    ctx = syn.uniform_ints(20, 120, n, 4, 1)
    sts = []
    for i, c in enumerate(ctx):
        st = head.alloc_state()
        head.prefill(st, syn.make_stack(geom, c, 4, idx=i))
        sim.new(i)
        sim.step([i], [c])
        sts.append(st)
    pos, n_new = list(ctx), [0] * n
    for rnd in range(12):
        new_rows = [syn.make_stack(geom, m, 4, idx=1000 + rnd * n + i) if m else None
                    for i, m in enumerate(n_new)]
        res = head.propose_batch(sts, [1] * n, pos, new_rows, 7)
        sim.step(list(range(n)), n_new)
        for i in range(n):
            assert head.block_table(sts[i]) == sim.table(i)
        ks = syn.uniform_ints(0, 7, n, 4, 100 + rnd)
        for i in range(n):
            assert res[i][1] == 7
            head.after_verify(sts[i], ks[i])
            sim.verify(i, pos[i], ks[i])
            assert head.block_table(sts[i]) == sim.table(i)
        _check_invariants(head, sts)
        pos = [p + k + 1 for p, k in zip(pos, ks)]
        n_new = [k + 1 for k in ks]
    for st in list(sts):
        head.free_state(st)
    assert head.pool.n_free() == head.pool.n_pages


def test_zero_window_stores_nothing():
    geom = replace(MICRO, ctx_window=0)
    head = oracle.DraftHeadOracle(cfg_of(geom), syn.make_weights(geom, 2))
    st = head.alloc_state()
    head.prefill(st, syn.make_stack(geom, 40, 2))
    assert head.block_table(st) == (40, -1, []) and not st.rows
    drafts, n_out, conf = head.propose(st, 3, 40, None, 3)
    assert n_out == 3
