"""Host-side checks of libdflash that need no GPU: every symbol the header
declares is exported, geometry validation, and the native page bookkeeping
(window retirement, trim, lowest-free-id allocation, all-or-nothing batches)
bit-exact against the oracle's on scripted call sequences."""
import ctypes as C
import os
import re
from dataclasses import replace

import pytest
import torch

import oracle
from block_diffusion_speculative_forward_gb300 import binding as B
from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.test_oracle_pins import MICRO, cfg_of

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_diffusion_speculative_forward_gb300 import build
    build.build()


def header_functions():
    src = open(os.path.join(ROOT, "include", "dflash.h")).read()
    return sorted(set(re.findall(r"DFLASH_API\s+[\w\s\*]*?\b(dflash_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = header_functions()
    assert len(names) >= 15
    lib = C.CDLL(B._LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_geometry_validation():
    cfg = cfg_of(MICRO)
    cfg["fc_in_features"] = 65
    with pytest.raises(B.DFlashError) as e:
        B.DraftHead(cfg, None)
    assert e.value.code == "EINVAL" and "validate_against_target" in str(e.value)
    for bad in (dict(head_dim=48), dict(num_q_heads=3), dict(gamma=1), dict(mask_token_id=256),
                dict(kv_dtype=2), dict(hidden=100)):
        c = cfg_of(MICRO)
        c.update(bad)
        with pytest.raises(B.DFlashError):
            B.DraftHead(c, None)
    h = B.DraftHead(cfg_of(MICRO), None)
    assert h.block_gamma() == MICRO.gamma and h.propose_batch_max() == 4


def _fake_rows(n):
    # bookkeeping-only heads never read rows; any non-NULL marker works
    return None if n == 0 else torch.empty((n, 8), dtype=torch.bfloat16)


def test_windowed_script_matches_oracle_bookkeeping():
    geom = replace(MICRO, gamma=16, ctx_window=100, kv_block=16, prefill_chunk=64)
    cfg = cfg_of(geom, max_seq_len=4096)
    w = syn.make_weights(geom, 3)
    ora = oracle.DraftHeadOracle(cfg, w)
    lib = B.DraftHead(cfg, None)
    so, sl = ora.alloc_state(), lib.alloc_state()
    prompt = 300
    ora.prefill(so, syn.make_stack(geom, prompt, 3))
    assert lib.prefill(sl, _fake_rows(prompt)) == B.BOOKKEEPING_ONLY
    assert lib.debug_state(sl) == ora.block_table(so)
    p, n_new = prompt, 0
    rows = syn.make_stack(geom, 64 * 16 + 1, 3, idx=1)
    used = 0
    for k in syn.uniform_ints(0, 15, 64, 3, 0):
        ora.propose(so, 5, p, rows[used:used + n_new] if n_new else None, 15)
        used += n_new
        lib.propose(sl, 5, p, _fake_rows(n_new), 15)
        assert lib.debug_state(sl) == ora.block_table(so)
        ora.after_verify(so, k)
        lib.after_verify(sl, k)
        assert lib.debug_state(sl) == ora.block_table(so)
        assert lib.debug_pool() == (ora.pool.n_pages - ora.pool.n_free(), ora.pool.n_pages)
        p, n_new = p + k + 1, k + 1
    lib.free_state(sl)
    assert lib.debug_pool()[0] == 0


def test_batched_script_matches_oracle_bookkeeping():
    geom = replace(MICRO, gamma=8, ctx_window=64, kv_block=16, prefill_chunk=64)
    n = 5
    cfg = cfg_of(geom, max_batch=n, max_seq_len=2048)
    w = syn.make_weights(geom, 4)
    ora = oracle.DraftHeadOracle(cfg, w)
    lib = B.DraftHead(cfg, None)
    ctx = syn.uniform_ints(20, 120, n, 4, 1)
    so, sl = [], []
    for i, c in enumerate(ctx):
        a, b = ora.alloc_state(), lib.alloc_state()
        ora.prefill(a, syn.make_stack(geom, c, 4, idx=i))
        lib.prefill(b, _fake_rows(c))
        so.append(a)
        sl.append(b)
    pos, n_new = list(ctx), [0] * n
    for rnd in range(12):
        ora.propose_batch(so, [1] * n, pos,
                          [syn.make_stack(geom, m, 4, idx=1000 + rnd * n + i) if m else None
                           for i, m in enumerate(n_new)], 7)
        res = lib.propose_batch(sl, [1] * n, pos, [_fake_rows(m) for m in n_new], 7)
        assert res is not None
        for i in range(n):
            assert lib.debug_state(sl[i]) == ora.block_table(so[i])
        ks = syn.uniform_ints(0, 7, n, 4, 100 + rnd)
        for i in range(n):
            ora.after_verify(so[i], ks[i])
            lib.after_verify(sl[i], ks[i])
            assert lib.debug_state(sl[i]) == ora.block_table(so[i])
        pos = [p + k + 1 for p, k in zip(pos, ks)]
        n_new = [k + 1 for k in ks]
    assert lib.propose_batch(sl[:1], [1], pos[:1], [None], 7) is None       # n < 2 declines
    assert lib.propose_batch(sl * 2, [1] * 10, pos * 2, [None] * 10, 7) is None  # n > max_batch


def test_errors_leave_state_unchanged():
    cfg = cfg_of(MICRO, kv_pool_blocks=3)
    lib = B.DraftHead(cfg, None)
    st = lib.alloc_state()
    lib.prefill(st, _fake_rows(10))
    before = lib.debug_state(st)
    with pytest.raises(B.DFlashError) as e:
        lib.prefill(st, _fake_rows(20))
    assert e.value.code == "ENOMEM" and lib.debug_state(st) == before
    for args, code in [((1, 11, None, 3), "EPOSITION"), ((1, 10, None, 4), "EINVAL"),
                       ((256, 10, None, 3), "EINVAL"), ((1, 10, None, 0), "EINVAL")]:
        with pytest.raises(B.DFlashError) as e:
            lib.propose(st, *args)
        assert e.value.code == code and lib.debug_state(st) == before
    lib.propose(st, 1, 10, None, 3)
    with pytest.raises(B.DFlashError) as e:
        lib.propose(st, 1, 10, None, 3)
    assert e.value.code == "ESTATE"
    with pytest.raises(B.DFlashError) as e:
        lib.prefill(st, _fake_rows(1))
    assert e.value.code == "ESTATE"
    with pytest.raises(B.DFlashError):
        lib.after_verify(st, 4)
    lib.after_verify(st, 2)
    with pytest.raises(B.DFlashError) as e:
        lib.propose(st, 1, 12, _fake_rows(2), 3)
    assert e.value.code == "EPOSITION"
    with pytest.raises(B.DFlashError):
        lib.after_verify(st, 0)
    other = B.DraftHead(cfg, None)
    with pytest.raises(B.DFlashError):
        other.free_state(st)
    lib.free_state(st)
    assert lib.debug_pool() == (0, 3)
    s2 = lib.alloc_state(budget_tokens=8)
    with pytest.raises(B.DFlashError) as e:
        lib.prefill(s2, _fake_rows(9))
    assert e.value.code == "EINVAL"


def test_repeated_state_in_batch_is_rejected():
    lib = B.DraftHead(cfg_of(MICRO), None)
    a = lib.alloc_state()
    with pytest.raises(B.DFlashError) as e:
        lib.propose_batch([a, a], [1, 1], [0, 0], [None, None], 3)
    assert e.value.code == "EINVAL"


def test_after_verify_batch_matches_per_sequence_calls():
    """[P3] after_verify applied to every state of a propose_batch in one call
    leaves the same block tables and pool as one call per state, and on any
    bad argument changes nothing."""
    geom = replace(MICRO, gamma=8, ctx_window=64, kv_block=16, prefill_chunk=64)
    n = 4
    cfg = cfg_of(geom, max_batch=n, max_seq_len=2048)
    one, many = B.DraftHead(cfg, None), B.DraftHead(cfg, None)
    ctx = syn.uniform_ints(20, 120, n, 6, 1)
    s1, s2 = [], []
    for c in ctx:
        a, b = one.alloc_state(), many.alloc_state()
        one.prefill(a, _fake_rows(c))
        many.prefill(b, _fake_rows(c))
        s1.append(a)
        s2.append(b)
    pos, n_new = list(ctx), [0] * n
    for rnd in range(10):
        one.propose_batch(s1, [1] * n, pos, [_fake_rows(m) for m in n_new], 7)
        many.propose_batch(s2, [1] * n, pos, [_fake_rows(m) for m in n_new], 7)
        ks = syn.uniform_ints(0, 7, n, 6, 200 + rnd)
        before = [many.debug_state(s) for s in s2]
        for bad in ([0, 0, 8, 0], [0, -1, 0, 0]):          # a count outside 0..n_out
            with pytest.raises(B.DFlashError, match="EINVAL"):
                many.after_verify_batch(s2, bad)
        with pytest.raises(B.DFlashError, match="EINVAL"):  # a state twice
            many.after_verify_batch([s2[0], s2[1], s2[0]], ks[:3])
        assert [many.debug_state(s) for s in s2] == before
        for i in range(n):
            one.after_verify(s1[i], ks[i])
        many.after_verify_batch(s2, ks)
        assert [one.debug_state(s) for s in s1] == [many.debug_state(s) for s in s2]
        assert one.debug_pool() == many.debug_pool()
        with pytest.raises(B.DFlashError, match="ESTATE"):  # no propose pending any more
            many.after_verify_batch(s2, ks)
        pos = [p + k + 1 for p, k in zip(pos, ks)]
        n_new = [k + 1 for k in ks]
