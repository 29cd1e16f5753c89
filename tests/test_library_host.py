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
                dict(kv_dtype=2), dict(hidden=100), dict(lm_head_dtype=3),
                dict(lm_head_dtype=2)):   # MICRO's hidden 128: NVFP4 stages take 256
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


def test_catchup_script_matches_oracle_bookkeeping():
    """[P2] catchup_batch in rounds: propose_batch, after_verify(k_i), then
    the first j_i of each sequence's k_i + 1 rows through the catch-up feed
    and the rest as the next propose's new rows; block tables after every
    call equal the oracle's."""
    geom = replace(MICRO, gamma=8, ctx_window=40, kv_block=8, prefill_chunk=64)
    n = 4
    cfg = cfg_of(geom, max_batch=n, max_seq_len=2048)
    ora = oracle.DraftHeadOracle(cfg, syn.make_weights(geom, 6))
    lib = B.DraftHead(cfg, None)
    ctx = syn.uniform_ints(5, 60, n, 6, 1)
    so, sl = [], []
    for i, c in enumerate(ctx):
        a, b = ora.alloc_state(), lib.alloc_state()
        ora.prefill(a, syn.make_stack(geom, c, 6, idx=i))
        lib.prefill(b, _fake_rows(c))
        so.append(a)
        sl.append(b)
    pos, pend = list(ctx), [0] * n
    for rnd in range(10):
        ora.propose_batch(so, [1] * n, pos,
                          [syn.make_stack(geom, m, 6, idx=1000 + rnd * n + i) if m else None
                           for i, m in enumerate(pend)], 7)
        lib.propose_batch(sl, [1] * n, pos, [_fake_rows(m) for m in pend], 7)
        ks = syn.uniform_ints(0, 7, n, 6, 100 + rnd)
        lib.after_verify_batch(sl, ks)
        for i in range(n):
            ora.after_verify(so[i], ks[i])
        js = [min(j, k + 1) for j, k in zip(syn.uniform_ints(0, 8, n, 6, 200 + rnd), ks)]
        first = [st.ctx_len for st in so]
        assert ora.catchup_batch(so, [syn.make_stack(geom, j, 6, idx=5000 + rnd * n + i)
                                      if j else None for i, j in enumerate(js)], first) == sum(js)
        assert lib.catchup_batch(sl, [_fake_rows(j) for j in js], first,
                                 tokens=[[3] * j for j in js]) == sum(js)
        for i in range(n):
            assert lib.debug_state(sl[i]) == ora.block_table(so[i])
        assert lib.debug_pool() == (ora.pool.n_pages - ora.pool.n_free(), ora.pool.n_pages)
        pos = [p + k + 1 for p, k in zip(pos, ks)]
        pend = [k + 1 - j for k, j in zip(ks, js)]


def test_catchup_errors_match_oracle_and_change_nothing():
    cfg = cfg_of(MICRO, kv_pool_blocks=6)
    ora = oracle.DraftHeadOracle(cfg, syn.make_weights(MICRO, 7))
    lib = B.DraftHead(cfg, None)
    o1, o2 = ora.alloc_state(), ora.alloc_state()
    l1, l2 = lib.alloc_state(), lib.alloc_state()
    ora.prefill(o1, syn.make_stack(MICRO, 18, 7))
    lib.prefill(l1, _fake_rows(18))
    rows = syn.make_stack(MICRO, 33, 7)
    cases = [
        ("EPOSITION", ([0], [2], [19], None)),
        ("EPOSITION", ([0], [2], [17], None)),
        ("EINVAL", ([0, 0], [1, 1], [18, 18], None)),
        ("EINVAL", ([0], [2], [18], [[1]])),
        ("EINVAL", ([0], [2], [18], [[1, 256]])),
        ("ENOMEM", ([0, 1], [1, 33], [18, 0], None)),
    ]
    for code, (idx, counts, first, toks) in cases:
        before = (lib.debug_state(l1), lib.debug_state(l2), lib.debug_pool())
        with pytest.raises(oracle.OracleError) as eo:
            ora.catchup_batch([(o1, o2)[i] for i in idx], [rows[:m] for m in counts], first, toks)
        with pytest.raises(B.DFlashError) as el:
            lib.catchup_batch([(l1, l2)[i] for i in idx], [_fake_rows(m) for m in counts], first,
                              tokens=toks)
        assert eo.value.code == el.value.code == code
        assert (lib.debug_state(l1), lib.debug_state(l2), lib.debug_pool()) == before
    ora.propose(o1, 4, 18, None, 3)
    lib.propose(l1, 4, 18, None, 3)
    with pytest.raises(B.DFlashError) as el:
        lib.catchup_batch([l1], [_fake_rows(1)], [18])
    assert el.value.code == "ESTATE"
    ora.after_verify(o1, 1)
    lib.after_verify(l1, 1)
    with pytest.raises(B.DFlashError) as el:
        lib.catchup_batch([l1], [_fake_rows(3)], [18])
    assert el.value.code == "EPOSITION"
    assert ora.catchup_batch([o1], [rows[:2]], [18]) == lib.catchup_batch([l1], [_fake_rows(2)],
                                                                            [18]) == 2
    assert lib.debug_state(l1) == ora.block_table(o1)
    with pytest.raises(B.DFlashError):
        B.DraftHead(cfg_of(MICRO, shifted_rows=2), None)


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


def test_drafter_kv_carry_matches_oracle_bookkeeping():
    """[P3] take_drafter_kv / install_drafter_kv / free_drafter_kv on the
    library's native scheduler against the oracle: the same bundles, block
    tables and pool counts after every call, and the same errors."""
    geom = replace(MICRO, gamma=8, ctx_window=40, kv_block=8, prefill_chunk=64)
    cfg = cfg_of(geom, max_batch=3, max_seq_len=1024)
    w = syn.make_weights(geom, 8)
    ora = oracle.DraftHeadOracle(cfg, w)
    lib = B.DraftHead(cfg, None)
    so, sl, pos, carried = {}, {}, {}, {}
    stack = syn.make_stack(geom, 96, 8)

    def same(sid):
        assert lib.debug_state(sl[sid]) == ora.block_table(so[sid]), sid
        assert lib.debug_pool() == (ora.pool.n_pages - ora.pool.n_free(), ora.pool.n_pages)

    script = [("new", 0, 70), ("new", 1, 9), ("turn", 0, 5), ("turn", 1, 7), ("take", 0, None),
              ("turn", 0, None), ("new", 2, 30), ("install", 3, 0), ("turn", 3, 2),
              ("take", 1, None), ("take", 2, None), ("free", 1, None), ("turn", 3, 7),
              ("take", 3, None), ("install", 4, 3), ("install", 5, 2), ("turn", 4, 0),
              ("turn", 5, 1)]
    for op, sid, arg in script:
        if op == "new" or (op == "turn" and arg is None):
            if op == "new":
                so[sid], sl[sid] = ora.alloc_state(), lib.alloc_state()
            n = arg if op == "new" else 20
            ora.prefill(so[sid], stack[:n])
            lib.prefill(sl[sid], _fake_rows(n))
            pos[sid] = so[sid].ctx_len
        elif op == "turn":
            p = pos[sid]
            n_new = p - so[sid].ctx_len
            ora.propose(so[sid], 3, p, stack[:n_new] if n_new else None, 7)
            lib.propose(sl[sid], 3, p, _fake_rows(n_new), 7)
            same(sid)
            ora.after_verify(so[sid], arg)
            lib.after_verify(sl[sid], arg)
            pos[sid] = p + arg + 1
        elif op == "take":
            a, b = ora.take_drafter_kv(so[sid]), lib.take_drafter_kv(sl[sid])
            assert a == b and a is not None
            carried[sid] = (a[0], a[1], pos[sid])
        elif op == "install":
            blocks, rows, nxt = carried.pop(arg)
            so[sid], sl[sid] = ora.alloc_state(), lib.alloc_state()
            assert ora.install_drafter_kv(so[sid], blocks, rows)
            assert lib.install_drafter_kv(sl[sid], blocks, rows)
            pos[sid] = nxt
        elif op == "free":
            blocks = carried.pop(sid)[0]
            ora.free_drafter_kv(blocks)
            lib.free_drafter_kv(blocks)
        for s_id in so:
            same(s_id)
    # nothing to carry; misuse changes nothing on either side
    fresh_o, fresh_l = ora.alloc_state(), lib.alloc_state()
    assert ora.take_drafter_kv(fresh_o) is None and lib.take_drafter_kv(fresh_l) is None
    p = pos[4]
    n_new = p - so[4].ctx_len
    ora.propose(so[4], 3, p, stack[:n_new] if n_new else None, 7)
    lib.propose(sl[4], 3, p, _fake_rows(n_new), 7)
    with pytest.raises(B.DFlashError, match="ESTATE"):
        lib.take_drafter_kv(sl[4])
    ora.after_verify(so[4], 7)
    lib.after_verify(sl[4], 7)
    blocks, rows, _ = lib.take_drafter_kv(sl[4])
    assert (blocks, rows, None) == ora.take_drafter_kv(so[4])
    before = lib.debug_pool()
    for bad in ([blocks, rows + 1], [blocks[:-1], rows], [[blocks[0] + 1000], rows]):
        with pytest.raises(B.DFlashError, match="EINVAL"):
            lib.install_drafter_kv(fresh_l, *bad)
    with pytest.raises(B.DFlashError, match="EINVAL"):       # not a fresh state
        lib.install_drafter_kv(sl[5], blocks, rows)
    with pytest.raises(B.DFlashError, match="EINVAL"):       # part of a bundle
        lib.free_drafter_kv(blocks[1:])
    assert lib.debug_pool() == before and lib.debug_state(fresh_l) == (0, -1, [])
    assert lib.install_drafter_kv(fresh_l, blocks, rows)
    assert ora.install_drafter_kv(fresh_o, blocks, rows)
    assert lib.debug_state(fresh_l) == ora.block_table(fresh_o)
    with pytest.raises(B.DFlashError, match="EINVAL"):       # installed: no longer carried
        lib.free_drafter_kv(blocks)
    # a window reaching below the first installed page is refused like the oracle does
    low = ora.block_table(fresh_o)[1] * geom.kv_block + geom.ctx_window - 1
    assert low > rows     # reachable by a propose that brings low - rows rows
    with pytest.raises(oracle.OracleError, match="EPOSITION"):
        ora.propose(fresh_o, 3, low, stack[:low - rows], 7)
    with pytest.raises(B.DFlashError, match="EPOSITION"):
        lib.propose(fresh_l, 3, low, _fake_rows(low - rows), 7)
    assert lib.debug_state(fresh_l) == ora.block_table(fresh_o)
    for s_id in so:
        lib.free_state(sl[s_id])
    lib.free_state(fresh_l)
    lib.free_state(lib.alloc_state())
    assert lib.debug_pool()[0] == 0


@pytest.mark.parametrize("theta,d,factor,fast,slow,orig", [
    (1e7, 128, 64.0, 32.0, 1.0, 4096),     # the shipped drafter's rope_scaling
    (1e6, 64, 16.0, 32.0, 1.0, 2048),
    (1e4, 128, 4.0, 32.0, 1.0, 512),
    (1e7, 128, 1.0, 32.0, 1.0, 4096)])     # no scaling: the plain table
def test_yarn_table_matches_oracle(theta, d, factor, fast, slow, orig):
    """The library's host-side YaRN table and temperature against the
    oracle's own evaluation of the published method (both in double, f32
    out): equal up to one f32 rounding of the same double."""
    got, att = B.yarn_inv_freq(theta, d, factor, fast, slow, orig)
    ref = oracle.yarn_inv_freq(theta, d, factor, fast, slow, orig)
    assert torch.allclose(got, ref, rtol=2 ** -23, atol=0)
    assert abs(att - oracle.yarn_attention_factor(factor)) <= 1e-6


def test_yarn_arguments_and_factor_validation():
    for bad in [(1.0, 128, 64.0, 32.0, 1.0, 4096), (1e7, 127, 64.0, 32.0, 1.0, 4096),
                (1e7, 128, 0.5, 32.0, 1.0, 4096), (1e7, 128, 64.0, 1.0, 1.0, 4096),
                (1e7, 128, 64.0, 32.0, 1.0, 0)]:
        with pytest.raises(B.DFlashError, match="EINVAL"):
            B.yarn_inv_freq(*bad)
    for f in (-1.0, float("nan")):
        with pytest.raises(B.DFlashError, match="EINVAL"):
            B.DraftHead(cfg_of(MICRO, rope_attn_factor=f), None)
    B.DraftHead(cfg_of(MICRO, rope_attn_factor=1.4158883), None).close()


def test_noalloc_gemm_rejects_bad_arguments_without_touching_memory():
    """dflash_gemm_noalloc's argument checks run before any CUDA call, so they
    are checked here with pointers that are never dereferenced."""
    f = C.CDLL(B._LIB_PATH).dflash_gemm_noalloc
    f.restype = C.c_int
    f.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32,
                  C.c_void_p]
    w, x, y, odd = 0x10000, 0x20000, 0x30000, 0x20008
    EINVAL = -1
    for args in [(None, x, y, 16, 128, 64), (w, None, y, 16, 128, 64), (w, x, None, 16, 128, 64),
                 (w, x, y, 0, 128, 64), (w, x, y, 17, 128, 64), (w, x, y, 16, 0, 64),
                 (w, x, y, 16, 4096 * 128 + 1, 64), (w, x, y, 16, 128, 0), (w, x, y, 16, 128, 96),
                 (w, odd, y, 16, 128, 64), (odd, x, y, 16, 128, 64)]:
        assert f(*args, None) == EINVAL, args
