"""Host-side split of a call's attention into work items, checked without a
GPU through dflash_debug_attn_work. [P1] "Struct BlockDiffusionDraftHead"
fields kv_cache and ctx_window fix what the attention covers: for every
sequence and kv head, the ctx keys of the window (positions ws..pos-1)
followed by the gamma block keys. The split must cover each of those keys
exactly once, start every ctx chunk after the window's first on a 64-key
tile boundary, stay within the partial-slot capacity, and spread the items
over the persistent CTAs so that no CTA carries more than the mean load plus
one item (the bound of any least-loaded-first list schedule)."""
import ctypes as C
import random

import pytest

from block_diffusion_speculative_forward_gb300 import binding as B

I32 = C.c_int32
P32 = C.POINTER(C.c_int32)
EINVAL = -1


@pytest.fixture(scope="module")
def fn():
    from block_diffusion_speculative_forward_gb300 import build
    build.build()
    f = C.CDLL(B._LIB_PATH).dflash_debug_attn_work
    f.restype = I32
    f.argtypes = [I32, P32, P32, I32, I32, I32, I32, I32, P32, I32, P32, P32]
    return f


def attn_work(fn, pos, ws, nkv, gamma, slot_cap, grid, sms=152, cap=1 << 15):
    n = len(pos)
    items = (I32 * (5 * cap))()
    off = (I32 * (grid + 1))()
    n_pairs = I32(-7)
    k = fn(n, (I32 * max(n, 1))(*pos), (I32 * max(n, 1))(*ws), nkv, gamma, slot_cap, grid, sms,
           items, cap, off if grid else None, C.byref(n_pairs))
    if k < 0:
        return k, None, None
    return [tuple(items[5 * i:5 * i + 5]) for i in range(k)], list(off), n_pairs.value


def tiles(item, pos, ws, gamma):
    """64-key tiles the tensor-core kernel runs for an item: ctx items start
    at the page (16 keys) holding their first key."""
    s, _, k0, k1, _ = item
    n_ctx = pos[s] - ws[s]
    if k0 >= n_ctx:
        return -(-gamma // 64)
    lo, hi = ws[s] + k0, ws[s] + k1
    return -(-(hi - (lo & ~15)) // 64)


def check_split(items, off, n_pairs, pos, ws, nkv, gamma, slot_cap, grid):
    n = len(pos)
    by_pair = {}
    for it in items:
        by_pair.setdefault((it[0], it[1]), []).append(it)
    assert set(by_pair) == {(s, g) for s in range(n) for g in range(nkv)}
    slots, split_pairs, lengths = [], 0, []
    for (s, g), its in by_pair.items():
        n_ctx = pos[s] - ws[s]
        if n_ctx == 0:
            assert its == [(s, g, 0, gamma, -1)]
            continue
        split_pairs += 1
        ctx = sorted((it for it in its if it[2] < n_ctx), key=lambda it: it[2])
        blk = [it for it in its if it[2] >= n_ctx]
        assert [(it[2], it[3]) for it in blk] == [(n_ctx, n_ctx + gamma)]
        # the ctx chunks tile [0, n_ctx) without gap or overlap
        assert ctx[0][2] == 0 and ctx[-1][3] == n_ctx
        for a, b in zip(ctx, ctx[1:]):
            assert a[3] == b[2]
        for it in ctx:
            assert it[2] < it[3]
            if it[2] > 0:
                assert (ws[s] + it[2]) % 64 == 0, it
        lengths += [it[3] - it[2] for it in ctx[1:-1]]
        # the pair's partials sit in consecutive slots
        ps = sorted(it[4] for it in its)
        assert ps == list(range(ps[0], ps[0] + len(ps)))
        slots += ps
    assert n_pairs == split_pairs
    assert len(slots) == len(set(slots)) and all(0 <= x for x in slots)
    assert len(slots) <= slot_cap
    # interior chunks share one length, a multiple of the 64-key tile
    assert len(set(lengths)) <= 1
    if lengths:
        assert lengths[0] % 64 == 0
    if not grid:
        return
    assert off[0] == 0 and off[-1] == len(items)
    assert all(a <= b for a, b in zip(off, off[1:]))
    cost = [tiles(it, pos, ws, gamma) + 1 for it in items]
    loads = [sum(cost[off[b]:off[b + 1]]) for b in range(grid)]
    assert max(loads) <= sum(cost) / grid + max(cost)
    # longest first within each CTA
    for b in range(grid):
        c = cost[off[b]:off[b + 1]]
        assert c == sorted(c, reverse=True)


def test_single_sequence_short_ctx(fn):
    """One sequence with 1024 ctx keys (four kv heads): 64-key chunks."""
    pos, ws = [1024], [0]
    items, off, npairs = attn_work(fn, pos, ws, 4, 16, 3 * 152 + 3 * 4 + 64, 152)
    check_split(items, off, npairs, pos, ws, 4, 16, 3 * 152 + 3 * 4 + 64, 152)
    assert sum(1 for it in items if it[2] < 1024) == 4 * 16


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_ragged_batch(fn, seed):
    """32 sequences with ctx U[256, 4096] and no window cap."""
    rng = random.Random(seed)
    pos = [rng.randint(256, 4096) + rng.randint(1, 16) for _ in range(32)]
    ws = [0] * 32
    cap = 3 * 152 + 3 * 32 * 4 + 64
    items, off, npairs = attn_work(fn, pos, ws, 4, 16, cap, 152)
    check_split(items, off, npairs, pos, ws, 4, 16, cap, 152)


def test_windows_and_empty_ctx(fn):
    """Window starts that are not multiples of 16 or 64, a sequence at
    position 0 and one whose window is empty (ws == pos)."""
    rng = random.Random(9)
    pos, ws = [], []
    for i in range(12):
        p = rng.randint(4200, 9000)
        pos.append(p)
        ws.append(p - 4096)
    pos += [0, 37, 5000]
    ws += [0, 37, 4999]
    cap = 3 * 152 + 3 * 16 * 2 + 64
    items, off, npairs = attn_work(fn, pos, ws, 2, 8, cap, 152)
    check_split(items, off, npairs, pos, ws, 2, 8, cap, 152)


def test_slot_cap_forces_longer_chunks(fn):
    """With few slots the chunks grow until every partial fits."""
    rng = random.Random(4)
    pos = [rng.randint(2000, 4000) for _ in range(8)]
    ws = [0] * 8
    wide, _, _ = attn_work(fn, pos, ws, 4, 16, 10000, 0)
    items, off, npairs = attn_work(fn, pos, ws, 4, 16, 80, 0)
    check_split(items, off, npairs, pos, ws, 4, 16, 80, 0)
    assert len(items) < len(wide)


def test_mma_sync_path_has_no_schedule(fn):
    """grid 0 (the mma.sync kernel): items only, no CTA offsets written."""
    pos, ws = [300, 40], [0, 0]
    items, off, npairs = attn_work(fn, pos, ws, 2, 4, 100, 0)
    check_split(items, off, npairs, pos, ws, 2, 4, 100, 0)
    assert off == [0]


def test_bad_arguments(fn):
    assert attn_work(fn, [10], [11], 2, 4, 100, 8)[0] == EINVAL      # ws > pos
    assert attn_work(fn, [10], [0], 0, 4, 100, 8)[0] == EINVAL       # no kv heads
    assert attn_work(fn, [10], [0], 2, 4, 100, 8, sms=0)[0] == EINVAL
    assert attn_work(fn, [5000] * 4, [0] * 4, 4, 16, 1000, 8, cap=3)[0] == EINVAL
    # 16 split pairs need at least 32 slots: refused, not silently truncated
    assert attn_work(fn, [5000] * 4, [0] * 4, 4, 16, 31, 8)[0] == EINVAL
    items, _, _ = attn_work(fn, [5000] * 4, [0] * 4, 4, 16, 32, 8)
    assert len(items) == 32
