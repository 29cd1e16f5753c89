"""GPU parity of the tensor-core block attention (bf16 cache, head dim 128,
pages of 16 rows) on small drafters, element by element against the oracle:
ragged window starts, items cut into several split-KV chunks and merged,
sequences with no ctx at all (block keys only), a full 128-vector query tile
(gamma 16 x 8 heads per kv head) and a mostly padded one (gamma 8 x 2)."""
from dataclasses import replace

import pytest
import torch

from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.parity import Pair, assert_tables, check_kv, check_seq

pytestmark = pytest.mark.gpu

# 8 q heads on one kv head, gamma 16: 128 query vectors per (sequence, kv head)
HD128_G16 = syn.Geometry(num_layers=2, hidden=256, intermediate=256, num_q_heads=8,
                         num_kv_heads=1, head_dim=128, vocab=1024, gamma=16,
                         mask_token_id=1023, n_target_layers=2, target_hidden=128,
                         rope_theta=1e4, ctx_window=200, kv_block=16, prefill_chunk=64)
# 4 q heads on 2 kv heads, gamma 8: 16 query vectors per (sequence, kv head)
HD128_G8 = replace(HD128_G16, num_q_heads=4, num_kv_heads=2, gamma=8)


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_diffusion_speculative_forward_gb300 import build
    build.build()


def _prefill(pair, n_rows, seed, idx=0):
    so, sl = pair.ora.alloc_state(), pair.lib.alloc_state()
    if n_rows:
        stack = syn.make_stack(pair.geom, n_rows, seed, idx)
        pair.ora.prefill(so, stack)
        pair.lib.prefill(sl, stack.cuda())
    return so, sl


@pytest.mark.parametrize("geom", [HD128_G16, HD128_G8], ids=["g16", "g8"])
@pytest.mark.parametrize("window", [200, 4096], ids=["window200", "window4096"])
def test_rounds(geom, window):
    """Prefill 301 rows, then propose/after_verify rounds: the window start
    moves through positions that are not multiples of 16."""
    geom = replace(geom, ctx_window=window)
    pair = Pair(geom, 41, cfg_kw=dict(max_batch=2))
    so, sl = _prefill(pair, 301, 41)
    p, n_new, used = 301, 0, 0
    rows = syn.make_stack(geom, 120, 41, idx=1)
    nd = geom.gamma - 1
    for k in [0, 5, 2, nd, 1]:
        r = rows[used:used + n_new] if n_new else None
        used += n_new
        taps = {}
        ref = pair.ora.propose(so, (13 * p) % geom.vocab, p, r, nd, taps=taps)
        got = pair.lib.propose(sl, (13 * p) % geom.vocab, p, None if r is None else r.cuda(), nd)
        check_seq(pair, taps["seq"][0], ref, got, 0, 1, nd)
        k = min(k, got[1])
        pair.ora.after_verify(so, k)
        pair.lib.after_verify(sl, k)
        assert_tables(pair, so, sl)
        p, n_new = p + k + 1, k + 1
    check_kv(pair, so, sl, range(max(0, p - window), p - n_new))


@pytest.mark.parametrize("geom", [HD128_G16, HD128_G8], ids=["g16", "g8"])
def test_batch_ragged_with_empty_ctx(geom):
    """propose_batch over four sequences: no ctx at all (position 0), a
    single page, a ragged 150-row ctx and 333 rows (several chunks)."""
    pair = Pair(geom, 43, cfg_kw=dict(max_batch=4))
    ctx = [0, 16, 150, 333]
    so, sl = zip(*[_prefill(pair, c, 43, idx=i) for i, c in enumerate(ctx)])
    n_new = [0, 1, 7, 0]
    rows = [syn.make_stack(geom, m, 43, idx=10 + i) if m else None for i, m in enumerate(n_new)]
    pos = [c + m for c, m in zip(ctx, n_new)]
    toks = [3, 500, 1000, 77]
    nd = geom.gamma - 1
    taps = {}
    ref = pair.ora.propose_batch(list(so), toks, pos, rows, nd, taps=taps)
    got = pair.lib.propose_batch(list(sl), toks, pos,
                                 [None if r is None else r.cuda() for r in rows], nd)
    for i in range(4):
        check_seq(pair, taps["seq"][i], ref[i], got[i], i, 4, nd)
        assert_tables(pair, so[i], sl[i])
    torch.cuda.synchronize()
