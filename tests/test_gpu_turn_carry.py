"""GPU parity of the drafter-KV carry across turns ([P3] "Trait
DraftProposer": take_drafter_kv, install_drafter_kv): a sequence carried
through take + install into another state proposes in its next turn what the
oracle, carrying the same way, proposes; the state it was taken from, reused
as a fresh one, matches too. Three geometries: the tiny drafter (mma.sync
attention, head dim 64), a window smaller than the context (the installed
pages start above logical page 0, pages of 8 rows) and head dim 128 (the
tensor-core attention)."""
import pytest

from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.parity import Pair, assert_tables, check_kv, check_seq
from tests.test_gpu_attention_tc import HD128_G8
from tests.test_oracle_pins import MICRO

pytestmark = pytest.mark.gpu

# geometry, ctx rows before the carry
GEOMS = {"tiny": (syn.TINY, 150), "window24": (MICRO, 45), "hd128": (HD128_G8, 150)}


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_diffusion_speculative_forward_gb300 import build
    build.build()


def carry_script(pair, geom, P, check):
    """The call sequence of the test; check(kind, so, sl, taps, ref, got) runs
    the comparisons after each propose."""
    nd, k = geom.gamma - 1, 2
    stack = syn.make_stack(geom, P + 8, 61)
    dev = pair.lib.bookkeeping_only is False
    so, sl = pair.ora.alloc_state(), pair.lib.alloc_state()
    pair.ora.prefill(so, stack[:P])
    pair.lib.prefill(sl, stack[:P].cuda() if dev else stack[:P])
    pair.ora.propose(so, 11, P, None, nd)
    got = pair.lib.propose(sl, 11, P, None, nd)
    assert got[1] == nd
    pair.ora.after_verify(so, k)
    pair.lib.after_verify(sl, k)
    bundle = pair.ora.take_drafter_kv(so)
    assert bundle is not None and pair.lib.take_drafter_kv(sl) == bundle
    assert_tables(pair, so, sl)                      # both fresh now
    so2, sl2 = pair.ora.alloc_state(), pair.lib.alloc_state()
    assert pair.ora.install_drafter_kv(so2, *bundle)
    assert pair.lib.install_drafter_kv(sl2, *bundle)
    assert_tables(pair, so2, sl2)
    p = P + k + 1
    taps = {}
    rows = stack[P:p]
    ref = pair.ora.propose(so2, 22, p, rows, nd, taps=taps)
    got = pair.lib.propose(sl2, 22, p, rows.cuda() if dev else rows, nd)
    assert_tables(pair, so2, sl2)
    check("carried", so2, sl2, taps, ref, got, p)
    # the state the pages were taken from, reused as a fresh one
    fresh = syn.make_stack(geom, 30, 61, idx=1)
    pair.ora.prefill(so, fresh[:29])
    pair.lib.prefill(sl, fresh[:29].cuda() if dev else fresh[:29])
    taps = {}
    ref = pair.ora.propose(so, 5, 30, fresh[29:30], nd, taps=taps)
    got = pair.lib.propose(sl, 5, 30, fresh[29:30].cuda() if dev else fresh[29:30], nd)
    assert_tables(pair, so, sl)
    check("reused", so, sl, taps, ref, got, 30)


@pytest.mark.parametrize("name", list(GEOMS))
def test_carry_to_next_turn(name):
    geom, P = GEOMS[name]
    pair = Pair(geom, 61, cfg_kw=dict(max_batch=2))
    W = pair.cfg["ctx_window"]
    nd = geom.gamma - 1

    def check(kind, so, sl, taps, ref, got, p):
        check_seq(pair, taps["seq"][0], ref, got, 0, 1, nd)
        check_kv(pair, so, sl, range(max(0, p - W), p))

    carry_script(pair, geom, P, check)
