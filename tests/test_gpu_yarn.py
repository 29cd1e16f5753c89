"""GPU parity of YaRN RoPE ([P1] field yarn_inv_freq): a head built with the
library's own YaRN table (dflash_yarn_inv_freq) and attention temperature
against the oracle built with its own evaluation of the same method, on the
tiny drafter (mma.sync attention) and at head dim 128 (tensor-core
attention). A short original context puts pairs in every regime of the ramp
at the positions reached; the ctx keys carry the temperature too."""
import pytest
import torch

import oracle
from block_diffusion_speculative_forward_gb300 import binding as B
from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.parity import Pair, assert_tables, cfg_for, check_kv, check_seq
from tests.test_gpu_attention_tc import HD128_G8

pytestmark = pytest.mark.gpu

# factor, beta_fast, beta_slow, original context
SCALING = (16.0, 32.0, 1.0, 64)
GEOMS = {"tiny": syn.TINY, "hd128": HD128_G8}


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_diffusion_speculative_forward_gb300 import build
    build.build()


def yarn_pair(geom, seed, dev=True):
    """A Pair whose two sides each compute their own YaRN table and
    temperature from the same rope_scaling parameters."""
    yarn = (geom.rope_theta, geom.head_dim) + SCALING
    base_cfg = cfg_for(geom, max_batch=2)
    w = syn.make_weights(geom, seed)
    pair = Pair.__new__(Pair)
    pair.geom, pair.fp8 = geom, False
    pair.w = dict(w, inv_freq=oracle.yarn_inv_freq(*yarn))
    pair.cfg = dict(base_cfg, rope_attn_factor=oracle.yarn_attention_factor(SCALING[0]))
    pair.ora = oracle.DraftHeadOracle(pair.cfg, pair.w)
    lib_tab, lib_att = B.yarn_inv_freq(*yarn)
    lib_w = dict(w, inv_freq=lib_tab)
    pair.wd = B.weights_to_device(lib_w) if dev else None
    pair.lib = B.DraftHead(dict(base_cfg, rope_attn_factor=lib_att), pair.wd)
    if dev:
        rows = base_cfg["max_batch"] * geom.gamma
        pair.tx = torch.zeros((geom.num_layers + 1, rows, geom.hidden), device="cuda")
        pair.tz = torch.zeros((rows, geom.hidden), dtype=torch.bfloat16, device="cuda")
        pair.tl = torch.zeros((rows, geom.vocab), device="cuda")
        pair.lib.set_taps(pair.tx, pair.tz, pair.tl)
    return pair


def yarn_script(pair, check, dev=True):
    geom = pair.geom
    nd = geom.gamma - 1
    stack = syn.make_stack(geom, 160, 71)
    on = (lambda t: t.cuda()) if dev else (lambda t: t)
    so, sl = pair.ora.alloc_state(), pair.lib.alloc_state()
    pair.ora.prefill(so, stack[:150])
    pair.lib.prefill(sl, on(stack[:150]))
    taps = {}
    ref = pair.ora.propose(so, 17, 150, None, nd, taps=taps)
    got = pair.lib.propose(sl, 17, 150, None, nd)
    assert_tables(pair, so, sl)
    check(so, sl, taps, ref, got, 150)
    pair.ora.after_verify(so, 2)
    pair.lib.after_verify(sl, 2)
    taps = {}
    ref = pair.ora.propose(so, 3, 153, stack[150:153], nd, taps=taps)
    got = pair.lib.propose(sl, 3, 153, on(stack[150:153]), nd)
    assert_tables(pair, so, sl)
    check(so, sl, taps, ref, got, 153)


@pytest.mark.parametrize("name", list(GEOMS))
def test_yarn_rope(name):
    pair = yarn_pair(GEOMS[name], 71)
    nd = pair.geom.gamma - 1

    def check(so, sl, taps, ref, got, p):
        check_seq(pair, taps["seq"][0], ref, got, 0, 1, nd)
        check_kv(pair, so, sl, range(p))

    yarn_script(pair, check)
