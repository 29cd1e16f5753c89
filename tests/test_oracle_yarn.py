"""Pins of the oracle's YaRN RoPE ([P1] field yarn_inv_freq: rope_scaling
factor 64, beta_fast 32, beta_slow 1, original_max_position_embeddings 4096)
against facts outside its formula: with factor 1 it is the plain table;
every pair that turns more than beta_fast times over the original context
keeps its frequency and every pair that turns fewer than beta_slow times is
divided by the factor (turn counts evaluated directly, pair by pair); the
pairs between blend the two along a linear ramp; the attention temperature
is the published 0.1 ln(s) + 1; and a factor of 2 on the rotated q and k
equals doubling the q/k norm gains, bit for bit, through a whole propose."""
import math
from dataclasses import replace

import torch

import oracle
from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.test_oracle_pins import MICRO, cfg_of

THETA, D, S, FAST, SLOW, ORIG = 1e7, 128, 64.0, 32.0, 1.0, 4096


def base_table(theta, d):
    return [theta ** (-2.0 * i / d) for i in range(d // 2)]


def test_factor_one_is_the_plain_table():
    got = oracle.yarn_inv_freq(THETA, D, 1.0, FAST, SLOW, ORIG)
    want = torch.tensor(base_table(THETA, D), dtype=torch.float64).to(torch.float32)
    assert torch.equal(got, want)


def test_shipped_setting_keeps_fast_pairs_and_interpolates_slow_ones():
    got = oracle.yarn_inv_freq(THETA, D, S, FAST, SLOW, ORIG).to(torch.float64)
    base = base_table(THETA, D)
    turns = [ORIG * b / (2 * math.pi) for b in base]      # turns over the original context
    kept = [i for i, t in enumerate(turns) if t > FAST]
    interp = [i for i, t in enumerate(turns) if t < SLOW]
    ramp = [i for i in range(D // 2) if i not in kept and i not in interp]
    assert kept and interp and ramp                        # all three regimes occur
    f32 = lambda x: float(torch.tensor(x, dtype=torch.float64).to(torch.float32))
    for i in kept:
        assert float(got[i]) == f32(base[i])
    for i in interp:
        assert float(got[i]) == f32(base[i] / S)
    # between: strictly between the two, blend weight linear in the pair index
    w = [(base[i] - float(got[i])) / (base[i] - base[i] / S) for i in ramp]
    assert all(0.0 < x < 1.0 for x in w)
    steps = [b - a for a, b in zip(w, w[1:])]
    assert max(steps) - min(steps) < 1e-5
    # the ramp reaches 0 one pair before its first pair and 1 at the first
    # interpolated pair
    assert abs(w[0] - steps[0]) < 1e-5 and abs(w[-1] + steps[0] - 1.0) < 1e-5


def test_attention_temperature():
    assert oracle.yarn_attention_factor(1.0) == 1.0
    assert abs(oracle.yarn_attention_factor(64.0) - (1 + 0.1 * math.log(64.0))) < 1e-15
    assert abs(oracle.yarn_attention_factor(64.0) - 1.4158883083359671) < 1e-12


def test_attention_temperature_shape():
    """The published temperature is affine in ln(s) with slope 1/10 and value
    1 at s = 1: checked through properties that fix such a function (no
    scaling is the identity; the excess over one adds across a product of
    factors; a factor of e^10 doubles the scale; shrinking (s < 1) never
    applies, the factor only grows), not through the formula itself."""
    f = oracle.yarn_attention_factor
    for a, b in [(2.0, 32.0), (4.0, 16.0), (8.0, 8.0), (3.0, 21.0)]:
        assert abs((f(a * b) - 1) - ((f(a) - 1) + (f(b) - 1))) < 1e-12
    assert abs(f(math.exp(10.0)) - 2.0) < 1e-12
    xs = [1.0, 1.5, 2.0, 16.0, 64.0, 1e3]
    assert all(f(x) < f(y) for x, y in zip(xs, xs[1:]))
    assert f(0.5) == 1.0


def test_factor_two_equals_doubled_qk_norm_gains():
    """The factor scales the rotated q and k (ctx keys included): with 2 the
    whole propose equals a head whose q_norm / k_norm gains are doubled."""
    geom = replace(MICRO, ctx_window=24)
    w = syn.make_weights(geom, 31)
    w2 = dict(w)
    w2["layers"] = [dict(lay, q_norm=lay["q_norm"] * 2, k_norm=lay["k_norm"] * 2)
                    for lay in w["layers"]]
    ha = oracle.DraftHeadOracle(cfg_of(geom, rope_attn_factor=2.0), w)
    hb = oracle.DraftHeadOracle(cfg_of(geom), w2)
    stack = syn.make_stack(geom, 40, 31)
    out = []
    for h in (ha, hb):
        st = h.alloc_state()
        h.prefill(st, stack[:37])
        taps = {}
        r = h.propose(st, 9, 40, stack[37:40], 3, taps=taps)
        out.append((r, taps["seq"][0]["logits"], h.gather_kv(st, 1, range(16, 40))))
    assert out[0][0] == out[1][0]
    assert torch.equal(out[0][1], out[1][1])
    assert torch.equal(out[0][2][0], out[1][2][0]) and torch.equal(out[0][2][1], out[1][2][1])
