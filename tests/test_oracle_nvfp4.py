"""Pins of the oracle's NVFP4 lm_head ([P1] field lm_head_nvfp4: the
target's NVFP4 head, 'packed + scales') against definitions outside it: the
16 E2M1 values of the OCP MX FP4 table; every E4M3 byte against torch's own
float8_e4m3fn decoding; the nibble order and the 16-element scale blocks on a
hand-built row; and the whole propose equal, bit for bit, to the bf16 path
run on the dequantised table (a power-of-two global scale keeps every
dequantised value exact in bf16)."""
import math
from dataclasses import replace

import torch

import oracle
from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.test_oracle_pins import MICRO, cfg_of

# OCP MX FP4 (E2M1): codes 0..7 positive, 8..15 the same magnitudes negated
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_table():
    for c in range(16):
        v = oracle.e2m1_value(c)
        want = E2M1_TABLE[c & 7] * (-1.0 if c >= 8 else 1.0)
        assert v == want and math.copysign(1.0, v) == (-1.0 if c >= 8 else 1.0)


def test_e4m3_bytes_match_torch():
    ref = torch.arange(256, dtype=torch.int64).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = ref.to(torch.float64)
    for c in range(256):
        got = oracle.e4m3_value(c)
        r = float(ref[c])
        assert (math.isnan(got) and math.isnan(r)) or got == r, (c, got, r)


def test_nibble_order_and_scale_blocks():
    # one row of 32 elements: bytes 0x21 -> (+0.5, +1.0), 0xf9 -> (-0.5, -6.0),
    # the rest zero; block 0 scale 2.0 (0x40), block 1 scale 0.5 (0x30)
    packed = torch.zeros((1, 16), dtype=torch.uint8)
    packed[0, 0], packed[0, 1], packed[0, 8] = 0x21, 0xF9, 0x67
    scales = torch.tensor([[0x40, 0x30]], dtype=torch.uint8)
    got = oracle.nvfp4_dequant(packed, scales, 0.25)
    want = torch.zeros(1, 32, dtype=torch.float64)
    want[0, 0], want[0, 1] = 0.5 * 2.0 * 0.25, 1.0 * 2.0 * 0.25
    want[0, 2], want[0, 3] = -0.5 * 2.0 * 0.25, -6.0 * 2.0 * 0.25
    want[0, 16], want[0, 17] = 6.0 * 0.5 * 0.25, 4.0 * 0.5 * 0.25
    assert torch.equal(got, want)


def test_propose_equals_bf16_path_on_dequantised_table():
    geom = replace(MICRO, ctx_window=24)
    w = syn.make_weights(geom, 41, lm_head_nvfp4=True)
    g = float(w["lm_head_nvfp4_global"])
    assert g == 2.0 ** round(math.log2(g))
    dq = oracle.nvfp4_dequant(w["lm_head_nvfp4"], w["lm_head_nvfp4_scale"], g)
    as_bf16 = dq.to(torch.bfloat16)
    assert torch.equal(as_bf16.to(torch.float64), dq)             # exact in bf16
    # the encoding stays close to the table it encodes: within half an E2M1
    # step (at most 1 at magnitudes 4..6) of each block's scale, plus the
    # block scale's own E4M3 rounding
    err = (dq - w["lm_head"].to(torch.float64)).abs().reshape(geom.vocab, -1, 16)
    amax = w["lm_head"].to(torch.float64).abs().reshape(geom.vocab, -1, 16).amax(dim=2)
    assert bool((err.amax(dim=2) <= amax / 6.0 * 1.07 + 1e-12).all())
    ha = oracle.DraftHeadOracle(cfg_of(geom, lm_head_dtype=2), w)
    hb = oracle.DraftHeadOracle(cfg_of(geom), dict(w, lm_head=as_bf16))
    stack = syn.make_stack(geom, 40, 41)
    out = []
    for h in (ha, hb):
        st = h.alloc_state()
        h.prefill(st, stack[:38])
        taps = {}
        out.append((h.propose(st, 7, 40, stack[38:40], 3, taps=taps), taps["seq"][0]["logits"]))
    assert out[0][0] == out[1][0]
    assert torch.equal(out[0][1], out[1][1])
