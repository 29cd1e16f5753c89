"""Pins of the CPU oracle against facts that do not come from the oracle:
closed forms, published format definitions, brute force on tiny inputs and
invariants the method must satisfy. A plausible slip anywhere in the oracle
(a dropped term, a wrong sign or index, a transposed operand, a wrong GQA map,
a wrong fused-K/V row order) fails at least one of these."""
import math
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests import brute_force as bf

GOLDEN = __import__("os").path.join(__import__("os").path.dirname(__file__), "golden")

# A micro drafter: 2 layers so that the layer loop and the fused K/V row order
# are exercised, GQA groups of 2, a window smaller than the context.
MICRO = syn.Geometry(num_layers=2, hidden=128, intermediate=128, num_q_heads=4,
                     num_kv_heads=2, head_dim=64, vocab=256, gamma=4, mask_token_id=255,
                     n_target_layers=2, target_hidden=64, rope_theta=1e4,
                     ctx_window=24, kv_block=8, prefill_chunk=10)


def cfg_of(geom, **kw):
    c = dict(num_layers=geom.num_layers, hidden=geom.hidden, intermediate=geom.intermediate,
             num_q_heads=geom.num_q_heads, num_kv_heads=geom.num_kv_heads,
             head_dim=geom.head_dim, vocab=geom.vocab, gamma=geom.gamma,
             mask_token_id=geom.mask_token_id, n_target_layers=geom.n_target_layers,
             target_hidden=geom.target_hidden, rms_eps=geom.rms_eps,
             ctx_window=geom.ctx_window, kv_block=geom.kv_block,
             prefill_chunk=geom.prefill_chunk, max_batch=4, max_seq_len=512,
             kv_pool_blocks=0, kv_dtype=0, lm_head_dtype=0)
    c.update(kw)
    return c


def make_micro(seed=7, **kw):
    w = syn.make_weights(MICRO, seed)
    return oracle.DraftHeadOracle(cfg_of(MICRO, **kw), w), w


# ------------------------------------------------------------- number formats
def test_bf16_rounding_midpoints():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1).
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: ties go to 1 + 2^-6.
    vals = torch.tensor([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -(1 + 2 ** -8)],
                        dtype=torch.float64)
    want = [1.0, 1 + 2 ** -6, 1 + 2 ** -7, -1.0]
    assert oracle.round_bf16(vals).tolist() == want
    # agrees with an independent bit-level RNE on random fp32 values
    x = torch.randn(20000, generator=torch.Generator().manual_seed(3), dtype=torch.float64) * 37
    assert np.array_equal(oracle.round_bf16(x).numpy(), bf.bf16_rne(x.numpy()))


def _e4m3_decode(code: int) -> float:
    """OCP 8-bit FP spec, E4M3: bias 7, 3 mantissa bits, subnormals at e=0,
    S.1111.111 is NaN, no infinities."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1 + m / 8.0) * 2.0 ** (e - 7)


def test_e4m3_exhaustive():
    finite = [c for c in range(256) if (c & 0x7F) != 0x7F]
    vals = sorted({_e4m3_decode(c) for c in finite})
    t = torch.tensor(vals, dtype=torch.float32)
    assert oracle.e4m3_codes(t).tolist() == vals                      # exact round trip
    assert max(vals) == 448.0 and min(v for v in vals if v > 0) == 2.0 ** -9
    pos = [v for v in vals if v >= 0]
    for a, b in zip(pos, pos[1:]):
        mid = (a + b) / 2
        got = oracle.e4m3_codes(torch.tensor([mid])).item()
        # ties go to the code whose mantissa is even
        code_a = [c for c in finite if _e4m3_decode(c) == a and not c & 0x80][0]
        assert got == (a if code_a % 2 == 0 else b), (a, b, got)
        assert oracle.e4m3_codes(torch.tensor([mid * (1 - 1e-6)])).item() == a
        assert oracle.e4m3_codes(torch.tensor([mid * (1 + 1e-6)])).item() == b
    sat = oracle.e4m3_codes(torch.tensor([449.0, 1e9, -1e9, 470.0]))
    assert sat.tolist() == [448.0, 448.0, -448.0, 448.0]


def test_golden_e4m3_anchors():
    # tests/golden/e4m3_anchors.txt: code -> value rows from the OCP FP8 spec tables.
    rows = [l.split() for l in open(f"{GOLDEN}/e4m3_anchors.txt") if l.strip() and l[0] != "#"]
    for code, val in rows:
        assert _e4m3_decode(int(code, 16)) == float(val)
        assert oracle.e4m3_codes(torch.tensor([float(val)])).item() == float(val)


# ------------------------------------------------------------------- RMSNorm
def test_rmsnorm_closed_form_and_scale_invariance():
    n, c, eps = 48, 0.37, 1e-6
    g = torch.linspace(0.5, 1.5, n, dtype=torch.float64)
    out = oracle.rms_norm(torch.full((n,), c, dtype=torch.float64), g, eps)
    assert torch.allclose(out, g * c / math.sqrt(c * c + eps), rtol=0, atol=1e-15)
    x = torch.randn(3, n, dtype=torch.float64, generator=torch.Generator().manual_seed(1))
    a = oracle.rms_norm(x, g, 0.0)
    b = oracle.rms_norm(x * 123.0, g, 0.0)
    assert torch.allclose(a, b, atol=1e-12)
    # mean of squares of the unit-gain output is one (eps = 0)
    u = oracle.rms_norm(x, torch.ones(n, dtype=torch.float64), 0.0)
    assert torch.allclose((u * u).mean(-1), torch.ones(3, dtype=torch.float64), atol=1e-12)


# ---------------------------------------------------------------------- RoPE
def test_rope_closed_form_pairs():
    d = 8
    inv = torch.tensor([1.0, 0.5, 0.25, 0.125], dtype=torch.float32)
    pos = torch.tensor([3])
    for i in range(d // 2):
        e = torch.zeros(1, d, dtype=torch.float64)
        e[0, i] = 1.0
        out = oracle.rope(e, pos, inv)[0]
        th = 3 * float(inv[i])
        want = torch.zeros(d, dtype=torch.float64)
        want[i], want[i + d // 2] = math.cos(th), math.sin(th)    # (1,0) -> (cos, sin)
        assert torch.allclose(out, want, atol=1e-15)
        e2 = torch.zeros(1, d, dtype=torch.float64)
        e2[0, i + d // 2] = 1.0
        out2 = oracle.rope(e2, pos, inv)[0]
        want2 = torch.zeros(d, dtype=torch.float64)
        want2[i], want2[i + d // 2] = -math.sin(th), math.cos(th)  # (0,1) -> (-sin, cos)
        assert torch.allclose(out2, want2, atol=1e-15)


def test_rope_invariants():
    d = 64
    inv = syn.make_inv_freq(d, 1e6)
    gen = torch.Generator().manual_seed(5)
    q = torch.randn(1, d, dtype=torch.float64, generator=gen)
    k = torch.randn(1, d, dtype=torch.float64, generator=gen)
    assert torch.allclose(oracle.rope(q, torch.tensor([0]), inv), q, atol=0)
    for a, b in [(5, 2), (16384, 16381), (9000, 8997), (40, 37)]:
        qa = oracle.rope(q, torch.tensor([a]), inv)
        kb = oracle.rope(k, torch.tensor([b]), inv)
        assert abs(qa.norm() - q.norm()) < 1e-12
        ref = (oracle.rope(q, torch.tensor([3]), inv) * oracle.rope(k, torch.tensor([0]), inv)).sum()
        assert abs(float((qa * kb).sum() - ref)) < 1e-9


# ----------------------------------------------------------------- attention
def test_attention_brute_force_and_special_cases():
    gen = torch.Generator().manual_seed(11)
    rows, nq, nkv, d, keys = 3, 4, 2, 8, 5
    q = torch.randn(rows, nq, d, dtype=torch.float64, generator=gen)
    k = torch.randn(keys, nkv, d, dtype=torch.float64, generator=gen)
    v = torch.randn(keys, nkv, d, dtype=torch.float64, generator=gen)
    out = oracle.attention(q, k, v)
    for r in range(rows):
        for j in range(nq):
            g = j // (nq // nkv)
            s = [sum(q[r, j, t].item() * k[u, g, t].item() for t in range(d)) / math.sqrt(d)
                 for u in range(keys)]
            e = [math.exp(x) for x in s]
            ref = [sum(e[u] * v[u, g, t].item() for u in range(keys)) / sum(e) for t in range(d)]
            assert np.allclose(out[r, j].numpy(), ref, atol=1e-12)
    zero = oracle.attention(torch.zeros_like(q), k, v)
    assert torch.allclose(zero[0, 0], v[:, 0].mean(0), atol=1e-14)
    assert torch.allclose(zero[0, 3], v[:, 1].mean(0), atol=1e-14)
    one = oracle.attention(q, k[:1], v[:1])
    assert torch.allclose(one[2, 1], v[0, 0], atol=1e-14)
    # nkv == nq is plain multi-head attention: head j reads kv head j
    kk = torch.randn(keys, nq, d, dtype=torch.float64, generator=gen)
    vv = torch.randn(keys, nq, d, dtype=torch.float64, generator=gen)
    mha = oracle.attention(q, kk, vv)
    for j in range(nq):
        assert torch.allclose(mha[:, j:j + 1], oracle.attention(q[:, j:j + 1], kk[:, j:j + 1], vv[:, j:j + 1]))


# ------------------------------------------------------- MLP / activation
def test_silu_values():
    x = torch.tensor([0.0, 1.0, -2.0, 30.0], dtype=torch.float64)
    want = [0.0, 1 / (1 + math.exp(-1)), -2 / (1 + math.exp(2)), 30 / (1 + math.exp(-30))]
    assert np.allclose(oracle.silu(x).numpy(), want, atol=1e-15)


def test_zero_gate_gives_zero_mlp():
    # silu(0) = 0, so zero gate weights remove the MLP: the residual after the
    # layer then equals x + attention only; compare against o_proj alone.
    head, w = make_micro()
    for lay in head.layers:
        lay["gate"].zero_()
    st = head.alloc_state()
    head.prefill(st, syn.make_stack(MICRO, 30, 7))
    taps = {"seq": []}
    head.propose_batch([st], [5], [30], [None], 3, taps=taps, _single=True)
    head2, _ = make_micro()
    for lay in head2.layers:
        lay["gate"].zero_()
        lay["down"].normal_(generator=torch.Generator().manual_seed(9))
    st2 = head2.alloc_state()
    head2.prefill(st2, syn.make_stack(MICRO, 30, 7))
    taps2 = {"seq": []}
    head2.propose_batch([st2], [5], [30], [None], 3, taps=taps2, _single=True)
    for a, b in zip(taps["seq"][0]["x"], taps2["seq"][0]["x"]):
        assert torch.equal(a, b)


# ------------------------------------------------- lm_head argmax / confidence
def test_select_drafts_cases():
    V = 40
    uni = torch.zeros(2, V, dtype=torch.float64)
    d, n, conf, _ = oracle.select_drafts(uni, None)
    assert d == [0, 0] and n == 2 and abs(conf - 1 / V) < 1e-15
    lg = torch.randn(3, V, dtype=torch.float64, generator=torch.Generator().manual_seed(2))
    one = torch.zeros(V, dtype=torch.bool)
    one[17] = True
    d, n, conf, _ = oracle.select_drafts(lg, one)
    assert d == [17, 17, 17] and conf == 1.0
    allm = torch.ones(V, dtype=torch.bool)
    assert oracle.select_drafts(lg, allm)[:3] == oracle.select_drafts(lg, None)[:3]
    assert oracle.select_drafts(lg, torch.zeros(V, dtype=torch.bool))[1:3] == (0, 0.0)
    tie = torch.zeros(1, V, dtype=torch.float64)
    tie[0, 9] = tie[0, 4] = 2.0
    d, _, conf, _ = oracle.select_drafts(tie, None)
    assert d == [4] and abs(conf - 1 / (2 + (V - 2) * math.exp(-2))) < 1e-15
    # conf is the minimum of the rows' top-1 probabilities
    _, _, conf, p1 = oracle.select_drafts(lg, None)
    ref = [1 / float(torch.exp(r - r.max()).sum()) for r in lg]
    assert np.allclose(p1, ref) and conf == min(p1)


def test_bitmask_bit_layout():
    words = torch.tensor([1, 0, -2 ** 31, 0], dtype=torch.int32)     # bits 0 and 95
    allowed = oracle.bitmask_allowed(words, 100)
    assert allowed.nonzero().flatten().tolist() == [0, 95]


# ----------------------------------------------------------- whole model
@pytest.mark.parametrize("window", [24, 0, 4096])
def test_whole_model_vs_brute_force(window):
    geom = replace(MICRO, ctx_window=window)
    w = syn.make_weights(geom, 21)
    head = oracle.DraftHeadOracle(cfg_of(geom), w)
    st = head.alloc_state()
    P = 37
    stack = syn.make_stack(geom, P, 21)
    head.prefill(st, stack)
    taps = {}
    mask = syn.make_bitmask(geom.vocab, 1, 21)[0]
    drafts, n_out, conf = head.propose(st, 17, P, None, 3, bitmask=mask, taps=taps)
    bd, bn, bconf, blog, btaps = bf.draft(geom, w, stack, 17, P, 3, bitmask_row=mask)
    for a, b in zip(taps["seq"][0]["x"], btaps):
        assert np.allclose(a.numpy(), b, atol=1e-9)
    assert np.allclose(taps["seq"][0]["logits"].numpy(), blog, atol=1e-9)
    assert drafts == bd and n_out == bn and abs(conf - bconf) < 1e-12


def test_whole_model_fp8_kv_and_lm_head_vs_dequantised_bf16_path():
    # FP8 lm_head (weight-only): logits = s_v * <z, codes_v>, the same as a bf16
    # head whose rows are the dequantised codes.
    geom = MICRO
    w = syn.make_weights(geom, 5, lm_head_fp8=True)
    h8 = oracle.DraftHeadOracle(cfg_of(geom, lm_head_dtype=1), w)
    w2 = dict(w)
    w2["lm_head"] = (w["lm_head_fp8"].to(torch.float64) * w["lm_head_scale"].to(torch.float64)[:, None])
    h16 = oracle.DraftHeadOracle(cfg_of(geom), w2)
    res = []
    for h in (h8, h16):
        st = h.alloc_state()
        h.prefill(st, syn.make_stack(geom, 20, 5))
        t = {}
        h.propose(st, 3, 20, None, 3, taps=t)
        res.append(t["seq"][0]["logits"])
    assert torch.allclose(res[0], res[1], rtol=1e-12, atol=1e-12)


def test_fp8_kv_cache_codes():
    w = syn.make_weights(MICRO, 6, kv_fp8=True)
    head = oracle.DraftHeadOracle(cfg_of(MICRO, kv_dtype=1), w)
    st = head.alloc_state()
    head.prefill(st, syn.make_stack(MICRO, 20, 6))
    for l in range(MICRO.num_layers):
        k, v = head.gather_kv(st, l, range(0, 20))
        for t, kind in ((k, 0), (v, 1)):
            s = w["kv_scale"][l, :, kind].to(torch.float64)
            codes = t / s[None, :, None]
            assert torch.equal(oracle.e4m3_codes(codes.to(torch.float32)), codes)
            assert codes.abs().max() <= 448


# -------------------------------------------------------------- invariants
def test_drafts_invariant_to_rows_before_window():
    geom = MICRO            # window 24, propose at 40: rows 0..15 are outside
    w = syn.make_weights(geom, 8)
    stack = syn.make_stack(geom, 40, 8)
    pert = stack.clone()
    pert[:16] = syn.make_stack(geom, 16, 99)
    outs = []
    for s in (stack, pert):
        h = oracle.DraftHeadOracle(cfg_of(geom), w)
        st = h.alloc_state()
        h.prefill(st, s)
        t = {}
        outs.append((h.propose(st, 9, 40, None, 3, taps=t), t["seq"][0]["logits"]))
    assert outs[0][0] == outs[1][0] and torch.equal(outs[0][1], outs[1][1])
    # and rows inside the window do matter
    pert[30] = syn.make_stack(geom, 1, 98)[0]
    h = oracle.DraftHeadOracle(cfg_of(geom), w)
    st = h.alloc_state()
    h.prefill(st, pert)
    t = {}
    h.propose(st, 9, 40, None, 3, taps=t)
    assert not torch.equal(t["seq"][0]["logits"], outs[0][1])


def test_chunking_does_not_change_values():
    w = syn.make_weights(MICRO, 4)
    stack = syn.make_stack(MICRO, 33, 4)
    res = []
    for chunk in (10, 512):
        g = replace(MICRO, prefill_chunk=chunk)
        h = oracle.DraftHeadOracle(cfg_of(g), w)
        st = h.alloc_state()
        h.prefill(st, stack)
        res.append(h.gather_kv(st, 1, range(9, 33)))
    assert torch.allclose(res[0][0], res[1][0], atol=0) and torch.allclose(res[0][1], res[1][1], atol=0)


@pytest.mark.parametrize("k", [0, 1, 2, 3])
def test_after_verify_then_propose_equals_fresh_prefill(k):
    geom = MICRO
    w = syn.make_weights(geom, 12)
    P = 29
    stack = syn.make_stack(geom, P + k + 1, 12)
    h1 = oracle.DraftHeadOracle(cfg_of(geom), w)
    s1 = h1.alloc_state()
    h1.prefill(s1, stack[:P])
    h1.propose(s1, 4, P, None, 3)
    h1.after_verify(s1, k)
    t1 = {}
    r1 = h1.propose(s1, 77, P + k + 1, stack[P:P + k + 1], 3, taps=t1)
    h2 = oracle.DraftHeadOracle(cfg_of(geom), w)
    s2 = h2.alloc_state()
    h2.prefill(s2, stack)
    t2 = {}
    r2 = h2.propose(s2, 77, P + k + 1, None, 3, taps=t2)
    assert r1 == r2
    assert torch.equal(t1["seq"][0]["logits"], t2["seq"][0]["logits"])
    ws = max(0, P + k + 1 - geom.ctx_window)
    for l in range(geom.num_layers):
        a, b = h1.gather_kv(s1, l, range(ws, P + k + 1)), h2.gather_kv(s2, l, range(ws, P + k + 1))
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_batch_equals_independent_proposes():
    geom = MICRO
    w = syn.make_weights(geom, 13)
    hb = oracle.DraftHeadOracle(cfg_of(geom), w)
    ctx = [5, 30, 17]
    sts = [hb.alloc_state() for _ in ctx]
    for i, (st, c) in enumerate(zip(sts, ctx)):
        hb.prefill(st, syn.make_stack(geom, c, 13, idx=i))
    masks = syn.make_bitmask(geom.vocab, 3, 13)
    rb = hb.propose_batch(sts, [1, 2, 3], ctx, [None] * 3, 3, bitmask=masks)
    for i, c in enumerate(ctx):
        h = oracle.DraftHeadOracle(cfg_of(geom), w)
        st = h.alloc_state()
        h.prefill(st, syn.make_stack(geom, c, 13, idx=i))
        assert h.propose(st, i + 1, c, None, 3, bitmask=masks[i]) == rb[i]
    assert hb.propose_batch(sts[:1], [1], [5], [None], 3) is None        # n < 2 declines


def test_errors_leave_state_unchanged():
    head, w = make_micro(kv_pool_blocks=3)
    st = head.alloc_state()
    head.prefill(st, syn.make_stack(MICRO, 10, 1))             # pages 0, 1
    before = head.block_table(st)
    with pytest.raises(oracle.OracleError) as e:                # needs 2 more pages, 1 free
        head.prefill(st, syn.make_stack(MICRO, 20, 2))
    assert e.value.code == "ENOMEM" and head.block_table(st) == before
    for bad, code in [(dict(position=11), "EPOSITION"), (dict(num_drafts=4), "EINVAL"),
                      (dict(last_token=256), "EINVAL"), (dict(num_drafts=0), "EINVAL")]:
        args = dict(last_token=1, position=10, new_rows=None, num_drafts=3)
        args.update(bad)
        with pytest.raises(oracle.OracleError) as e:
            head.propose(st, **args)
        assert e.value.code == code and head.block_table(st) == before
    head.propose(st, 1, 10, None, 3)
    with pytest.raises(oracle.OracleError) as e:
        head.propose(st, 1, 10, None, 3)
    assert e.value.code == "ESTATE"
    with pytest.raises(oracle.OracleError):
        head.after_verify(st, 4)
    head.after_verify(st, 2)
    with pytest.raises(oracle.OracleError) as e:
        head.propose(st, 1, 12, syn.make_stack(MICRO, 2, 3), 3)       # needs k+1 = 3 rows
    assert e.value.code == "EPOSITION"
    head.free_state(st)
    assert head.pool.n_free() == 3


def test_fc_width_mismatch_is_hard_error():
    w = syn.make_weights(MICRO, 1)
    with pytest.raises(oracle.OracleError):
        oracle.DraftHeadOracle(cfg_of(MICRO, fc_in_features=65), w)
