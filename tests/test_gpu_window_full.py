"""GPU parity at the ctx_window cap with the shipped geometry ([P1]/[P2] field
ctx_window; the 8192-row prompt, 4096-row window configuration).

One sequence: an 8191-row prompt prefilled through the library's 512-row
chunks (rows below the window are neither computed nor stored), then
propose / after_verify rounds with accept counts drawn uniform in [0, 15],
each round bringing the k + 1 target rows the previous verify accepted. Every
round compares the page table bit-exactly against the oracle; sampled rounds
compare every layer teacher-forced (each oracle layer fed the GPU's residual
entering it, attending over the oracle's own 4096-row window), the final norm,
the logits and the lm_head stage row by row, and the drafts and confidence
end to end within the fp32 envelope; the stored ctx K/V are gathered at the
window's edges."""
import pytest
import torch

import oracle
from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.parity import (CONF_TOL, E2E_GAP, E2E_LOGIT_TOL, HIDDEN_TOL, LOGIT_TOL, Pair,
                          assert_tables, check_abs, check_kv, check_logits, check_rows, gaps)

pytestmark = pytest.mark.gpu

PROMPT, WINDOW, ROUNDS = 8192, 4096, 10
TEACHER_ROUNDS = (0, 4, 9)


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_diffusion_speculative_forward_gb300 import build
    build.build()


def test_full_geometry_window_cap_rounds():
    geom, seed = syn.FULL, 1003
    nd = geom.gamma - 1
    pair = Pair(geom, seed, cfg_kw=dict(max_batch=1, ctx_window=WINDOW,
                                        max_seq_len=PROMPT + geom.gamma * (ROUNDS + 2) + 64))
    stack = syn.make_stack(geom, PROMPT + geom.gamma * (ROUNDS + 1), seed)
    so, sl = pair.ora.alloc_state(), pair.lib.alloc_state()
    pair.ora.prefill(so, stack[:PROMPT - 1])
    pair.lib.prefill(sl, stack[:PROMPT - 1].cuda())
    torch.cuda.synchronize()
    assert_tables(pair, so, sl)
    lo = PROMPT - 1 - WINDOW
    check_kv(pair, so, sl, [lo, lo + 1, lo + 15, lo + 16] + list(range(PROMPT - 9, PROMPT - 1)))
    ks = syn.uniform_ints(0, nd, ROUNDS, seed, 7)
    toks = syn.uniform_ints(0, geom.vocab - 1, ROUNDS, seed, 8)
    g, H, L = geom.gamma, geom.hidden, geom.num_layers
    pos, used, n_new = PROMPT - 1, PROMPT - 1, 1
    for r in range(ROUNDS):
        pos += n_new
        rows = stack[used:used + n_new]
        used += n_new
        taps = {}
        ref = pair.ora.propose(so, toks[r], pos, rows, nd, taps=taps)
        got = pair.lib.propose(sl, toks[r], pos, rows.cuda(), nd)
        torch.cuda.synchronize()
        assert_tables(pair, so, sl)
        assert got[1] == ref[1] == nd
        tap = taps["seq"][0]
        lg_got = pair.tl[:nd]
        # end to end against the fp64 oracle, within the fp32 envelope
        check_logits(tap["logits"], lg_got, E2E_LOGIT_TOL)
        ge = gaps(tap["logits"], None)
        for j in range(nd):
            if ge[j] > E2E_GAP:
                assert ref[0][j] == got[0][j], (r, j, ref[0][j], got[0][j])
        assert abs(ref[2] - got[2]) <= CONF_TOL
        if r in TEACHER_ROUNDS:
            tx = pair.tx.reshape(-1)[:(L + 1) * g * H].reshape(L + 1, g, H).double().cpu()
            check_abs(tap["x"][0], tx[0], 0.0, "embed")
            for l in range(L):
                ref_l = pair.ora.layer_forward(so, l, tx[l], pos)
                check_abs(ref_l, tx[l + 1], HIDDEN_TOL, f"round {r} layer {l} (teacher-forced)")
            z_got = pair.tz[:g].double().cpu()
            z_ref = oracle.round_bf16(oracle.rms_norm(tx[L], pair.ora.norm, geom.rms_eps))
            check_abs(z_ref, z_got, HIDDEN_TOL, f"round {r} final norm")
            lg_ref = pair.ora.draft_logits(z_got, nd)
            check_logits(lg_ref, lg_got, LOGIT_TOL)
            ids, p1 = pair.lib.debug_rows(nd)
            check_rows(lg_ref, None, ids, p1, got)
        k = min(ks[r], got[1])
        pair.ora.after_verify(so, k)
        pair.lib.after_verify(sl, k)
        assert_tables(pair, so, sl)
        n_new = k + 1
    # the first rows of the next propose's window and the newest stored rows
    ws = max(0, pos + n_new - WINDOW)
    check_kv(pair, so, sl, [ws, ws + 1] + list(range(pos - 4, pos)))
