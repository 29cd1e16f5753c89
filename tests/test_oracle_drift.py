"""The end-to-end envelope of the GPU parity tests, measured on the oracle.

The GPU computes in fp32 (residual, accumulations, norms, softmax) with bf16
GEMM operands; the oracle computes the same steps in float64. Over a deep
stack the two drift apart without any error on either side: summation-order
differences of ~1e-7 move a value across a bf16 rounding point now and then,
and the next layer amplifies it. This test measures that drift with no GPU at
all, by running the oracle itself a second time in float32 (every step the
same, only the arithmetic narrower) on an 8-layer head, and asserts that it
stays inside the envelope the end-to-end GPU checks use (logits within
E2E_LOGIT_TOL of the row's largest logit; drafts equal where the top-1/top-2
gap exceeds E2E_GAP), and that the drift is real (far above float64
rounding), which is why deep stacks are compared layer by layer
(teacher-forced) against the tighter bars."""
import pytest
import torch

import oracle
import oracle.draft_head as dh
from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.parity import E2E_GAP, E2E_LOGIT_TOL, HIDDEN_TOL, cfg_for, gaps

# 8 layers like the shipped drafter, narrower so that the CPU suite stays fast
DEEP = syn.Geometry(num_layers=8, hidden=1024, intermediate=2048, num_q_heads=8,
                    num_kv_heads=2, head_dim=128, vocab=16384, gamma=16, mask_token_id=16383,
                    n_target_layers=2, target_hidden=512, rope_theta=1e7)


def _run(precision, monkeypatch, w, cfg, stack):
    with monkeypatch.context() as m:
        m.setattr(dh, "F64", precision)
        ora = oracle.DraftHeadOracle(cfg, w)
        st = ora.alloc_state()
        ora.prefill(st, stack[:96])
        taps = {}
        out = ora.propose(st, 321, 97, stack[96:97], 15, taps=taps)
    t = taps["seq"][0]
    return out, [x.to(torch.float64) for x in t["x"]], t["logits"].to(torch.float64)


def test_fp32_evaluation_stays_inside_the_end_to_end_envelope(monkeypatch):
    seed = 1301
    w = syn.make_weights(DEEP, seed)
    cfg = cfg_for(DEEP, max_batch=1, max_seq_len=256)
    stack = syn.make_stack(DEEP, 97, seed)
    (d64, n64, c64), x64, l64 = _run(torch.float64, monkeypatch, w, cfg, stack)
    (d32, n32, c32), x32, l32 = _run(torch.float32, monkeypatch, w, cfg, stack)
    assert x32[0].dtype == torch.float64 and n64 == n32 == 15
    drift = [float((a - b).abs().max()) for a, b in zip(x64, x32)]
    # the drift is real: far above float64 rounding after the first layers
    assert drift[-1] > 1e-4, drift
    # ... and grows with depth rather than staying at one layer's rounding
    assert drift[-1] > drift[1], drift
    # inside the envelope of the end-to-end checks
    rel = float(((l64 - l32).abs().amax(1) / l64.abs().amax(1)).max())
    assert rel <= E2E_LOGIT_TOL, (rel, drift)
    g = gaps(l64, None)
    for i in range(15):
        if g[i] > E2E_GAP:
            assert d64[i] == d32[i], (i, float(g[i]))
    assert abs(c64 - c32) <= 1e-2
    # per layer (teacher-forced) the fp32 evaluation is far inside the hidden bar
    assert max(drift[l + 1] - drift[l] for l in range(len(drift) - 1)) < HIDDEN_TOL, drift
