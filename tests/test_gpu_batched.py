"""GPU parity of the batched propose at the shipped geometry.

32 sequences (gamma 16, ragged ctx 256..4096, 1..16 new rows each, a 50%
grammar bitmask per sequence) and 128 sequences (gamma 8, FP8 E4M3 KV cache
with per-head scales, FP8 lm_head with per-row scales, two propose/verify
rounds). Sequences are independent, so the oracle replays a sample of them
(the shortest, the longest and the first): layer by layer (each oracle layer
fed the GPU's residual), logits from the GPU's final norm, drafts and
confidence, end to end within the fp32 envelope. Every sequence's page table
is checked against the position-level page simulator."""
import pytest
import torch

import oracle
from block_diffusion_speculative_forward_gb300 import binding as B
from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.parity import (CONF_TOL, E2E_GAP, E2E_LOGIT_TOL, HIDDEN_TOL, LOGIT_TOL, LOGIT_TOL_FP8,
                          cfg_for, check_abs, check_drafts, check_fp8_kv, check_logits,
                          check_rows, gaps)
from tests.test_oracle_state import PositionSim

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_diffusion_speculative_forward_gb300 import build
    build.build()


def _gpu_stack(geom, rows, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn((rows, geom.stack_width), device="cuda", generator=g).to(torch.bfloat16)


class Batch:
    def __init__(self, geom, seed, n, ctx, fp8):
        self.geom, self.seed, self.n, self.ctx = geom, seed, n, ctx
        self.cfg = cfg_for(geom, max_batch=n, max_seq_len=4096 + 64, kv_dtype=int(fp8),
                           lm_head_dtype=int(fp8))
        self.w = syn.make_weights(geom, seed, lm_head_fp8=fp8, kv_fp8=fp8)
        self.lib = B.DraftHead(self.cfg, B.weights_to_device(self.w))
        self.ora = oracle.DraftHeadOracle(self.cfg, self.w)
        self.fp8 = fp8
        self.sampled = sorted({0, min(range(n), key=lambda i: ctx[i]),
                               max(range(n), key=lambda i: ctx[i])})
        R, H, L = n * geom.gamma, geom.hidden, geom.num_layers
        self.tx = torch.zeros((L + 1) * R * H, device="cuda")
        self.tz = torch.zeros((R, H), dtype=torch.bfloat16, device="cuda")
        self.tl = torch.zeros((n * (geom.gamma - 1), geom.vocab), device="cuda")
        self.lib.set_taps(self.tx, self.tz, self.tl)
        self.sim = PositionSim(self.lib.debug_pool()[1], geom.kv_block, geom.ctx_window)
        self.sl, self.so, self.stacks = [], {}, {}
        for i in range(n):
            st = self.lib.alloc_state()
            self.sl.append(st)
            self.sim.new(i)
            if i in self.sampled:
                stack = syn.make_stack(geom, ctx[i] + 64, seed, idx=i)
                self.so[i] = self.ora.alloc_state()
                self.ora.prefill(self.so[i], stack[:ctx[i]])
                self.lib.prefill(st, stack[:ctx[i]].cuda())
            else:
                stack = _gpu_stack(geom, ctx[i] + 64, seed * 1000 + i)
                self.lib.prefill(st, stack[:ctx[i]])
            torch.cuda.synchronize()
            self.stacks[i] = stack[ctx[i]:].clone()   # rows of the later rounds
            self.sim.step([i], [ctx[i]])
        self.pos = list(ctx)
        self.used = [0] * n

    def rows(self, i, m):
        if m == 0:
            return None, None
        r = self.stacks[i][self.used[i]:self.used[i] + m]
        self.used[i] += m
        return (r.cuda() if not r.is_cuda else r), (r if not r.is_cuda else None)

    def round(self, n_new, nd, bitmask):
        geom = self.geom
        dev_rows, cpu_rows = zip(*[self.rows(i, m) for i, m in enumerate(n_new)])
        pos = [p + m for p, m in zip(self.pos, n_new)]
        toks = syn.uniform_ints(0, geom.vocab - 1, self.n, self.seed, 500 + pos[0])
        got = self.lib.propose_batch(self.sl, toks, pos, list(dev_rows), nd,
                                     bitmask=None if bitmask is None else bitmask.cuda())
        torch.cuda.synchronize()
        self.sim.step(list(range(self.n)), list(n_new))
        for i in range(self.n):
            assert self.lib.debug_state(self.sl[i]) == self.sim.table(i), i
        g, H, L = geom.gamma, geom.hidden, geom.num_layers
        R = self.n * g
        tx = self.tx[:(L + 1) * R * H].reshape(L + 1, R, H)
        ids, p1 = self.lib.debug_rows(self.n * nd)
        for i in self.sampled:
            allowed = None if bitmask is None else oracle.bitmask_allowed(bitmask[i], geom.vocab)
            taps = {}
            ref = self.ora.propose(self.so[i], toks[i], pos[i], cpu_rows[i], nd,
                                   bitmask=None if bitmask is None else bitmask[i], taps=taps)
            xs = tx[:, i * g:(i + 1) * g].double().cpu()
            check_abs(taps["seq"][0]["x"][0], xs[0], 0.0, "embed")
            for l in range(L):
                ref_l = self.ora.layer_forward(self.so[i], l, xs[l], pos[i])
                check_abs(ref_l, xs[l + 1], HIDDEN_TOL, f"seq {i} layer {l}")
            z_got = self.tz[i * g:(i + 1) * g].double().cpu()
            z_ref = oracle.round_bf16(oracle.rms_norm(xs[L], self.ora.norm, geom.rms_eps))
            check_abs(z_ref, z_got, HIDDEN_TOL, f"seq {i} final norm")
            lg_ref = self.ora.draft_logits(z_got, nd)
            lg_got = self.tl[i * nd:(i + 1) * nd]
            check_logits(lg_ref, lg_got, LOGIT_TOL_FP8 if self.fp8 else LOGIT_TOL)
            check_rows(lg_ref, allowed, ids[i * nd:(i + 1) * nd], p1[i * nd:(i + 1) * nd], got[i])
            d_ref, n_ref, c_ref, _ = oracle.select_drafts(lg_ref, allowed)
            assert got[i][1] == n_ref == ref[1]
            check_drafts(d_ref, got[i][0], lg_ref, allowed)
            assert abs(got[i][2] - c_ref) <= CONF_TOL
            check_logits(taps["seq"][0]["logits"], lg_got, E2E_LOGIT_TOL)
            ge = gaps(taps["seq"][0]["logits"], allowed)
            for j in range(n_ref):
                if ge[j] > E2E_GAP:
                    assert ref[0][j] == got[i][0][j]
            if allowed is not None:
                for d in got[i][0][:got[i][1]]:
                    assert allowed[d]
        self.pos = pos
        return got


def test_full_geometry_batch32_ragged_with_bitmask():
    geom, seed, n = syn.FULL, 1004, 32
    ctx = syn.uniform_ints(256, 4096, n, seed, 1)
    b = Batch(geom, seed, n, ctx, fp8=False)
    n_new = syn.uniform_ints(1, 16, n, seed, 2)
    mask = syn.make_bitmask(geom.vocab, n, seed)
    got = b.round(n_new, geom.gamma - 1, mask)
    assert all(r[1] == geom.gamma - 1 for r in got)


def test_full_geometry_fp8_batch128_two_rounds():
    geom, seed, n = syn.FULL_G8, 1005, 128
    ctx = syn.uniform_ints(512, 4096, n, seed, 1)
    b = Batch(geom, seed, n, ctx, fp8=True)
    for i in b.sampled:
        s = b.so[i]
        pos = list(range(ctx[i] - 24, ctx[i]))
        for l in (0, geom.num_layers - 1):
            k, v = b.lib.gather_kv(b.sl[i], l, pos[0], len(pos))
            kr, vr = b.ora.gather_kv(s, l, pos)
            check_fp8_kv(b, l, kr, k, 0)
            check_fp8_kv(b, l, vr, v, 1)
    n_new = [0] * n
    for rnd in range(2):
        got = b.round(n_new, geom.gamma - 1, None)
        ks = syn.uniform_ints(0, geom.gamma - 1, n, seed, 700 + rnd)
        for i in range(n):
            b.lib.after_verify(b.sl[i], ks[i])
            b.sim.verify(i, b.pos[i], ks[i])
            if i in b.sampled:
                b.ora.after_verify(b.so[i], ks[i])
            assert b.lib.debug_state(b.sl[i]) == b.sim.table(i)
        n_new = [k + 1 for k in ks]
