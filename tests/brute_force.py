"""A second, independent float64 evaluation of the draft head for tiny shapes.

Written apart from the oracle, in numpy with explicit loops, to pin the oracle:
its own bf16 rounding (bit-level round-to-nearest-even on fp32 words), RoPE as
an explicit 2x2 rotation per (i, i + d/2) pair, attention as per-query,
per-key loops, and each layer's ctx K/V from that layer's own k/v matrices
(not the fused weight). It keeps no pages: the ctx rows of the window are
recomputed from the target stack for every call.
"""
from __future__ import annotations

import math

import numpy as np


def bf16_rne(x) -> np.ndarray:
    """fp64 -> fp32 -> bf16 (round to nearest, ties to even) -> fp64."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def _np(t):
    return np.asarray(t.to(dtype=__import__("torch").float64).numpy(), dtype=np.float64)


def _rms(v, g, eps):
    ms = sum(float(a) * float(a) for a in v) / len(v)
    return np.array([g[i] * v[i] / math.sqrt(ms + eps) for i in range(len(v))])


def _rope(v, pos, inv_freq):
    d = len(v)
    out = np.array(v, dtype=np.float64)
    for i in range(d // 2):
        th = pos * float(inv_freq[i])
        c, s = math.cos(th), math.sin(th)
        a, b = v[i], v[i + d // 2]
        out[i] = c * a - s * b
        out[i + d // 2] = s * a + c * b
    return out


def _matvec(W, v):
    return np.array([float(np.dot(W[r], v)) for r in range(W.shape[0])])


def draft(geom, w, stack, last_token, p, num_drafts, bitmask_row=None):
    """Drafts, n_out, conf, logits [num_drafts, V] and the per-layer residuals.

    stack: [p, S] target stack rows for positions 0..p-1 (rows below the
    window are ignored)."""
    L, H = geom.num_layers, geom.hidden
    nq, nkv, d = geom.num_q_heads, geom.num_kv_heads, geom.head_dim
    eps, W, g = geom.rms_eps, geom.ctx_window, geom.gamma
    inv = w["inv_freq"].numpy().astype(np.float64)
    E = _np(w["embed"])
    LM = _np(w["lm_head"])
    FC = _np(w["fc"])
    layers = [{k: _np(v) for k, v in lay.items()} for lay in w["layers"]]
    X = _np(stack)
    ws = max(0, p - W) if W > 0 else p
    # ctx keys/values of the window, per layer: [n_ctx][nkv][d]
    ctxK = [[] for _ in range(L)]
    ctxV = [[] for _ in range(L)]
    for j in range(ws, p):
        c = bf16_rne(_rms(_matvec(FC, X[j]), _np(w["hidden_norm"]), eps))
        for l in range(L):
            k = _matvec(layers[l]["k"], c)
            v = _matvec(layers[l]["v"], c)
            ks, vs = [], []
            for h in range(nkv):
                kh = _rope(_rms(k[h * d:(h + 1) * d], layers[l]["k_norm"], eps), j, inv)
                ks.append(bf16_rne(kh))
                vs.append(bf16_rne(v[h * d:(h + 1) * d]))
            ctxK[l].append(ks)
            ctxV[l].append(vs)
    toks = [last_token] + [geom.mask_token_id] * (g - 1)
    x = [E[t].copy() for t in toks]
    taps = [np.array(x)]
    for l in range(L):
        lay = layers[l]
        qs, ks, vs = [], [], []
        for i in range(g):
            h = bf16_rne(_rms(x[i], lay["in_norm"], eps))
            q, k, v = _matvec(lay["q"], h), _matvec(lay["k"], h), _matvec(lay["v"], h)
            qs.append([bf16_rne(_rope(_rms(q[a * d:(a + 1) * d], lay["q_norm"], eps), p + i, inv))
                       for a in range(nq)])
            ks.append([bf16_rne(_rope(_rms(k[a * d:(a + 1) * d], lay["k_norm"], eps), p + i, inv))
                       for a in range(nkv)])
            vs.append([bf16_rne(v[a * d:(a + 1) * d]) for a in range(nkv)])
        grp = nq // nkv
        new_x = []
        for i in range(g):
            o = np.zeros(nq * d)
            for a in range(nq):
                kvh = a // grp
                keys = [ctxK[l][t][kvh] for t in range(len(ctxK[l]))] + [ks[t][kvh] for t in range(g)]
                vals = [ctxV[l][t][kvh] for t in range(len(ctxV[l]))] + [vs[t][kvh] for t in range(g)]
                sc = [float(np.dot(qs[i][a], kk)) / math.sqrt(d) for kk in keys]
                m = max(sc)
                e = [math.exp(s - m) for s in sc]
                z = sum(e)
                acc = np.zeros(d)
                for t in range(len(keys)):
                    acc += (e[t] / z) * vals[t]
                o[a * d:(a + 1) * d] = acc
            o = bf16_rne(o)
            xi = x[i] + _matvec(lay["o"], o)
            h2 = bf16_rne(_rms(xi, lay["post_norm"], eps))
            gt, up = _matvec(lay["gate"], h2), _matvec(lay["up"], h2)
            u = bf16_rne(np.array([gt[r] / (1 + math.exp(-gt[r])) * up[r] for r in range(len(gt))]))
            new_x.append(xi + _matvec(lay["down"], u))
        x = new_x
        taps.append(np.array(x))
    allowed = None
    if bitmask_row is not None:
        words = [int(v) & 0xFFFFFFFF for v in bitmask_row.tolist()]
        allowed = [(words[t // 32] >> (t % 32)) & 1 == 1 for t in range(geom.vocab)]
    drafts, p1s, logits = [], [], []
    for i in range(1, 1 + num_drafts):
        z = bf16_rne(_rms(x[i], _np(w["norm"]), eps))
        lg = LM @ z
        logits.append(lg)
        best, bi = -math.inf, -1
        for t in range(geom.vocab):
            if allowed is not None and not allowed[t]:
                continue
            if lg[t] > best:
                best, bi = lg[t], t
        if bi < 0:
            break
        tot = sum(math.exp(lg[t] - best) for t in range(geom.vocab)
                  if allowed is None or allowed[t])
        drafts.append(bi)
        p1s.append(1.0 / tot)
    conf = min(p1s) if p1s else 0.0
    return drafts, len(drafts), conf, np.array(logits), taps
