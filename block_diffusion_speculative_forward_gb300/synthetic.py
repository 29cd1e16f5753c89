"""Seeded synthetic inputs for the block-diffusion draft head.

This module only DRAWS data: drafter weights, target hidden stacks, tokens,
accept counts and grammar bitmasks, each from its own fixed seed, on the CPU.
It holds none of the draft head's arithmetic. Both the CUDA path (through the
C-ABI) and the CPU oracle consume exactly these tensors, so neither side ever
produces an input for the other.

Two inputs are tables that a checkpoint loader builds and hands to the head
("Struct BlockDiffusionDraftHead", fields ``yarn_inv_freq`` and
``lm_head_shared_fp8``): the RoPE inverse-frequency table and the FP8 mirror of
the shared lm_head. They are built here the way a loader would build them.

Recipe (every tensor has its own ``torch.Generator`` seeded with
``seed * 1000 + tensor_index`` so any subset can be regenerated alone):
  * matrices: N(0, 0.02) in fp32, rounded to bf16;
  * RMSNorm gains: 1 + N(0, 0.02), rounded to bf16 (gains start at one);
  * embed and lm_head: two separate N(0, 0.02) [vocab, hidden] tables;
  * target hidden stacks: N(0, 1) bf16, ``[rows, n_target_layers * target_hidden]``;
  * inv_freq[i] = theta ** (-2 i / head_dim), evaluated in double, stored f32;
  * FP8 lm_head: per-row scale amax/448, codes = e4m3(w / scale) (torch cast);
  * NVFP4 lm_head: a power-of-two global scale at or above amax/(448*6), one
    E4M3 scale per 16 elements of a row = e4m3(block amax / (6 * global))
    (torch cast), E2M1 codes of w / (scale * global) at the nearest magnitude
    (ties to the smaller), packed two per byte, element 2j in the low nibble;
  * FP8 KV scales: U[6, 10] / 448 per (layer, kv head, K|V).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

LAYER_KEYS = ("in_norm", "q", "k", "v", "q_norm", "k_norm", "o", "post_norm",
              "gate", "up", "down")


@dataclass(frozen=True)
class Geometry:
    num_layers: int
    hidden: int
    intermediate: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    vocab: int
    gamma: int
    mask_token_id: int
    n_target_layers: int
    target_hidden: int
    rope_theta: float
    rms_eps: float = 1e-6
    ctx_window: int = 4096
    kv_block: int = 16
    prefill_chunk: int = 512

    @property
    def stack_width(self) -> int:
        return self.n_target_layers * self.target_hidden

    @property
    def kv_dim(self) -> int:
        return self.num_kv_heads * self.head_dim

    @property
    def q_dim(self) -> int:
        return self.num_q_heads * self.head_dim


# Tiny drafter: 1 layer, hidden 256, 4 q / 2 kv heads of 64, vocab 4096.
TINY = Geometry(num_layers=1, hidden=256, intermediate=512, num_q_heads=4,
                num_kv_heads=2, head_dim=64, vocab=4096, gamma=4,
                mask_token_id=4095, n_target_layers=2, target_hidden=256,
                rope_theta=1e6)

# Shipped drafter geometry: 8 layers, hidden 2048, 32 q / 4 kv heads of 128,
# intermediate 6144, vocab 248320, 5 captured target layers of 2048, theta 1e7.
# The mask token is the last vocab id, as in the tiny drafter.
FULL = Geometry(num_layers=8, hidden=2048, intermediate=6144, num_q_heads=32,
                num_kv_heads=4, head_dim=128, vocab=248320, gamma=16,
                mask_token_id=248319, n_target_layers=5, target_hidden=2048,
                rope_theta=1e7)

FULL_G8 = replace(FULL, gamma=8)


def _gen(seed: int, idx: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed * 1000 + idx)
    return g


def _normal(shape, std, seed, idx, mean=0.0):
    t = torch.randn(shape, generator=_gen(seed, idx), dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(torch.bfloat16)


def make_inv_freq(head_dim: int, theta: float) -> torch.Tensor:
    """[head_dim/2] f32 table theta^(-2i/head_dim), evaluated in double."""
    return torch.tensor([theta ** (-2.0 * i / head_dim) for i in range(head_dim // 2)],
                        dtype=torch.float64).to(torch.float32)


def make_weights(geom: Geometry, seed: int, *, lm_head_fp8: bool = False,
                 kv_fp8: bool = False, lm_head_nvfp4: bool = False) -> dict:
    """All drafter weights (CPU tensors). bf16 unless noted."""
    H, I, S = geom.hidden, geom.intermediate, geom.stack_width
    w = {
        "embed": _normal((geom.vocab, H), 0.02, seed, 0),
        "lm_head": _normal((geom.vocab, H), 0.02, seed, 1),
        "fc": _normal((H, S), 0.02, seed, 2),
        "hidden_norm": _normal((H,), 0.02, seed, 3, mean=1.0),
        "norm": _normal((H,), 0.02, seed, 4, mean=1.0),
        "inv_freq": make_inv_freq(geom.head_dim, geom.rope_theta),
        "layers": [],
    }
    shapes = {"in_norm": (H,), "q": (geom.q_dim, H), "k": (geom.kv_dim, H),
              "v": (geom.kv_dim, H), "q_norm": (geom.head_dim,),
              "k_norm": (geom.head_dim,), "o": (H, geom.q_dim),
              "post_norm": (H,), "gate": (I, H), "up": (I, H), "down": (H, I)}
    for l in range(geom.num_layers):
        layer = {}
        for j, key in enumerate(LAYER_KEYS):
            idx = 100 + l * 20 + j
            if key.endswith("norm"):
                layer[key] = _normal(shapes[key], 0.02, seed, idx, mean=1.0)
            else:
                layer[key] = _normal(shapes[key], 0.02, seed, idx)
        w["layers"].append(layer)
    if lm_head_fp8:
        lm = w["lm_head"].to(torch.float32)
        scale = lm.abs().amax(dim=1) / 448.0
        scale = torch.where(scale > 0, scale, torch.ones_like(scale))
        codes = (lm / scale[:, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
        w["lm_head_fp8"] = codes
        w["lm_head_scale"] = scale.to(torch.float32)
    if lm_head_nvfp4:
        p, sc, g = quantize_nvfp4(w["lm_head"])
        w["lm_head_nvfp4"], w["lm_head_nvfp4_scale"] = p, sc
        w["lm_head_nvfp4_global"] = torch.tensor(g, dtype=torch.float32)
    if kv_fp8:
        u = torch.rand((geom.num_layers, geom.num_kv_heads, 2), generator=_gen(seed, 7),
                       dtype=torch.float32)
        w["kv_scale"] = ((6.0 + 4.0 * u) / 448.0).to(torch.float32)
    return w


def quantize_nvfp4(w: torch.Tensor, rows_per_pass: int = 8192):
    """NVFP4 encoding of a [rows, k] table (k % 16 == 0), the way a
    checkpoint carries an NVFP4 lm_head: (packed E2M1 codes [rows, k/2] uint8,
    E4M3 block scales [rows, k/16] uint8, f32 global scale)."""
    rows, k = w.shape
    top = float(w.to(torch.float32).abs().max()) if w.numel() else 0.0
    # the smallest power of two that keeps every block scale within E4M3's 448
    g = 2.0 ** math.ceil(math.log2(top / (448.0 * 6.0))) if top > 0 else 1.0
    mids = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])   # between E2M1 magnitudes
    packed = torch.empty((rows, k // 2), dtype=torch.uint8)
    scales = torch.empty((rows, k // 16), dtype=torch.uint8)
    for r0 in range(0, rows, rows_per_pass):
        x = w[r0:r0 + rows_per_pass].to(torch.float32).reshape(-1, k // 16, 16)
        s8 = (x.abs().amax(dim=2) / (6.0 * g)).clamp(max=448.0).to(torch.float8_e4m3fn)
        sv = s8.to(torch.float32)
        q = (x / (torch.where(sv > 0, sv, torch.ones_like(sv))[..., None] * g)).clamp(-6.0, 6.0)
        code = torch.bucketize(q.abs(), mids) | ((q < 0).to(torch.int64) << 3)
        code = code.reshape(x.shape[0], k)
        packed[r0:r0 + x.shape[0]] = (code[:, 0::2] | (code[:, 1::2] << 4)).to(torch.uint8)
        scales[r0:r0 + x.shape[0]] = s8.view(torch.uint8)
    return packed, scales, g


def make_stack(geom: Geometry, n_rows: int, seed: int, idx: int = 0) -> torch.Tensor:
    """Target hidden stack rows [n_rows, n_target_layers*target_hidden], N(0,1) bf16."""
    return _normal((n_rows, geom.stack_width), 1.0, seed, 50_000 + idx)


def make_bitmask(vocab: int, n: int, seed: int, idx: int = 0) -> torch.Tensor:
    """[n, ceil(vocab/32)] int32 words with each bit set with probability 1/2."""
    words = (vocab + 31) // 32
    g = _gen(seed, 60_000 + idx)
    u = torch.randint(0, 2 ** 32, (n, words), generator=g, dtype=torch.int64)
    return (u - (u >= 2 ** 31).to(torch.int64) * 2 ** 32).to(torch.int32)


def uniform_ints(lo: int, hi: int, n: int, seed: int, idx: int) -> list[int]:
    """n integers uniform in [lo, hi] (inclusive)."""
    g = _gen(seed, 70_000 + idx)
    return [int(v) for v in torch.randint(lo, hi + 1, (n,), generator=g)]


def weight_bytes(geom: Geometry) -> dict:
    """Bytes of every weight the propose forward streams once (bf16)."""
    H, I = geom.hidden, geom.intermediate
    per_layer = 2 * (geom.q_dim * H + 2 * geom.kv_dim * H + H * geom.q_dim + 3 * I * H
                     + 2 * H + 2 * geom.head_dim)
    return {"layers": geom.num_layers * per_layer,
            "fc": 2 * H * geom.stack_width,
            "lm_head": 2 * geom.vocab * H}


# The five workloads. Sizes only; the drivers (tests, bench) run their call
# sequences.
WORKLOADS = {
    "tiny_b1": dict(geom=TINY, seed=1001, n_seq=1, ctx=64, n_new=0, num_drafts=3),
    "full_b1": dict(geom=FULL, seed=1002, n_seq=1, ctx=1023, n_new=1, num_drafts=15),
    "full_b1_window": dict(geom=FULL, seed=1003, n_seq=1, prompt=8192, ctx_window=4096,
                           rounds=64, num_drafts=15),
    "full_b32": dict(geom=FULL, seed=1004, n_seq=32, ctx_lo=256, ctx_hi=4096,
                     new_lo=1, new_hi=16, num_drafts=15, bitmask=True),
    "fp8_b128": dict(geom=FULL_G8, seed=1005, n_seq=128, ctx_lo=512, ctx_hi=4096,
                     rounds=32, num_drafts=7, fp8=True),
}
