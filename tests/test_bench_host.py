"""bench.py's batch-1 and batched legs run end to end on the CPU against a
bookkeeping-only head (no weights, nothing computed), with CUDA events,
streams and device placement replaced by stand-ins: the call sequences, the
position and row budgets, the verify bookkeeping and the JSON assembly are
exercised without a GPU. Timings here are meaningless; only the flow and the
line's keys are checked."""
import importlib.util
import os
from dataclasses import replace

import pytest
import torch

from block_diffusion_speculative_forward_gb300 import binding as B
from tests.test_oracle_pins import MICRO

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMALL = replace(MICRO, hidden=256, gamma=16, ctx_window=4096, kv_block=16, vocab=4096,
                mask_token_id=4095)


class _Event:
    def __init__(self, **kw):
        pass

    def record(self, stream=None):
        pass

    def elapsed_time(self, other):
        return 1.5

    cuda_event = None


class _Stream:
    cuda_stream = None


@pytest.fixture
def bench(monkeypatch):
    from block_diffusion_speculative_forward_gb300 import build
    build.build()
    spec = importlib.util.spec_from_file_location("bench_under_test",
                                                  os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    monkeypatch.setattr(torch.cuda, "Event", _Event)
    monkeypatch.setattr(torch.cuda, "current_stream", lambda *a: _Stream())
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a: None)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(torch.cuda, "set_device", lambda *a: None)
    monkeypatch.setattr(torch.cuda, "empty_cache", lambda: None)
    monkeypatch.setattr(torch.Tensor, "cuda", lambda self, *a, **k: self)
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self, *a, **k: self)
    gen = torch.Generator
    monkeypatch.setattr(torch, "Generator", lambda device=None: gen())
    randn = torch.randn

    def cpu_randn(*a, **k):
        k.pop("device", None)
        return randn(*a, **k)

    monkeypatch.setattr(torch, "randn", cpu_randn)
    monkeypatch.setattr(B, "weights_to_device", lambda w, device="cuda": None)
    monkeypatch.setattr(b.syn, "FULL", SMALL)
    return b


def test_batch1_leg(bench):
    args = bench.argparse.Namespace(gpus=1, steps=12, warmup=3, impl="ours", cpu_steps=1,
                                    no_cpu=True, no_batch=True, batch_only=False,
                                    no_window=True, no_fp8=True, no_lowp=True, kernel=None,
                                    lm_traffic=1.0)
    out = {}
    bench.print = lambda s, **k: out.setdefault("line", s)
    bench.run_ours(args)
    line = bench.json.loads(out["line"])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e",
                "gpu_launches", "roofline", "clocks", "device_spread", "lm_head_roofline"):
        assert key in line, key
    assert line["roofline"]["kernel"].startswith("whole propose step")
    assert "error" not in line["b1_new16"], line["b1_new16"]


def test_window_leg(bench):
    r = bench.run_window(5, 3)
    assert r["rounds"] == 5 and r["ctx_window"] == 4096
    for key in ("roofline", "clocks", "device_spread", "workload", "device_us"):
        assert key in r, key
    assert r["roofline"]["frac"] > 0


@pytest.mark.parametrize("fp8", [False, True])
def test_batched_leg(bench, fp8):
    r = bench.run_batched(SMALL, 1004, 6, 64, 300, 15, fp8, not fp8, 5, 3)
    assert r["steps"] == 5 and r["batch"] == 6
    assert set(r["phase_roofline"]["phases"]) == {"layers", "lm_head", "ctx_rows", "attention"}
    assert r["phase_roofline"]["frac"] > 0 and r["device_spread"]["p90_us"] > 0
