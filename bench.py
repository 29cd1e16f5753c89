"""Benchmark of the draft-head propose forward on GB300.

A step is one dflash_propose of the whole hot path (ctx append of the new
target row: fc, hidden_norm, fused K/V, k_norm, RoPE, paged write; the
gamma-row block through all layers; final norm, lm_head, argmax, confidence),
followed by the host-only after_verify. The default workload is the shipped
geometry at batch 1: 8 layers, hidden 2048, 32/4 heads of 128, vocab 248320,
gamma 16 (15 drafts), ctx 1024, one new row per step. Inputs are seeded
synthetic tensors; weights are random N(0, 0.02) (no checkpoint exists here).

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]

N > 1 runs under torchrun: every rank runs its own replica (the single-
sequence path does not shard); value = drafted tokens of all ranks / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from block_diffusion_speculative_forward_gb300 import synthetic as syn  # noqa: E402

METRIC = "drafted tokens/s (gamma=16, batch 1)"
UNIT = "tokens/s"
PATH = "auto"   # few-row propose path (--path)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


def max_over_ranks(vals, dist, device):
    """The slowest rank's value of each timing (the job is as slow as it)."""
    if dist is None:
        return list(vals)
    t = torch.tensor([float(v) for v in vals], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def shard(n, rank, world):
    """Sequences of a sequence-partitioned batch that this rank runs: every
    sequence is independent given the (replicated) weights, so the shards
    need no exchange on the data path."""
    return list(range(rank, n, world))


def head_cfg(geom, max_batch, max_seq_len, **kw):
    c = dict(num_layers=geom.num_layers, hidden=geom.hidden, intermediate=geom.intermediate,
             num_q_heads=geom.num_q_heads, num_kv_heads=geom.num_kv_heads,
             head_dim=geom.head_dim, vocab=geom.vocab, gamma=geom.gamma,
             mask_token_id=geom.mask_token_id, n_target_layers=geom.n_target_layers,
             target_hidden=geom.target_hidden, rms_eps=geom.rms_eps,
             ctx_window=geom.ctx_window, kv_block=geom.kv_block,
             prefill_chunk=geom.prefill_chunk, max_batch=max_batch, max_seq_len=max_seq_len,
             kv_pool_blocks=0, kv_dtype=0, lm_head_dtype=0)
    c.update(kw)
    return c


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- workloads --
def build_b1(geom, seed, ctx, n_steps_total, extra_positions=0):
    """Head + one sequence prefilled with ctx-1 rows; device rows for every
    step's new target row; pinned host copies of the same rows. The state's
    budget leaves extra_positions more positions for later steps."""
    from block_diffusion_speculative_forward_gb300 import binding as B
    w = syn.make_weights(geom, seed)
    wd = B.weights_to_device(w)
    cfg = head_cfg(geom, 1, ctx + n_steps_total + extra_positions + 64)
    head = B.DraftHead(cfg, wd)
    if PATH != "auto":
        head.set_chain(PATH == "chained")
    st = head.alloc_state()
    head.prefill(st, syn.make_stack(geom, ctx - 1, seed).cuda())
    rows_host = syn.make_stack(geom, n_steps_total + 1, seed, idx=1).pin_memory()
    rows_dev = rows_host.cuda()
    torch.cuda.synchronize()
    return w, wd, head, st, rows_dev, rows_host, cfg


def lm_head_bytes(geom, n_rows):
    """Algorithmic bytes of the lm_head stage: the vocab table once, the draft
    rows' z in, (id, p1) per row out."""
    return 2 * geom.vocab * geom.hidden + 2 * n_rows * geom.hidden + 8 * n_rows


def step_bytes(geom, ctx, n_new):
    wb = syn.weight_bytes(geom)
    kv_row = geom.num_layers * 2 * geom.kv_dim * 2
    return sum(wb.values()) + ctx * kv_row + n_new * geom.stack_width * 2


def run_ours(args):
    from block_diffusion_speculative_forward_gb300 import binding as B
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    geom, seed, ctx = syn.FULL, 1002, 1024
    nd = geom.gamma - 1
    K, W = args.steps, args.warmup
    KP = min(K, 50)                       # steps of the probed (instrumented) loop
    total = 2 * (K + W) + KP + 6
    K16, W16 = max(3, K // 10), 3
    w, wd, head, st, rows_dev, rows_host, cfg = build_b1(geom, seed, ctx, total,
                                                         geom.gamma * (K16 + W16 + 2))
    lib = B.lib()
    stream = torch.cuda.current_stream()
    pos = ctx
    used = 0

    def step(row):
        nonlocal pos
        d, n, c = head.propose(st, 1000 + pos % 1000, pos, row, nd)
        head.after_verify(st, 0)
        pos += 1
        return d

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pb, pe = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sb, se = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for e in (pb, pe, sb, se):
        e.record(stream)   # creates the events so their handles exist
    torch.cuda.synchronize()
    import ctypes as C
    lib.dflash_debug_set_probe.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p]
    lib.dflash_debug_set_step_probe.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p]
    lib.dflash_debug_launch_count.restype = C.c_int64
    for _ in range(W):
        step(rows_dev[used:used + 1])
        used += 1
    # device-timed region, inputs resident, no probes in the replayed graph
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = lib.dflash_debug_launch_count()
    with ClockSampler(local) as clk:
        torch.cuda.nvtx.range_push("propose_rounds")   # (selects the steps in a profiler)
        ev0.record(stream)
        for _ in range(K):
            step(rows_dev[used:used + 1])
            used += 1
        ev1.record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    launches = lib.dflash_debug_launch_count() - launches0
    t_ms = ev0.elapsed_time(ev1)
    # then the probes (events around the lm_head stage and the whole forward,
    # recorded inside the graph, so a probed graph is captured first): the
    # roofline's kernel time and the device time per step
    lib.dflash_debug_set_probe(head.ptr, C.c_void_p(pb.cuda_event), C.c_void_p(pe.cuda_event))
    lib.dflash_debug_set_step_probe(head.ptr, C.c_void_p(sb.cuda_event), C.c_void_p(se.cuda_event))
    probe_ms, dev_ms = [], []
    for i in range(KP + 2):
        step(rows_dev[used:used + 1])
        used += 1
        if i >= 2:
            probe_ms.append(pb.elapsed_time(pe))
            dev_ms.append(sb.elapsed_time(se))
    lib.dflash_debug_set_probe(head.ptr, None, None)
    lib.dflash_debug_set_step_probe(head.ptr, None, None)
    # end to end through the public call, host buffers: H2D of the step's new
    # row from pinned memory inside the timed region; drafts come back to host.
    for _ in range(2):
        step(rows_host[used:used + 1])
        used += 1
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(K):
        step(rows_host[used:used + 1])
        used += 1
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    try:
        new16 = run_b1_new16(lib, head, st, pos, geom, seed, nd, K16, W16)
    except Exception as e:   # reported in the line; never fatal for the metric's leg
        new16 = {"error": f"{type(e).__name__}: {e}"[:300]}
    t_ms, e2e_s = max_over_ranks([t_ms, e2e_s], dist, "cuda")
    hbm, tf, src = peaks()
    lm_ms = statistics.mean(probe_ms)
    lm_bytes = lm_head_bytes(geom, nd)
    lm_kernel = "lm_head stage (GEMM over the vocab + argmax/confidence)"
    lib.dflash_debug_last_path.argtypes = [C.c_void_p]
    chained = lib.dflash_debug_last_path(head.ptr) == 1
    achieved = lm_bytes / (lm_ms * 1e-3) / 1e9
    traffic = None if chained else args.lm_traffic
    sbytes = step_bytes(geom, ctx, 1)
    dev_med = statistics.median(dev_ms)
    out = {
        "metric": METRIC, "value": world * K * nd / (t_ms * 1e-3), "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": t_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded; random-init weights of the shipped drafter geometry)",
        "config": {"workload": "full_b1: L=8 H=2048 heads 32/4x128 I=6144 V=248320 gamma=16 "
                               "ctx=1024 n_new=1 drafts=15",
                   "batch": 1, "ctx": ctx, "gamma": geom.gamma, "num_drafts": nd,
                   "l2": "no flush: every step streams 1.98 GB of weights, > 129 MB L2",
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": world * K * nd / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": geom.stack_width * 2,
                "d2h_bytes_per_step": 4 * nd + 12},
        "gpu_launches": int(launches),
        # the whole propose step as the roofline's unit: every weight and the
        # window's K/V read once, over the device time of the step's kernels
        # (CUDA events at its first and after its last kernel, on its stream)
        "roofline": {"bound": "hbm", "achieved": sbytes / (dev_med * 1e-3) / 1e9, "peak": hbm,
                     "unit": "GB/s", "frac": sbytes / (dev_med * 1e-3) / 1e9 / hbm,
                     "traffic": None,
                     "traffic_note": "per-kernel ncu DRAM bytes are in profiles/ (launch lists)",
                     "kernel": "whole propose step (all kernels of one dflash_propose)",
                     "peak_source": f"{src} hbm_gbs",
                     "algorithmic_bytes_per_launch": sbytes, "avg_ms": dev_med,
                     "wall_frac": sbytes / (t_ms / K * 1e-3) / 1e9 / hbm},
        "lm_head_roofline": ({"note": "the chained path runs the lm_head inside its single "
                                      "persistent launch; the step roofline covers it"}
                             if chained else
                             {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                              "frac": achieved / hbm, "traffic": traffic,
                              "traffic_note": "ncu constant for the build named in profiles/"
                                              "lm_head_b1_dram_traffic.md, or null",
                              "kernel": lm_kernel,
                              "peak_source": f"{src} hbm_gbs",
                              "algorithmic_bytes_per_launch": lm_bytes, "avg_ms": lm_ms}),
        "path": "chained" if chained else "kernel per step",
        "propose_us": 1e3 * t_ms / K,
        "device_us": 1e3 * statistics.median(dev_ms),
        "device_spread": spread(dev_ms),
        "clocks": clk.summary(),
        "b1_new16": new16,
    }
    head.close()
    del wd
    torch.cuda.empty_cache()
    if not args.no_batch:
        # the metric's batch-32 leg: 32 sequences, gamma 16, ragged ctx, bitmask
        out["batch32"] = run_batched(syn.FULL, 1004, 32, 256, 4096, 15, False, True,
                                     max(3, K // 2), W)
        out["batch32"]["workload"] = ("full_b32: propose_batch of 32 sequences, ctx U[256,4096], "
                                      "new rows U[1,16], 50% bitmask, confidence on")
        torch.cuda.empty_cache()
    if not args.no_window:
        # the ctx_window cap: 8192-row prompt, 4096-row window, 64 rounds
        out["window"] = run_window(64, W)
        torch.cuda.empty_cache()
    if not args.no_lowp:
        # the metric's batch-1 step with the lm_head streamed as FP8 / NVFP4 codes
        for fmt in ("fp8", "nvfp4"):
            out[f"b1_lm_{fmt}"] = run_b1_lowp(fmt, max(5, K // 2), W)
            torch.cuda.empty_cache()
    if not args.no_fp8:
        # FP8 lm_head and FP8 KV cache, 128 sequences, gamma 8, 32 rounds
        out["fp8_b128"] = run_batched(syn.FULL_G8, 1005, 128, 512, 4096, 7, True, False, 32, W)
        out["fp8_b128"]["workload"] = ("fp8_b128: propose_batch of 128 sequences, gamma 8, "
                                       "ctx U[512,4096], FP8 E4M3 lm_head (row scales) and KV "
                                       "cache (per-head scales), 32 propose/after_verify rounds")
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(w, cfg, geom, seed, ctx, args.cpu_steps)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


def run_b1_new16(lib, head, st, pos, geom, seed, nd, K, W):
    """The batch-1 propose when a round accepted every draft: each propose
    brings gamma new ctx rows (the last token's and the accepted drafts'
    target hiddens), so the fc, hidden_norm, fused K/V and paged write run
    over 16 rows on top of the block forward. st must be due at position pos
    with one new row; device rows, inputs resident."""
    import ctypes as C
    g = geom.gamma
    rows = syn.make_stack(geom, g * (K + W + 2), seed, idx=2).cuda()
    s = torch.cuda.current_stream()
    sb, se = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for e in (sb, se):
        e.record(s)
    torch.cuda.synchronize()
    lib.dflash_debug_set_step_probe(head.ptr, C.c_void_p(sb.cuda_event), C.c_void_p(se.cuda_event))
    dev_ms, used = [], 0

    def propose(n_rows):
        nonlocal pos, used
        _, n_out, _ = head.propose(st, 1000 + pos % 1000, pos, rows[used:used + n_rows], nd)
        used += n_rows
        if n_out != nd:
            raise RuntimeError(f"{n_out} drafts where {nd} were expected")
        head.after_verify(st, nd)
        pos += nd + 1
        dev_ms.append(sb.elapsed_time(se))

    try:
        propose(1)   # the round whose drafts are all accepted
        for _ in range(W):
            propose(g)
        dev_ms.clear()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(s)
        for _ in range(K):
            propose(g)
        e1.record(s)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / K
    finally:
        lib.dflash_debug_set_step_probe(head.ptr, None, None)
    return {"n_new": g, "value": nd / (ms * 1e-3), "unit": UNIT, "propose_us": 1e3 * ms,
            "device_spread": spread(dev_ms), "steps": K, "warmup": W,
            "bytes_per_step": step_bytes(geom, pos - g, g)}


def batched_phases(geom, ctx_list, n_new_list, nd, kv_elem):
    """Algorithmic (FLOPs, HBM bytes) of each phase of one propose_batch step:
    the block rows through the layers' GEMMs, the lm_head over the draft rows,
    the new ctx rows' projections (fc + fused K/V) and the attention over the
    ctx windows; every weight and every stored ctx K/V row read once."""
    H, I, L, S = geom.hidden, geom.intermediate, geom.num_layers, geom.stack_width
    n = len(ctx_list)
    R, D, m = n * geom.gamma, n * nd, sum(n_new_list)
    layer_w = geom.q_dim * H + 2 * geom.kv_dim * H + H * geom.q_dim + 3 * I * H
    wb = syn.weight_bytes(geom)
    keys = sum(c + geom.gamma for c in ctx_list)
    return {
        "layers": (2 * R * layer_w * L, wb["layers"]),
        "lm_head": (2 * D * geom.vocab * H, geom.vocab * H * (1 if kv_elem == 1 else 2)),
        "ctx_rows": (2 * m * (H * S + L * 2 * geom.kv_dim * H), wb["fc"]),
        "attention": (4 * geom.gamma * geom.q_dim * keys * L,
                      sum(ctx_list) * L * 2 * geom.kv_dim * kv_elem),
    }


def phase_roofline(phases, t_ms, tf, hbm):
    """T_roof = sum over phases of max(F / P, B / BW) against the measured step
    time: the fraction of the roofline the whole step reaches when every phase
    sits on its own bound."""
    out, t_roof = {}, 0.0
    for name, (f, b) in phases.items():
        t_f, t_b = f / (tf * 1e12), b / (hbm * 1e9)
        t_roof += max(t_f, t_b)
        out[name] = {"tflop": f / 1e12, "gb": b / 1e9, "bound": "tensor" if t_f >= t_b else "hbm",
                     "t_roof_us": 1e6 * max(t_f, t_b)}
    return {"t_roof_us": 1e6 * t_roof, "frac": t_roof / (t_ms * 1e-3), "phases": out}


def spread(ms):
    """Median, 10th and 90th percentile of per-step times in ms, as us."""
    if len(ms) < 2:
        return {"median_us": 1e3 * ms[0], "p10_us": 1e3 * ms[0], "p90_us": 1e3 * ms[0]}
    q = statistics.quantiles(ms, n=10, method="inclusive")
    return {"median_us": 1e3 * statistics.median(ms), "p10_us": 1e3 * q[0], "p90_us": 1e3 * q[-1]}


def run_batched(geom, seed, n, ctx_lo, ctx_hi, nd, fp8, use_mask, K, W):
    """propose_batch over n sequences with ragged ctx; each step brings the
    target rows of the drafts the previous verify accepted (1..gamma rows)."""
    from block_diffusion_speculative_forward_gb300 import binding as B
    steps = K + W + 2
    w = syn.make_weights(geom, seed, lm_head_fp8=fp8, kv_fp8=fp8)
    wd = B.weights_to_device(w)
    del w
    cfg = head_cfg(geom, n, ctx_hi + geom.gamma * (steps + 2), kv_dtype=int(fp8),
                   lm_head_dtype=int(fp8))
    head = B.DraftHead(cfg, wd)
    ctx = syn.uniform_ints(ctx_lo, ctx_hi, n, seed, 1)
    states, tails = [], []
    for i in range(n):
        g = torch.Generator(device="cuda").manual_seed(seed * 1000 + i)
        stack = torch.randn((ctx[i] + geom.gamma * steps, geom.stack_width), device="cuda",
                            generator=g).to(torch.bfloat16)
        st = head.alloc_state()
        head.prefill(st, stack[:ctx[i]])
        torch.cuda.synchronize()
        tails.append(stack[ctx[i]:].clone())
        states.append(st)
        del stack
    mask = syn.make_bitmask(geom.vocab, n, seed).cuda() if use_mask else None
    pos, used = list(ctx), [0] * n
    n_new = syn.uniform_ints(1, geom.gamma, n, seed, 2)
    work = []

    # Every step's inputs (target rows, last tokens, accept counts) are drawn
    # before the timed region; a step is one propose_batch plus the verify
    # bookkeeping of every sequence.
    plan = []
    for t in range(W + K):
        rows = [tails[i][used[i]:used[i] + n_new[i]] for i in range(n)]
        for i in range(n):
            used[i] += n_new[i]
        newpos = [p + m for p, m in zip(pos, n_new)]
        toks = syn.uniform_ints(0, geom.vocab - 1, n, seed, 900 + t)
        ks = syn.uniform_ints(0, nd, n, seed, 1900 + t)
        plan.append((rows, toks, newpos, ks))
        if t >= W:
            work.append(batched_phases(geom, [p - m for p, m in zip(newpos, n_new)], n_new, nd,
                                       1 if fp8 else 2))
        pos = newpos
        n_new = [k + 1 for k in ks]
    host = [0.0, 0.0]
    # device time of each propose_batch forward (events recorded at the first
    # and after the last kernel of the forward, inside its graph)
    import ctypes as C
    lib = B.lib()
    lib.dflash_debug_set_step_probe.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p]
    sb, se = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for e in (sb, se):
        e.record(torch.cuda.current_stream())
    torch.cuda.synchronize()
    lib.dflash_debug_set_step_probe(head.ptr, C.c_void_p(sb.cuda_event), C.c_void_p(se.cuda_event))
    dev_ms = []

    def step(t):
        rows, toks, newpos, ks = plan[t]
        t0 = time.perf_counter()
        head.propose_batch(states, toks, newpos, rows, nd, bitmask=mask)
        t1 = time.perf_counter()
        dev_ms.append(sb.elapsed_time(se))
        head.after_verify_batch(states, ks)
        host[0] += t1 - t0
        host[1] += time.perf_counter() - t1

    for t in range(W):
        step(t)
    host[0] = host[1] = 0.0
    dev_ms.clear()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.nvtx.range_push("propose_rounds")   # (selects the rounds in a profiler)
        e0.record(s)
        for t in range(W, W + K):
            step(t)
        e1.record(s)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    ms = e0.elapsed_time(e1) / K
    phases = {name: (sum(w[name][0] for w in work) / K, sum(w[name][1] for w in work) / K)
              for name in work[0]}
    flops = sum(f for f, _ in phases.values())
    byts = sum(b for _, b in phases.values())
    hbm, tf, src = peaks()
    lib.dflash_debug_set_step_probe(head.ptr, None, None)
    head.close()
    return {"value": n * nd / (ms * 1e-3), "unit": UNIT, "propose_us": 1e3 * ms,
            "device_us": 1e3 * statistics.median(dev_ms),
            "device_spread": spread(dev_ms),
            "batch": n, "gamma": geom.gamma, "num_drafts": nd, "steps": K, "warmup": W,
            "ctx": f"U[{ctx_lo},{ctx_hi}]", "bitmask": use_mask, "fp8_kv_and_lm_head": fp8,
            "flops_per_step": flops, "bytes_per_step": byts,
            "propose_call_us": 1e6 * host[0] / K, "verify_calls_us": 1e6 * host[1] / K,
            "clocks": clk.summary(),
            "roofline": {"bound": "tensor", "achieved": flops / (ms * 1e-3) / 1e12, "peak": tf,
                         "unit": "TFLOP/s", "frac": flops / (ms * 1e-3) / 1e12 / tf,
                         "peak_source": f"{src} bf16_tflops (burst)",
                         "hbm_frac": byts / (ms * 1e-3) / 1e9 / hbm},
            "phase_roofline": phase_roofline(phases, ms, tf, hbm)}


def run_window(K, W):
    """C3: one sequence with an 8192-row prompt and a 4096-row window (rows
    below the window are neither computed nor stored), then propose /
    after_verify rounds with accept counts drawn U[0, 15]; every round brings
    the k + 1 target rows the previous verify accepted."""
    from block_diffusion_speculative_forward_gb300 import binding as B
    geom, seed, prompt, window = syn.FULL, 1003, 8192, 4096
    nd = geom.gamma - 1
    rounds = K + W
    probed = 16                       # further rounds with the device-time probe
    w = syn.make_weights(geom, seed)
    wd = B.weights_to_device(w)
    del w
    cfg = head_cfg(geom, 1, prompt + geom.gamma * (rounds + probed + 2) + 64, ctx_window=window)
    head = B.DraftHead(cfg, wd)
    st = head.alloc_state()
    g = torch.Generator(device="cuda").manual_seed(seed)
    stack = torch.randn((prompt + geom.gamma * (rounds + probed + 2), geom.stack_width),
                        device="cuda", generator=g).to(torch.bfloat16)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    head.prefill(st, stack[:prompt - 1])
    torch.cuda.synchronize()
    prefill_ms = 1e3 * (time.perf_counter() - t0)
    ks = syn.uniform_ints(0, nd, rounds, seed, 7)
    pos, used, n_new = prompt - 1, prompt - 1, 1
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    import ctypes as C
    lib = B.lib()
    lib.dflash_debug_set_step_probe.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p]
    sb, se = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for e in (sb, se):
        e.record(s)
    torch.cuda.synchronize()
    dev_ms, round_bytes = [], []
    # the timed rounds and the device-time probe are separate passes over the
    # same call sequence shape: rounds W.. are timed without probes, then a
    # second set of rounds is probed
    clk = ClockSampler(torch.cuda.current_device())
    for r in range(rounds):
        if r == W:
            torch.cuda.synchronize()
            clk.__enter__()
            e0.record(s)
        pos += n_new
        got = head.propose(st, 1000 + r, pos, stack[used:used + n_new], nd)
        if r >= W:
            round_bytes.append(step_bytes(geom, min(window, pos - n_new), n_new))
        used += n_new
        k = min(ks[r], got[1])
        head.after_verify(st, k)
        n_new = k + 1
    e1.record(s)
    torch.cuda.synchronize()
    clk.__exit__()
    ms = e0.elapsed_time(e1) / K
    lib.dflash_debug_set_step_probe(head.ptr, C.c_void_p(sb.cuda_event), C.c_void_p(se.cuda_event))
    ks2 = syn.uniform_ints(0, nd, probed, seed, 8)
    for r in range(probed):
        pos += n_new
        got = head.propose(st, 2000 + r, pos, stack[used:used + n_new], nd)
        used += n_new
        if r >= 2:
            dev_ms.append(sb.elapsed_time(se))
        k = min(ks2[r], got[1])
        head.after_verify(st, k)
        n_new = k + 1
    lib.dflash_debug_set_step_probe(head.ptr, None, None)
    head.close()
    hbm, _, src = peaks()
    byts = statistics.mean(round_bytes)
    dev = statistics.median(dev_ms)
    return {"value": nd / (ms * 1e-3), "unit": UNIT, "propose_us": 1e3 * ms, "rounds": K,
            "warmup": W, "prompt": prompt, "ctx_window": window, "prefill_ms": prefill_ms,
            "device_us": 1e3 * dev, "device_spread": spread(dev_ms),
            "bytes_per_round": byts, "clocks": clk.summary(),
            "roofline": {"bound": "hbm", "achieved": byts / (dev * 1e-3) / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": byts / (dev * 1e-3) / 1e9 / hbm,
                         "wall_frac": byts / (ms * 1e-3) / 1e9 / hbm,
                         "peak_source": f"{src} hbm_gbs",
                         "kernel": "whole propose round (device time of its kernels)"},
            "workload": "full_b1_window: prompt 8192 (8191 prefilled, 4096-row window), then "
                        "64 propose/after_verify rounds, k ~ U[0, 15], k + 1 new rows per round"}


def lm_lowp_bytes(geom, fmt, n_rows):
    """Algorithmic bytes of the streamed lm_head stage: the codes and their
    scales once, the draft rows' z in, (id, p1) per row out."""
    V, H = geom.vocab, geom.hidden
    table = V * H + 4 * V if fmt == "fp8" else V * H // 2 + V * H // 16
    return table + 2 * n_rows * H + 8 * n_rows


def run_b1_lowp(fmt, K, W):
    """The batch-1 propose of the metric's workload with the lm_head
    streamed as codes: FP8 E4M3 with per-row scales, or NVFP4 (E2M1 codes,
    E4M3 scales per 16 elements, global scale). Device time per step and of
    the lm_head stage (CUDA events inside the replayed graph)."""
    from block_diffusion_speculative_forward_gb300 import binding as B
    import ctypes as C
    geom, seed, ctx = syn.FULL, 1002, 1024
    nd = geom.gamma - 1
    w = syn.make_weights(geom, seed, lm_head_fp8=fmt == "fp8", lm_head_nvfp4=fmt == "nvfp4")
    del w["lm_head"]
    w["lm_head"] = torch.empty(0, dtype=torch.bfloat16)   # not needed: the codes stream
    wd = B.weights_to_device(w)
    del w
    n_steps = K + W + 4
    cfg = head_cfg(geom, 1, ctx + n_steps + 64, lm_head_dtype=1 if fmt == "fp8" else 2)
    head = B.DraftHead(cfg, wd)
    st = head.alloc_state()
    head.prefill(st, syn.make_stack(geom, ctx - 1, seed).cuda())
    rows = syn.make_stack(geom, n_steps + 1, seed, idx=1).cuda()
    lib = B.lib()
    lib.dflash_debug_set_probe.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p]
    lib.dflash_debug_set_step_probe.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p]
    s = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in ev:
        e.record(s)
    torch.cuda.synchronize()
    pos, used = ctx, 0

    def step():
        nonlocal pos, used
        head.propose(st, 1000 + pos % 1000, pos, rows[used:used + 1], nd)
        head.after_verify(st, 0)
        pos += 1
        used += 1

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        ev[0].record(s)
        for _ in range(K):
            step()
        ev[1].record(s)
        torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1]) / K
    lib.dflash_debug_set_probe(head.ptr, C.c_void_p(ev[2].cuda_event), C.c_void_p(ev[3].cuda_event))
    lib.dflash_debug_set_step_probe(head.ptr, C.c_void_p(ev[4].cuda_event),
                                    C.c_void_p(ev[5].cuda_event))
    lm_ms, dev_ms = [], []
    for i in range(4):
        step()
        if i >= 2:
            lm_ms.append(ev[2].elapsed_time(ev[3]))
            dev_ms.append(ev[4].elapsed_time(ev[5]))
    lib.dflash_debug_set_probe(head.ptr, None, None)
    lib.dflash_debug_set_step_probe(head.ptr, None, None)
    head.close()
    hbm, _, src = peaks()
    lm_b = lm_lowp_bytes(geom, fmt, nd)
    wb = syn.weight_bytes(geom)
    sbytes = (sum(wb.values()) - wb["lm_head"] + lm_b + ctx * geom.num_layers * 2 * geom.kv_dim * 2
              + geom.stack_width * 2)
    lm, dev = statistics.mean(lm_ms), statistics.median(dev_ms)
    return {"value": nd / (ms * 1e-3), "unit": UNIT, "propose_us": 1e3 * ms, "steps": K,
            "warmup": W, "device_us": 1e3 * dev, "clocks": clk.summary(),
            "roofline": {"bound": "hbm", "achieved": sbytes / (dev * 1e-3) / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": sbytes / (dev * 1e-3) / 1e9 / hbm,
                         "peak_source": f"{src} hbm_gbs", "algorithmic_bytes_per_launch": sbytes,
                         "kernel": "whole propose step (device time of its kernels)"},
            "lm_head_roofline": {"bound": "hbm", "achieved": lm_b / (lm * 1e-3) / 1e9,
                                 "peak": hbm, "unit": "GB/s",
                                 "frac": lm_b / (lm * 1e-3) / 1e9 / hbm, "avg_ms": lm,
                                 "algorithmic_bytes_per_launch": lm_b, "traffic": None,
                                 "kernel": "k_lm_lowp (codes dequantised into TMEM) + merge"},
            "workload": f"full_b1 with the lm_head streamed as {fmt.upper()} codes "
                        f"(no bf16 table): ctx 1024, one new row, 15 drafts"}


def cpu_baseline(w, cfg, geom, seed, ctx, n_steps):
    """The oracle, as it stands, on the host cores: prefill untimed, then a
    bounded number of single-sequence proposes of the same workload."""
    import oracle
    ora = oracle.DraftHeadOracle(cfg, w)
    st = ora.alloc_state()
    ora.prefill(st, syn.make_stack(geom, ctx - 1, seed))
    rows = syn.make_stack(geom, n_steps + 2, seed, idx=1)
    ora.lm_head()
    pos = ctx
    ora.propose(st, 1, pos, rows[0:1], geom.gamma - 1)
    ora.after_verify(st, 0)
    pos += 1
    t0 = time.perf_counter()
    for i in range(n_steps):
        ora.propose(st, 1000 + pos % 1000, pos, rows[1 + i:2 + i], geom.gamma - 1)
        ora.after_verify(st, 0)
        pos += 1
    dt = time.perf_counter() - t0
    return {"value": n_steps * (geom.gamma - 1) / dt, "unit": UNIT,
            "cores": torch.get_num_threads(), "kind": "oracle",
            "sample": f"{n_steps} single-sequence proposes of full_b1 after an untimed "
                      f"{ctx - 1}-row prefill (torch CPU float64)",
            "s_per_propose": dt / n_steps}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    geom, seed, ctx = syn.FULL, 1002, 1024
    nd = geom.gamma - 1
    w = syn.make_weights(geom, seed)
    cfg = head_cfg(geom, 1, ctx + 4096)
    import oracle
    ora = oracle.DraftHeadOracle(cfg, w)
    st = ora.alloc_state()
    ora.prefill(st, syn.make_stack(geom, ctx - 1, seed))
    ora.lm_head()
    rows = syn.make_stack(geom, args.steps + args.warmup + 2, seed, idx=1)
    pos, used = ctx, 0
    for _ in range(args.warmup):
        ora.propose(st, 1, pos, rows[used:used + 1], nd)
        ora.after_verify(st, 0)
        pos += 1
        used += 1
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ora.propose(st, 1000 + pos % 1000, pos, rows[used:used + 1], nd)
        ora.after_verify(st, 0)
        pos += 1
        used += 1
    dt = time.perf_counter() - t0
    v = args.steps * nd / dt
    out = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded)",
           "config": {"workload": "full_b1: L=8 H=2048 heads 32/4x128 I=6144 V=248320 gamma=16 "
                                  "ctx=1024 n_new=1 drafts=15", "batch": 1},
           "cpu_baseline": {"value": v, "unit": UNIT, "cores": torch.get_num_threads(),
                            "kind": "oracle",
                            "sample": f"{args.steps} proposes after an untimed prefill"},
           "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_kernel_case(args):
    """One tensor-core GEMM at the lm_head shape (15 draft rows x 248320 vocab
    rows x 2048), 1.02 GB of bf16 weights, timed alone with CUDA events: the
    small case used for detailed profiles of the weight-streaming kernel.
    lm_head_b32: the many-row lm_head kernel at 480 draft rows (32 sequences
    x 15 drafts)."""
    import ctypes as C
    from block_diffusion_speculative_forward_gb300 import binding as B
    L = B.lib()
    if args.kernel == "lm_head_b32":
        L.dflash_debug_lmhead.argtypes = [C.c_void_p] * 3 + [C.c_int32] * 3 + [C.c_void_p]
        m, n, k = 480, syn.FULL.vocab, syn.FULL.hidden
        g = torch.Generator(device="cuda").manual_seed(6)
        w = (torch.randn(n, k, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        x = torch.randn(m, k, device="cuda", generator=g).to(torch.bfloat16)
        part = torch.empty(m * ((n + 255) // 256) * 4, dtype=torch.int32, device="cuda")
        s = torch.cuda.current_stream()
        times = []
        for i in range(args.warmup + args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            rc = L.dflash_debug_lmhead(w.data_ptr(), x.data_ptr(), part.data_ptr(), m, n, k,
                                       s.cuda_stream)
            e1.record(s)
            torch.cuda.synchronize()
            assert rc == 0, rc
            if i >= args.warmup:
                times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        _, tf, src = peaks()
        fl = 2.0 * m * n * k
        print(json.dumps({"kernel": "lm_head, 480 draft rows", "median_ms": ms,
                          "TFLOP/s": fl / (ms * 1e-3) / 1e12,
                          "frac_bf16": fl / (ms * 1e-3) / 1e12 / tf, "peak_source": src}))
        return
    L.dflash_gemm_noalloc.argtypes = [C.c_void_p] * 3 + [C.c_int32] * 3 + [C.c_void_p]
    m, n, k = 15, syn.FULL.vocab, syn.FULL.hidden
    g = torch.Generator(device="cuda").manual_seed(5)
    w = (torch.randn(n, k, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    x = torch.randn(m, k, device="cuda", generator=g).to(torch.bfloat16)
    y = torch.empty(m, n, device="cuda")
    s = torch.cuda.current_stream()
    times = []
    for i in range(args.warmup + args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        rc = L.dflash_gemm_noalloc(w.data_ptr(), x.data_ptr(), y.data_ptr(), m, n, k, s.cuda_stream)
        e1.record(s)
        torch.cuda.synchronize()
        assert rc == 0, rc
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    nbytes = 2 * n * k + 2 * m * k + 4 * m * n
    hbm, _, src = peaks()
    print(json.dumps({"kernel": "tcgen05 GEMM, lm_head shape", "m": m, "n": n, "k": k,
                      "median_ms": ms, "GB/s": nbytes / (ms * 1e-3) / 1e9,
                      "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm, "peak_source": src}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-steps", type=int, default=4)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-batch", action="store_true", help="skip the batch-32 leg")
    ap.add_argument("--batch-only", action="store_true",
                    help="only the batch-32 leg (for profiling it alone)")
    ap.add_argument("--no-window", action="store_true",
                    help="skip the 8192-row prompt / 4096-row window leg (64 rounds)")
    ap.add_argument("--no-lowp", action="store_true",
                    help="skip the batch-1 legs with the lm_head streamed as FP8 / NVFP4 codes")
    ap.add_argument("--no-fp8", action="store_true",
                    help="skip the 128-sequence FP8 leg (32 rounds)")
    ap.add_argument("--leg", default=None,
                    choices=["batch32", "window", "fp8_b128", "b1_lm_fp8", "b1_lm_nvfp4"],
                    help="run one secondary leg alone and print its JSON (for profiling it)")
    ap.add_argument("--path", default="auto", choices=["auto", "per-step", "chained"],
                    help="batch-1 leg: the library's default path, the kernel-per-step path, or "
                         "the chained single launch")
    ap.add_argument("--kernel", default=None, choices=["lm_head", "lm_head_b32"],
                    help="time one kernel alone instead of the propose step")
    # dram__bytes_read.sum + dram__bytes_write.sum of one batch-1 lm_head GEMM
    # launch (1,017,561,344 + 4,292,096 B), ncu at this workload; re-capture
    # (or pass None) whenever that kernel changes.
    ap.add_argument("--lm-traffic", type=float, default=1021853440.0,
                    help="ncu dram bytes per lm_head launch, when captured for this build")
    args = ap.parse_args()
    global PATH
    PATH = args.path
    if args.warmup < 3:
        args.warmup = 3
    if args.kernel:
        from block_diffusion_speculative_forward_gb300 import build
        build.build()
        run_kernel_case(args)
    elif args.leg:
        from block_diffusion_speculative_forward_gb300 import build
        build.build()
        if args.leg == "batch32":
            r = run_batched(syn.FULL, 1004, 32, 256, 4096, 15, False, True, args.steps, args.warmup)
        elif args.leg == "window":
            r = run_window(args.steps, args.warmup)
        elif args.leg == "fp8_b128":
            r = run_batched(syn.FULL_G8, 1005, 128, 512, 4096, 7, True, False, args.steps,
                            args.warmup)
        else:
            r = run_b1_lowp(args.leg[6:], args.steps, args.warmup)
        print(json.dumps({args.leg: r}), flush=True)
    elif args.batch_only:
        from block_diffusion_speculative_forward_gb300 import build
        build.build()
        r = run_batched(syn.FULL, 1004, 32, 256, 4096, 15, False, True, args.steps, args.warmup)
        print(json.dumps({"batch32": r}), flush=True)
    elif args.impl == "reference":
        run_reference(args)
    else:
        from block_diffusion_speculative_forward_gb300 import build
        if int(os.environ.get("LOCAL_RANK", "0")) == 0:
            build.build()
        run_ours(args)


if __name__ == "__main__":
    main()
