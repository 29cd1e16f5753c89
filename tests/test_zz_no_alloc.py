"""dflash_gemm_noalloc: the GEMM for callers that may not allocate device
memory while running (an engine whose arena already owns the GPU, or a decode
loop that cannot take cudaMalloc's device-wide synchronisation). On two calls
in a row (its fixed scratch array keeps the previous call's contents) it must
give the same result as the allocating GEMM entry point, and both must match
an fp32 matmul of the same bf16 inputs. Collected last so that a
stop-at-first-failure run has run every other test first."""
import ctypes as C

import pytest
import torch

from block_diffusion_speculative_forward_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from block_diffusion_speculative_forward_gb300 import build
    build.build()
    L = B.lib()
    for name in ("dflash_gemm_noalloc", "dflash_debug_gemm"):
        f = getattr(L, name)
        f.restype = C.c_int
    L.dflash_gemm_noalloc.argtypes = [C.c_void_p] * 3 + [C.c_int32] * 3 + [C.c_void_p]
    L.dflash_debug_gemm.argtypes = [C.c_void_p] * 3 + [C.c_int32] * 4 + [C.c_void_p]
    return L


def _run(L, fn, w, x, m, n, k):
    y = torch.full((m, n), float("nan"), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    if fn == "noalloc":
        rc = L.dflash_gemm_noalloc(w.data_ptr(), x.data_ptr(), y.data_ptr(), m, n, k, s)
    else:
        rc = L.dflash_debug_gemm(w.data_ptr(), x.data_ptr(), y.data_ptr(), m, n, k, 0, s)
    assert rc == 0, (fn, rc)
    return y


def test_noalloc_matches_allocating_gemm_twice(lib):
    cases = [(16, 5120, 2048), (15, 2048, 4096)]     # two calls in a row, different shapes
    for i, (m, n, k) in enumerate(cases):
        g = torch.Generator(device="cuda").manual_seed(100 + i)
        w = (torch.randn(n, k, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        x = torch.randn(m, k, device="cuda", generator=g).to(torch.bfloat16)
        ref = _run(lib, "alloc", w, x, m, n, k)
        got = _run(lib, "noalloc", w, x, m, n, k)
        err = (got - ref).abs().max().item()
        assert err <= 1e-3 * max(1.0, ref.abs().max().item()), (i, err)
        # both against an fp32 matmul of the bf16 operands
        mm = x.float() @ w.float().T
        tol = 1e-3 * max(1.0, mm.abs().max().item())
        assert (got - mm).abs().max().item() <= tol, (i, "noalloc vs fp32 matmul")
        assert (ref - mm).abs().max().item() <= tol, (i, "allocating GEMM vs fp32 matmul")


def test_noalloc_rejects_oversize(lib):
    w = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(17, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(17, 128, device="cuda")
    rc = lib.dflash_gemm_noalloc(w.data_ptr(), x.data_ptr(), y.data_ptr(), 17, 128, 64,
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == -1
