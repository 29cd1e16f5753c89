"""The tensor-core GEMM (tcgen05 + TMA, stream-K) in isolation against a
plain PyTorch fp32 matmul of the same bf16 operands, over tile widths, ragged
row and column counts and forced split k-ranges."""
import ctypes as C

import pytest
import torch

from block_diffusion_speculative_forward_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_diffusion_speculative_forward_gb300 import build
    build.build()
    L = B.lib()
    L.dflash_debug_gemm.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                    C.c_int32, C.c_int32, C.c_void_p]
    L.dflash_debug_gemm.restype = C.c_int


@pytest.mark.parametrize("m,n,k,cap", [
    (16, 256, 128, 0), (4, 512, 256, 0), (15, 1000, 2048, 0), (16, 5120, 2048, 0),
    (16, 2048, 4096, 0), (16, 384, 1024, 7), (33, 640, 512, 5), (64, 256, 192, 3),
    (100, 300, 320, 0), (128, 1024, 512, 11), (200, 512, 1024, 0), (256, 256, 256, 2),
    (300, 384, 512, 0), (512, 2048, 2048, 0), (1000, 640, 256, 9),
])
def test_gemm_matches_fp32_matmul(m, n, k, cap):
    g = torch.Generator(device="cuda").manual_seed(m * 7919 + n * 31 + k)
    w = (torch.randn(n, k, device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    x = torch.randn(m, k, device="cuda", generator=g).to(torch.bfloat16)
    y = torch.full((m, n), float("nan"), device="cuda")
    rc = B.lib().dflash_debug_gemm(w.data_ptr(), x.data_ptr(), y.data_ptr(), m, n, k, cap,
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == 0, B.lib().dflash_last_error().decode()
    ref = x.float() @ w.float().T
    err = (y - ref).abs().max().item()
    assert err <= 1e-3 * max(1.0, ref.abs().max().item()), err
