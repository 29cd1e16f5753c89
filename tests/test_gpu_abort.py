"""The bounded-wait abort path on the GPU, made to run out without any fault.

Every mbarrier wait in the library's tcgen05 kernels gives up after a time
limit: the CTA raises the device status word, stops issuing work, waits
(bounded) for its own copies and MMAs, frees its TMEM and exits, and the call
returns DFLASH_EDEVICE. The test hook dflash_debug_set_fault makes one thread
of every CTA of every tensor-core GEMM wait 1 ms on a barrier that nothing
arrives on, so the limit runs out mid-stream (weight copies and MMAs in flight)
on every GEMM of the forward. The call must report DFLASH_EDEVICE, leave the
state and the pool as they were, and the same handle must then run the same
propose normally and match the oracle; the allocation-free GEMM entry point
must still work after it."""
import ctypes as C

import pytest
import torch

from block_diffusion_speculative_forward_gb300 import binding as B
from block_diffusion_speculative_forward_gb300 import synthetic as syn
from tests.parity import Pair, assert_tables, check_seq

pytestmark = pytest.mark.gpu

D128 = syn.Geometry(num_layers=2, hidden=256, intermediate=256, num_q_heads=8,
                    num_kv_heads=1, head_dim=128, vocab=1024, gamma=16, mask_token_id=1023,
                    n_target_layers=2, target_hidden=128, rope_theta=1e4, ctx_window=200,
                    kv_block=16, prefill_chunk=64)


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_diffusion_speculative_forward_gb300 import build
    build.build()


@pytest.mark.parametrize("geom,seed,n_ctx,nd", [(syn.TINY, 1201, 40, 3), (D128, 1202, 150, 15)])
def test_timeout_returns_edevice_and_handle_recovers(geom, seed, n_ctx, nd):
    pair = Pair(geom, seed)
    so, sl = pair.ora.alloc_state(), pair.lib.alloc_state()
    stack = syn.make_stack(geom, n_ctx + 2, seed)
    pair.ora.prefill(so, stack[:n_ctx])
    pair.lib.prefill(sl, stack[:n_ctx].cuda())
    before = pair.lib.debug_state(sl), pair.lib.debug_pool()
    row = stack[n_ctx:n_ctx + 1]
    pair.lib.set_fault(1_000_000)
    with pytest.raises(B.DFlashError) as e:
        pair.lib.propose(sl, 7, n_ctx + 1, row.cuda(), nd)
    assert e.value.code == "EDEVICE", str(e.value)
    assert "bounded wait" in str(e.value)
    assert (pair.lib.debug_state(sl), pair.lib.debug_pool()) == before
    # the same propose again, normally: the handle and the state are intact
    pair.lib.set_fault(0)
    taps = {}
    ref = pair.ora.propose(so, 7, n_ctx + 1, row, nd, taps=taps)
    got = pair.lib.propose(sl, 7, n_ctx + 1, row.cuda(), nd)
    check_seq(pair, taps["seq"][0], ref, got, 0, 1, nd)
    assert_tables(pair, so, sl)
    # and the allocation-free GEMM afterwards
    L = B.lib()
    L.dflash_gemm_noalloc.restype = C.c_int
    L.dflash_gemm_noalloc.argtypes = [C.c_void_p] * 3 + [C.c_int32] * 3 + [C.c_void_p]
    g = torch.Generator(device="cuda").manual_seed(seed)
    w = (torch.randn(384, 256, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    x = torch.randn(16, 256, device="cuda", generator=g).to(torch.bfloat16)
    y = torch.empty(16, 384, device="cuda")
    rc = L.dflash_gemm_noalloc(w.data_ptr(), x.data_ptr(), y.data_ptr(), 16, 384, 256,
                               torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    ref_y = x.float() @ w.float().T
    assert (y - ref_y).abs().max().item() <= 1e-3 * max(1.0, ref_y.abs().max().item())
