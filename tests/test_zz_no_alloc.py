"""The allocation-free LM head + argmax entry point, called through the C ABI.

For callers that cannot allocate device memory per call (device-synchronising
cudaMalloc/cudaFree, memory owned by another framework's allocator, serving
loops that forbid allocation): its scratch is a fixed array inside the library.
It must give the same tokens and logits as bloom_op_lmhead_argmax, on
consecutive calls (the shared array is cleared by each call), and reject row
counts beyond the array.  This file is collected last on purpose.
"""
import ctypes as C

import pytest
import torch

import bloom_decoder_token_gb300 as bg
from parity import assert_kernel_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _inputs(seed, M, V, K):
    g = torch.Generator(device="cpu").manual_seed(seed)
    E = (0.02 * torch.randn(V, K, generator=g)).to(torch.bfloat16).to(DEV)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16).to(DEV)
    return x, E


def test_noalloc_matches_allocating_entry_on_consecutive_calls():
    L = bg.lib()
    for seed, (M, V, K) in enumerate([(8, 250880, 1024), (3, 50000, 4096), (8, 250880, 1024)]):
        x, E = _inputs(100 + seed, M, V, K)
        tok_ref, lg_ref = bg.op_lmhead_argmax(x, E)
        tok = torch.empty(M, dtype=torch.int32, device=DEV)
        lg = torch.empty(M, V, dtype=torch.float32, device=DEV)
        st = L.bloom_op_lmhead_argmax_noalloc(C.c_void_p(x.data_ptr()), C.c_void_p(E.data_ptr()),
                                              M, V, K, C.c_void_p(tok.data_ptr()),
                                              C.c_void_p(lg.data_ptr()),
                                              C.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, L.bloom_last_error()
        torch.cuda.synchronize()
        assert torch.equal(tok.cpu(), tok_ref.cpu())
        assert_kernel_close(lg, lg_ref.cpu().double().numpy(), rel=1e-6, atol_rms=1e-6,
                            what="noalloc logits")
    # and through the Python wrapper, without logits
    x, E = _inputs(7, 5, 3000, 512)
    tok_ref, _ = bg.op_lmhead_argmax(x, E, logits=False)
    tok, none = bg.op_lmhead_argmax_noalloc(x, E, logits=False)
    assert none is None and torch.equal(tok.cpu(), tok_ref.cpu())


def test_noalloc_rejects_rows_beyond_scratch():
    L = bg.lib()
    x, E = _inputs(9, 1, 64, 64)
    out = torch.empty(300, dtype=torch.int32, device=DEV)
    st = L.bloom_op_lmhead_argmax_noalloc(C.c_void_p(x.data_ptr()), C.c_void_p(E.data_ptr()), 257,
                                          64, 64, C.c_void_p(out.data_ptr()), None, None)
    assert st == 4
    assert "fixed scratch" in L.bloom_last_error().decode()
