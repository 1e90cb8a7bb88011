"""KV offload to host memory (bloom_kv_init_offload): the K and V of layers
[offload_from, n_layer) live in page-locked host memory that the kernels read
and write directly over the host link.

The offloaded cache runs the same kernels on the same numbers as a cache held
entirely in HBM, so prefill and decode give bit-identical logits and tokens,
the host part holds exactly the K / V rows the device cache holds for those
layers, and the whole generation matches the oracle.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import bloom_decoder_token_gb300 as bg
from bloom_decoder_token_gb300 import synth
import oracle
from parity import greedy_agree, max_abs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def run(gm, kv, ids, mask, steps, V):
    B = ids.shape[0]
    lg = torch.empty(B, V, dtype=torch.float32, device=DEV)
    tok = gm.prefill(kv, ids.to(DEV), mask.to(DEV), logits=lg)
    out = [(tok.clone(), lg.clone())]
    for _ in range(steps):
        tok = gm.decode_step(kv, tok, logits=lg)
        out.append((tok.clone(), lg.clone()))
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("offload_from", [0, 1, 2])
def test_offloaded_cache_is_bit_identical(offload_from):
    shape = synth.PRESETS["560m"].with_(n_layer=3, vocab=4000, batch=4, prompt=8, ragged=True)
    w = synth.make_weights(shape, seed=71, random_affine=True).to(DEV)
    ids, mask = synth.make_prompts(shape, seed=71)
    B, T = ids.shape
    S = T + 5
    gm = bg.Model(w, max_batch=B, max_tokens=B * T, max_seq=S)
    kv_d = gm.new_kv(B, S)
    kv_h = gm.new_kv(B, S, offload_from=offload_from)
    assert kv_h.host is not None
    ref = run(gm, kv_d, ids, mask, 4, shape.vocab)
    got = run(gm, kv_h, ids, mask, 4, shape.vocab)
    for (t0, l0), (t1, l1) in zip(ref, got):
        assert torch.equal(t0, t1)
        assert torch.equal(l0, l1)
    td, th = kv_d.tensors(gm), kv_h.tensors(gm)
    n = kv_d.len
    assert torch.equal(td["k"][:offload_from, :, :, :n], th["k"][:, :, :, :n])
    assert torch.equal(td["k"][offload_from:, :, :, :n].cpu(), th["k_host"][:, :, :, :n].cpu())
    assert torch.equal(td["v"][offload_from:, :, :, :n].cpu(), th["v_host"][:, :, :, :n].cpu())
    gm.check_device()
    gm.close()


def test_offloaded_cache_is_bit_identical_where_device_layers_stage_kv_by_bulk_copies():
    # 7b1 heads (32 x 128) at 48 sequences: 1536 attention CTAs, beyond the 64-thread
    # CTAs resident at once, so the device-resident layer stages its K / V by bulk
    # copies while the host-resident one reads them directly -- the same bits
    shape = synth.PRESETS["7b1"].with_(n_layer=2, vocab=1000, batch=48, prompt=20, ragged=True)
    w = synth.make_weights(shape, seed=74, random_affine=True).to(DEV)
    ids, mask = synth.make_prompts(shape, seed=74)
    B, T = ids.shape
    S = T + 4
    gm = bg.Model(w, max_batch=B, max_tokens=B * T, max_seq=S)
    kv_d = gm.new_kv(B, S)
    kv_h = gm.new_kv(B, S, offload_from=1)
    ref = run(gm, kv_d, ids, mask, 3, shape.vocab)
    got = run(gm, kv_h, ids, mask, 3, shape.vocab)
    for (t0, l0), (t1, l1) in zip(ref, got):
        assert torch.equal(t0, t1)
        assert torch.equal(l0, l1)
    gm.check_device()
    gm.close()


def test_offloaded_generation_against_oracle():
    shape = synth.PRESETS["560m"].with_(n_layer=2, vocab=3000, batch=3, prompt=8, ragged=True)
    w = synth.make_weights(shape, seed=72, random_affine=True)
    ids, mask = synth.make_prompts(shape, seed=72)
    B, T = ids.shape
    S = T + 4
    gm = bg.Model(w.to(DEV), max_batch=B, max_tokens=B * T, max_seq=S)
    kv = gm.new_kv(B, S, offload_from=1)
    om = oracle.Model(w)
    seqs = om.new_seqs(B, S)
    lg = torch.empty(B, shape.vocab, dtype=torch.float32, device=DEV)
    tok = gm.prefill(kv, ids.to(DEV), mask.to(DEV), logits=lg)
    ref = om.prefill(seqs, ids.numpy(), mask.numpy())
    assert max_abs(lg, ref) <= 2e-2
    greedy_agree(tok.cpu().numpy(), ref, 0.1)
    nxt_d = torch.empty(B, dtype=torch.int32, device=DEV)
    for _ in range(3):
        nxt = torch.from_numpy(ref.argmax(axis=1).astype(np.int32))
        nxt_d.copy_(nxt)
        tok = gm.decode_step(kv, nxt_d, logits=lg)
        ref = om.decode(seqs, nxt.numpy())
        assert max_abs(lg, ref) <= 2e-2
        greedy_agree(tok.cpu().numpy(), ref, 0.1)
    gm.check_device()
    gm.close()


def test_offload_rejects_memory_the_device_cannot_address():
    shape = synth.PRESETS["block"].with_(vocab=512)
    w = synth.make_weights(shape, seed=73).to(DEV)
    gm = bg.Model(w, max_batch=2, max_tokens=16, max_seq=9)
    dn, hn = C.c_size_t(), C.c_size_t()
    bg.check(bg.lib().bloom_kv_bytes_offload(C.byref(gm.cfg), 2, 9, 0, C.byref(dn), C.byref(hn)))
    dev = torch.empty(dn.value + 256, dtype=torch.uint8, device=DEV)
    dptr = dev.data_ptr() + (-dev.data_ptr()) % 256
    kvc = bg.KVC()
    # device memory, and pageable host memory, in place of page-locked host memory
    other = torch.empty(hn.value + 256, dtype=torch.uint8, device=DEV)
    pageable = np.zeros(hn.value + 512, dtype=np.uint8)
    for hptr in (other.data_ptr() + (-other.data_ptr()) % 256,
                 pageable.ctypes.data + (-pageable.ctypes.data) % 256):
        st = bg.lib().bloom_kv_init_offload(gm.h, C.byref(kvc), C.c_void_p(dptr), dn.value,
                                            C.c_void_p(hptr), hn.value, 2, 9, 0, None)
        assert st == 1, bg.lib().bloom_last_error()
    # too small a host buffer
    pinned = torch.empty(hn.value + 256, dtype=torch.uint8, pin_memory=True)
    hptr = pinned.data_ptr() + (-pinned.data_ptr()) % 256
    st = bg.lib().bloom_kv_init_offload(gm.h, C.byref(kvc), C.c_void_p(dptr), dn.value,
                                        C.c_void_p(hptr), hn.value - 256, 2, 9, 0, None)
    assert st == 1
    gm.close()
