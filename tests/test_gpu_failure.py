"""Failure paths on the GPU, made without faulting it.

* Bounded waits: a model whose tensor-core kernels may wait at most 1 us for
  any barrier (bloom_config.wait_us) runs decode steps and a prefill; every
  launch gives up instead of hanging, the device flag carries 8 (a bounded
  wait expired) through bloom_check_device, and the device stays usable: a
  model with the default bound then decodes against the oracle.
* Host-side injection: BLOOM_INJECT_FAILURE=workspace makes bloom_create's
  workspace allocation fail with BLOOM_E_OOM, and the next create succeeds.
* Poisoned workspace: BLOOM_POISON_WORKSPACE fills the workspace with NaN bytes
  instead of zeros; generations are bit-identical.
"""
import pytest
import torch

import bloom_decoder_token_gb300 as bg
from bloom_decoder_token_gb300 import synth
from test_gpu_model import generate_parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _expect_timeout_flag(gm):
    with pytest.raises(bg.BloomError) as ei:
        gm.check_device()
    assert ei.value.status == 6
    flag = int(str(ei.value).split("device flag 0x")[1].split()[0], 16)
    assert flag & 8, str(ei.value)
    gm.check_device()   # read and cleared


def test_expired_waits_are_reported_and_the_device_stays_usable():
    shape = synth.PRESETS["560m"].with_(n_layer=2, vocab=4000, batch=8, prompt=8, ragged=True)
    w = synth.make_weights(shape, seed=61, random_affine=True)
    wd = w.to(DEV)
    ids, mask = synth.make_prompts(shape, seed=61)
    B, T = ids.shape
    S = T + 6
    gm = bg.Model(wd, max_batch=B, max_tokens=B * T, max_seq=S, wait_us=1)
    kv = gm.new_kv(B, S)
    # 8 x <= 32 tokens: weight-streaming block linears, the LM head (8 rows) on the
    # tensor-core decode kernel, whose waits may run out too
    tok = gm.prefill(kv, ids.to(DEV), mask.to(DEV))
    torch.cuda.synchronize()
    try:
        gm.check_device()
    except bg.BloomError as e:
        assert e.status == 6 and "device flag 0x8 " in str(e), str(e)
    for _ in range(4):                                # tensor-core decode kernels, 1 us bound
        gm.decode_step(kv, tok, tok)
    torch.cuda.synchronize()
    _expect_timeout_flag(gm)
    gm.close()
    # the prefill GEMM (>= 128 tokens) with the same bound: at 7b1 width every
    # output tile's main loop (64 k-blocks) outlasts the epilogue's 3 us bound
    shape2 = synth.PRESETS["7b1"].with_(n_layer=1, batch=4, prompt=64, vocab=2000)
    w2 = synth.make_weights(shape2, seed=62).to(DEV)
    ids2, mask2 = synth.make_prompts(shape2, seed=62)
    gm2 = bg.Model(w2, max_batch=4, max_tokens=4 * 64, max_seq=65, wait_us=1)
    kv2 = gm2.new_kv(4, 65)
    gm2.prefill(kv2, ids2.to(DEV), mask2.to(DEV))
    torch.cuda.synchronize()
    _expect_timeout_flag(gm2)
    gm2.close()
    # the same device, the default bound: correct against the oracle
    generate_parity(shape, w, steps=3, tol=2e-2)


def test_poisoned_workspace_changes_nothing(monkeypatch):
    """BLOOM_POISON_WORKSPACE: the workspace starts as 0xff bytes (NaN in bf16
    and float32) instead of zeros.  A prefill and decode steps -- streaming and
    tensor-core linears, split-K partials, attention partials, LayerNorms, the
    head's argmax -- give bit-identical logits and tokens, so no kernel reads an
    activation or a partial before writing it."""
    shape = synth.PRESETS["560m"].with_(n_layer=2, vocab=3000, batch=6, prompt=8, ragged=True)
    w = synth.make_weights(shape, seed=64, random_affine=True).to(DEV)
    ids, mask = synth.make_prompts(shape, seed=64)
    B, T = ids.shape
    S = T + 5
    outs = []
    for poison in (False, True):
        if poison:
            monkeypatch.setenv("BLOOM_POISON_WORKSPACE", "1")
        gm = bg.Model(w, max_batch=B, max_tokens=B * T, max_seq=S)
        monkeypatch.delenv("BLOOM_POISON_WORKSPACE", raising=False)
        kv = gm.new_kv(B, S)
        lg = torch.empty(B, shape.vocab, dtype=torch.float32, device=DEV)
        tok = gm.prefill(kv, ids.to(DEV), mask.to(DEV), logits=lg)
        run = [(tok.clone(), lg.clone())]
        for _ in range(4):
            tok = gm.decode_step(kv, tok, logits=lg)
            run.append((tok.clone(), lg.clone()))
        torch.cuda.synchronize()
        gm.check_device()
        gm.close()
        outs.append(run)
    for (t0, l0), (t1, l1) in zip(*outs):
        assert torch.isfinite(l1).all()
        assert torch.equal(t0, t1)
        assert torch.equal(l0, l1)


def test_injected_workspace_allocation_failure(monkeypatch):
    shape = synth.PRESETS["block"].with_(vocab=512)
    w = synth.make_weights(shape, seed=63).to(DEV)
    monkeypatch.setenv("BLOOM_INJECT_FAILURE", "workspace")
    with pytest.raises(bg.BloomError) as ei:
        bg.Model(w, max_batch=1, max_tokens=8, max_seq=9)
    assert ei.value.status == 3
    assert "workspace" in str(ei.value)
    monkeypatch.delenv("BLOOM_INJECT_FAILURE")
    gm = bg.Model(w, max_batch=1, max_tokens=8, max_seq=9)
    gm.close()
