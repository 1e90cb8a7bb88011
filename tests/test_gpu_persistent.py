"""The persistent decode step (one cooperative launch per token step, batches
of 1..16 sequences) against the oracle, against the per-launch step, and
against itself (run-to-run bitwise)."""
import gc

import numpy as np
import pytest
import torch

import bloom_decoder_token_gb300 as bg
from bloom_decoder_token_gb300 import synth
from parity import max_abs
from test_gpu_model import generate_parity

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,over,seed,affine,tol", [
    ("block", dict(batch=1), 0, True, 2e-2),                         # one sequence
    ("block", dict(batch=16, ragged=True), 1, False, 2e-2),          # largest persistent batch
    ("block", dict(batch=3, int8=True, ragged=True), 2, True, 6e-2), # int8 block, bf16 head
    ("560m", dict(n_layer=3, vocab=7000, batch=5), 3, True, 2e-2),   # ragged 560m width
    ("block", dict(hidden=512, n_head=4, ffn=2048, vocab=333, batch=2), 4, True, 2e-2),  # d = 128
])
def test_persistent_matches_oracle(name, over, seed, affine, tol):
    shape = synth.PRESETS[name].with_(**over)
    w = synth.make_weights(shape, seed=seed, random_affine=affine)
    generate_parity(shape, w, steps=5, tol=tol, flags=bg.FLAG_PERSISTENT)


def run_steps(w, shape, flags, steps=6):
    ids, mask = synth.make_prompts(shape, seed=7)
    B, T = ids.shape
    S = T + steps + 1
    gm = bg.Model(w, max_batch=B, max_tokens=B * T, max_seq=S, flags=flags)
    kv = gm.new_kv(B, S)
    lg = torch.empty(B, shape.vocab, dtype=torch.float32, device=DEV)
    tok = gm.prefill(kv, ids.to(DEV), mask.to(DEV))
    toks, logits = [tok.clone()], []
    for _ in range(steps):
        tok = gm.decode_step(kv, tok, tok, logits=lg)
        toks.append(tok.clone())
        logits.append(lg.clone())
    gm.check_device()
    gm.close()
    return torch.stack(toks).cpu(), torch.stack(logits).cpu()


def test_persistent_is_deterministic_and_matches_per_launch_step():
    shape = synth.PRESETS["560m"].with_(n_layer=3, vocab=5000, batch=8)
    w = synth.make_weights(shape, seed=8, random_affine=True).to(DEV)
    t1, l1 = run_steps(w, shape, bg.FLAG_PERSISTENT)
    t2, l2 = run_steps(w, shape, bg.FLAG_PERSISTENT)
    assert torch.equal(t1, t2) and torch.equal(l1, l2)
    t3, l3 = run_steps(w, shape, 0)
    # same arithmetic up to the LayerNorm statistics' summation order
    assert torch.equal(t1[0], t3[0])   # the prefill is the same kernels
    assert max_abs(l1[0], l3[0].double().numpy()) <= 2e-2


def test_launch_accounting_and_fallback_above_16():
    shape = synth.PRESETS["block"].with_(vocab=700, batch=17, ragged=True)
    w = synth.make_weights(shape, seed=9, random_affine=True)
    gm = bg.Model(w.to(DEV), max_batch=17, max_tokens=17 * shape.prompt, max_seq=shape.max_seq,
                  flags=bg.FLAG_PERSISTENT)
    assert gm.decode_launches(8) == 1
    assert gm.decode_launches(17) > 1
    gm.close()
    gmp = bg.Model(w.to(DEV), max_batch=17, max_tokens=17 * shape.prompt, max_seq=shape.max_seq)
    assert gmp.decode_launches(8) > 1
    gmp.close()
    # 17 sequences: the per-launch step even when the persistent one is asked for
    generate_parity(shape, w, steps=3, tol=2e-2, flags=bg.FLAG_PERSISTENT)
