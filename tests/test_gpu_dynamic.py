"""Dynamic batching (rows leave and join between decode steps) against the
oracle: each row of the cache is its own oracle sequence.

Four rows are prefilled and decoded; rows 1 and 3 retire and decode steps
give -1 for them while rows 0 and 2 continue; two new prompts of another
length are admitted into rows 3 and 1 (in that order) and all four rows then
decode together.  Every active row's logits stay within 2e-2 of its oracle
sequence (teacher-forced with the oracle's tokens), on the tensor-core decode
path, the weight-streaming path and without CUDA graphs (one captured graph
serves every step: it reads the rows' state on the device).
"""
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


@pytest.mark.parametrize("flags", [0, bg.FLAG_NO_TC_GEMM, bg.FLAG_NO_GRAPH],
                         ids=["tcgen05", "streaming", "no_graph"])
def test_rows_leave_and_join(flags):
    shape = synth.PRESETS["560m"].with_(n_layer=2, vocab=3000, batch=4, prompt=12, ragged=True)
    w = synth.make_weights(shape, seed=71, random_affine=True)
    ids, mask = synth.make_prompts(shape, seed=71)
    B, T = ids.shape
    new_ids, new_mask = synth.make_prompts(shape.with_(batch=2, prompt=9), seed=72)
    T2 = new_ids.shape[1]
    S = T + 12
    gm = bg.Model(w.to(DEV), max_batch=B, max_tokens=B * T, max_seq=S, flags=flags)
    kv = gm.new_kv(B, S)
    om = oracle.Model(w)
    seqs = [om.new_seqs(1, S) for _ in range(B)]
    lg = torch.empty(B, shape.vocab, dtype=torch.float32, device=DEV)
    tok = gm.prefill(kv, ids.to(DEV), mask.to(DEV), logits=lg)
    ref = np.concatenate([om.prefill(seqs[b], ids[b:b + 1].numpy(), mask[b:b + 1].numpy())
                          for b in range(B)])
    assert max_abs(lg, ref) <= 2e-2
    active = [True] * B
    nxt_d = torch.empty(B, dtype=torch.int32, device=DEV)

    def step():
        nonlocal ref
        nxt = np.array([int(ref[b].argmax()) if active[b] else 0 for b in range(B)], np.int32)
        nxt_d.copy_(torch.from_numpy(nxt))
        out = gm.decode_step(kv, nxt_d, logits=lg).cpu().numpy()
        new_ref = ref.copy()
        for b in range(B):
            if active[b]:
                new_ref[b] = om.decode(seqs[b], nxt[b:b + 1])[0]
        ref = new_ref
        rows = [b for b in range(B) if active[b]]
        assert max_abs(lg[rows], ref[rows]) <= 2e-2
        greedy_agree(out[rows], ref[rows])
        for b in range(B):
            if not active[b]:
                assert out[b] == -1
        for b in range(B):
            assert kv.row_active(b) == active[b]

    for _ in range(3):
        step()
    lens_before = [kv.row_len(b) for b in range(B)]
    gm.kv_retire(kv, [1, 3])
    active[1] = active[3] = False
    for _ in range(2):
        step()
    assert [kv.row_len(b) for b in range(B)] == [lens_before[0] + 2, lens_before[1],
                                                 lens_before[2] + 2, lens_before[3]]
    # two new prompts into rows 3 and 1
    lg2 = torch.empty(2, shape.vocab, dtype=torch.float32, device=DEV)
    tok2 = gm.kv_admit(kv, [3, 1], new_ids.to(DEV), new_mask.to(DEV), logits=lg2)
    for i, row in enumerate([3, 1]):
        seqs[row] = om.new_seqs(1, S)
        r = om.prefill(seqs[row], new_ids[i:i + 1].numpy(), new_mask[i:i + 1].numpy())[0]
        assert max_abs(lg2[i], r) <= 2e-2
        greedy_agree(tok2[i:i + 1].cpu().numpy(), r[None, :])
        ref[row] = r
        active[row] = True
        assert kv.row_len(row) == T2
    for _ in range(3):
        step()
    gm.check_device()
    gm.close()
