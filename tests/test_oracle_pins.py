"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself: each check is a closed form, a
library routine (torch / numpy), an invariant of the method, or an independent
dense restatement on tiny shapes.  CPU only.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as orc
from bloom_decoder_token_gb300 import synth
import restatement


# ---------------------------------------------------------------- ALiBi slopes
@pytest.mark.parametrize("n,expo", [(8, lambda i: -i), (16, lambda i: -i / 2),
                                    (32, lambda i: -i / 4), (64, lambda i: -i / 8)])
def test_slopes_power_of_two_closed_form(n, expo):
    s = orc.alibi_slopes(n)
    ref = np.array([2.0 ** expo(i) for i in range(1, n + 1)])
    np.testing.assert_allclose(s, ref, rtol=1e-15, atol=0)


def test_slopes_112_heads_interleave():
    # 112 heads: largest power of two 64; heads 1..64 get 2^(-i/8),
    # heads 65..112 get 2^(-(2j-1)/16), j = 1..48
    s = orc.alibi_slopes(112)
    ref = [2.0 ** (-i / 8) for i in range(1, 65)] + [2.0 ** (-(2 * j - 1) / 16)
                                                     for j in range(1, 49)]
    np.testing.assert_allclose(s, np.array(ref), rtol=1e-15, atol=0)
    # every extra slope lies strictly between two consecutive base slopes
    base = s[:64]
    for e in s[64:]:
        assert np.any((base[:-1] > e) & (e > base[1:])) or e > base[0]


@pytest.mark.parametrize("n", [1, 2, 3, 5, 6, 12, 16, 20, 24, 40, 96, 112, 120])
def test_slopes_match_geometric_construction(n):
    np.testing.assert_allclose(orc.alibi_slopes(n), restatement.slopes_geometric(n).numpy(),
                               rtol=1e-14, atol=0)


# ---------------------------------------------------------------- GeLU
def test_gelu_special_values():
    assert orc.gelu(0.0) == 0.0
    for x in [0.1, 0.5, 1.0, 2.5, 7.0]:
        # the tanh form is x * sigma-like(x): g(x) - g(-x) = x exactly in reals
        assert abs(orc.gelu(x) - orc.gelu(-x) - x) < 1e-15 * max(1.0, x)
    assert abs(orc.gelu(30.0) - 30.0) < 1e-12
    assert abs(orc.gelu(-30.0)) < 1e-12


def test_gelu_matches_library_tanh_form():
    xs = torch.linspace(-8, 8, 1601, dtype=torch.float64)
    ref = F.gelu(xs, approximate="tanh")   # constant sqrt(2/pi) = 0.7978845608...
    got = torch.tensor([orc.gelu(float(x)) for x in xs], dtype=torch.float64)
    # 0.79788456 vs sqrt(2/pi) differ by 8e-11 relative
    assert float((got - ref).abs().max()) < 1e-9


# ---------------------------------------------------------------- LayerNorm
def test_layernorm_matches_library():
    g = torch.Generator().manual_seed(3)
    for h in [1, 7, 64, 1024]:
        x = torch.randn(5, h, generator=g, dtype=torch.float64) * 3 + 1.5
        gam = (1 + 0.1 * torch.randn(h, generator=g)).to(torch.bfloat16)
        bet = (0.1 * torch.randn(h, generator=g)).to(torch.bfloat16)
        got = orc.layernorm(x.numpy(), orc.host_bits(gam), orc.host_bits(bet), 1e-5)
        ref = F.layer_norm(x, (h,), gam.double(), bet.double(), 1e-5)
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_layernorm_invariants():
    x = np.random.default_rng(0).normal(2.0, 5.0, size=(3, 4096))
    y = orc.layernorm(x)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose(y.var(axis=1), 1.0 - 1e-5 / (x.var(axis=1) + 1e-5), rtol=1e-9)
    # a constant row normalises to 0, so the output is beta
    beta = orc.bf16_bits(np.linspace(-1, 1, 16))
    c = orc.layernorm(np.full((1, 16), 3.25), None, beta)
    np.testing.assert_array_equal(c[0], [orc.lib().orc_bf16_to_double(int(b)) for b in beta])


# ---------------------------------------------------------------- linear
def test_linear_bf16_matches_matmul():
    g = torch.Generator().manual_seed(4)
    W = (0.02 * torch.randn(37, 53, generator=g)).to(torch.bfloat16)
    b = (0.02 * torch.randn(37, generator=g)).to(torch.bfloat16)
    x = torch.randn(6, 53, generator=g, dtype=torch.float64)
    got = orc.linear(x.numpy(), orc.host_bits(W), orc.host_bits(b))
    ref = x.numpy() @ W.double().numpy().T + b.double().numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


def test_linear_int8_dequant_identity():
    g = torch.Generator().manual_seed(5)
    W = (0.02 * torch.randn(29, 64, generator=g)).to(torch.bfloat16)
    W[3] = 0  # a zero row gets s = 0, q = 0
    q, s = synth.quantize_rows_int8(W)
    assert q.dtype == torch.int8 and int(q.abs().max()) <= 127 and int(q[3].abs().max()) == 0
    assert float(s[3]) == 0.0
    # s = bf16(absmax / 127); every w is reproduced by q*s within one step s
    np.testing.assert_array_equal(orc.host_bits(s),
                                  orc.host_bits((W.float().abs().amax(1) / 127).to(torch.bfloat16)))
    err = (q.double() * s.double()[:, None] - W.double()).abs()
    assert bool((err <= s.double()[:, None] * 0.5 * (1 + 2 ** -7) + 1e-30).all())
    x = torch.randn(3, 64, generator=g, dtype=torch.float64)
    got = orc.linear(x.numpy(), q=orc.host_bits(q), s_bits=orc.host_bits(s))
    ref = x.numpy() @ (q.double() * s.double()[:, None]).numpy().T
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- attention
def test_attention_softmax_rows_and_mask():
    rng = np.random.default_rng(6)
    d, nk = 16, 23
    q, K, V = rng.normal(size=d), rng.normal(size=(nk, d)), rng.normal(size=(nk, d))
    pos = np.arange(nk, dtype=np.int32) - 5
    pos[pos < 0] = -1            # five left pads
    pos[11] = -1                 # and one hole
    o, p = orc.attend(q, K, V, pos, 0.25)
    assert abs(p.sum() - 1.0) < 1e-12
    assert np.all(p[pos < 0] == 0.0)
    assert np.all(p[pos >= 0] > 0.0)


def test_attention_special_cases():
    rng = np.random.default_rng(7)
    d = 8
    v = rng.normal(size=(1, d))
    o, p = orc.attend(rng.normal(size=d), rng.normal(size=(1, d)), v, np.array([0], np.int32), 0.5)
    np.testing.assert_allclose(o, v[0], rtol=1e-15)       # one key: o = v
    # equal keys, slope 0: uniform weights, o = mean of the values
    K = np.tile(rng.normal(size=(1, d)), (9, 1))
    V = rng.normal(size=(9, d))
    o, p = orc.attend(rng.normal(size=d), K, V, np.arange(9, dtype=np.int32), 0.0)
    np.testing.assert_allclose(o, V.mean(axis=0), rtol=1e-12, atol=1e-14)
    # q = 0: p_k proportional to exp(slope * pos_k)
    pos = np.array([-1, -1, 0, 1, 2, 3], np.int32)
    o, p = orc.attend(np.zeros(d), rng.normal(size=(6, d)), rng.normal(size=(6, d)), pos, 0.375)
    w = np.exp(0.375 * np.arange(4))
    np.testing.assert_allclose(p[2:], w / w.sum(), rtol=1e-14)
    # every key masked: output 0
    o, p = orc.attend(rng.normal(size=d), rng.normal(size=(3, d)), rng.normal(size=(3, d)),
                      np.array([-1, -1, -1], np.int32), 0.5)
    assert np.all(o == 0.0) and np.all(p == 0.0)


def test_attention_matches_library_sdpa():
    rng = np.random.default_rng(8)
    d, nk = 32, 40
    q, K, V = rng.normal(size=d), rng.normal(size=(nk, d)), rng.normal(size=(nk, d))
    pos = np.arange(nk, dtype=np.int32) - 3
    pos[pos < 0] = -1
    slope = 2.0 ** -1.5
    o, _ = orc.attend(q, K, V, pos, slope)
    m = torch.where(torch.tensor(pos) >= 0, slope * torch.tensor(pos, dtype=torch.float64),
                    torch.tensor(-math.inf, dtype=torch.float64))
    ref = F.scaled_dot_product_attention(torch.tensor(q)[None, None], torch.tensor(K)[None],
                                         torch.tensor(V)[None], attn_mask=m[None, None])
    np.testing.assert_allclose(o, ref[0, 0].numpy(), rtol=1e-12, atol=1e-14)


def test_argmax_lowest_index_on_ties():
    assert orc.argmax(np.array([0.0, 3.0, 1.0, 3.0])) == 1
    assert orc.argmax(np.array([-5.0])) == 0


# ---------------------------------------------------------------- whole model
TINY = synth.Shape("tiny", 2, 8, 2, 32, 16, 3, 6, 4)
TINY3 = synth.Shape("tiny3", 2, 12, 3, 48, 20, 2, 5, 3)     # 3 heads: non-power-of-two ALiBi
TINY8 = TINY.with_(name="tiny8", int8=True)


@pytest.mark.parametrize("shape", [TINY, TINY3, TINY8], ids=lambda s: s.name)
def test_forward_full_matches_restatement(shape):
    w = synth.make_weights(shape, seed=11, random_affine=True)
    om = orc.Model(w)
    gen = torch.Generator().manual_seed(12)
    T = 7
    toks = torch.randint(0, shape.vocab, (T,), generator=gen)
    for mask in [torch.ones(T, dtype=torch.uint8), torch.tensor([0, 0, 1, 1, 1, 1, 1],
                                                                dtype=torch.uint8),
                 torch.tensor([1, 0, 1, 1, 0, 1, 1], dtype=torch.uint8)]:
        got = om.forward_full(toks.numpy(), mask.numpy())
        ref = restatement.forward(w, toks, mask).numpy()
        np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-9)


@pytest.mark.parametrize("shape", [TINY, TINY3, TINY8], ids=lambda s: s.name)
def test_kv_cached_decode_equals_recompute(shape):
    """Prefill then decode with the cache equals a full recompute of the prefix
    at every step (the KV cache only saves work)."""
    w = synth.make_weights(shape, seed=13, random_affine=True)
    om = orc.Model(w)
    ids, mask = synth.make_prompts(shape.with_(ragged=True, prompt=6), seed=14)
    B, T = ids.shape
    steps = 4
    seqs = om.new_seqs(B, T + steps)
    logits = om.prefill(seqs, ids.numpy(), mask.numpy())
    extra = synth.make_tokens(shape, steps, seed=15, batch=B).numpy()
    hist_ids, hist_mask = ids.numpy().copy(), mask.numpy().copy()
    for b in range(B):
        full = om.forward_full(hist_ids[b], hist_mask[b])
        np.testing.assert_allclose(logits[b], full[-1], rtol=1e-11, atol=1e-11)
    for s in range(steps):
        logits = om.decode(seqs, extra[s])
        hist_ids = np.concatenate([hist_ids, extra[s][:, None]], axis=1)
        hist_mask = np.concatenate([hist_mask, np.ones((B, 1), np.uint8)], axis=1)
        for b in range(B):
            full = om.forward_full(hist_ids[b], hist_mask[b])
            np.testing.assert_allclose(logits[b], full[-1], rtol=1e-11, atol=1e-11)


def test_left_padding_is_invisible():
    """ALiBi positions count from the first token, so left pads change nothing."""
    w = synth.make_weights(TINY3, seed=16, random_affine=True)
    om = orc.Model(w)
    toks = np.array([3, 9, 1, 4, 17], np.int32)
    a = om.forward_full(toks, np.ones(5, np.uint8))[-1]
    b = om.forward_full(np.concatenate([[0, 0, 0], toks]).astype(np.int32),
                        np.array([0, 0, 0, 1, 1, 1, 1, 1], np.uint8))[-1]
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_prefill_taps_and_decode_taps_consistent():
    w = synth.make_weights(TINY, seed=17, random_affine=True)
    om = orc.Model(w)
    ids, mask = synth.make_prompts(TINY, seed=18)
    seqs = om.new_seqs(ids.shape[0], ids.shape[1] + 1)
    logits, taps = om.prefill(seqs, ids.numpy(), mask.numpy(), taps=True)
    # last tap, last slot, through the head = returned logits
    np.testing.assert_allclose(om.head(taps[-1][:, -1]), logits, rtol=1e-13, atol=1e-13)
    # a layer applied on its own reproduces the next tap
    x1 = om.layer_prefill(0, taps[0][1], mask[1].numpy())
    np.testing.assert_allclose(x1, taps[1][1], rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- top-p sampling
LN2, LN3 = math.log(2.0), math.log(3.0)


def test_sample_closed_form():
    # logits 0, ln 2, ln 3 -> p = 1/6, 1/3, 1/2
    z = [0.0, LN2, LN3]
    # top_p 0.5: the most probable token alone reaches it
    for u in (0.0, 0.3, 0.999):
        assert orc.sample_top_p(z, 1.0, 0.5, u) == 2
    # top_p 0.51: nucleus {2, 1} of mass 5/6, renormalised 0, 0.4, 0.6 in vocabulary order
    assert orc.sample_top_p(z, 1.0, 0.51, 0.39) == 1
    assert orc.sample_top_p(z, 1.0, 0.51, 0.41) == 2
    # top_p 1: cumulative 1/6, 1/2, 1 in vocabulary order
    assert orc.sample_top_p(z, 1.0, 1.0, 0.1) == 0
    assert orc.sample_top_p(z, 1.0, 1.0, 0.3) == 1
    assert orc.sample_top_p(z, 1.0, 1.0, 0.9) == 2


def test_sample_temperature_scales_logits():
    z = np.array([0.0, LN2, LN3, -1.0])
    for u in np.linspace(0.0, 0.999, 37):
        for tp in (0.4, 0.8, 1.0):
            assert orc.sample_top_p(2.0 * z, 2.0, tp, u) == orc.sample_top_p(z, 1.0, tp, u)


def test_sample_greedy_and_tiny_nucleus():
    assert orc.sample_top_p([1.0, 3.0, 3.0, 2.0], 0.0, 0.9, 0.5) == 1   # greedy, lowest index
    assert orc.sample_top_p([1.0, 3.0, 3.0, 2.0], -1.0, 0.9, 0.5) == 1
    z = np.random.default_rng(3).normal(size=50)
    top = int(np.argmax(z))
    for u in (0.0, 0.5, 0.99):
        assert orc.sample_top_p(z, 0.7, 1e-9, u) == top


def test_sample_ties_enter_the_nucleus_by_index():
    # p = e, e, e, 1 over 3e + 1: the ordering keeps ties in index order, so the
    # two-token nucleus is {0, 1}, renormalised 1/2, 1/2
    z = [1.0, 1.0, 1.0, 0.0]
    assert orc.sample_top_p(z, 1.0, 0.5, 0.49) == 0
    assert orc.sample_top_p(z, 1.0, 0.5, 0.51) == 1
    assert orc.sample_top_p(z, 1.0, 0.5, 0.99) == 1


@pytest.mark.parametrize("seed,top_p,temp", [(0, 0.7, 1.0), (1, 0.3, 0.5), (2, 0.95, 1.7)])
def test_sample_distribution_by_brute_force(seed, top_p, temp):
    """Over a fine grid of u, each token is drawn with its probability
    renormalised over the nucleus, and the nucleus is the smallest set of
    most-probable tokens reaching top_p -- found here by enumerating subsets."""
    rng = np.random.default_rng(seed)
    z = rng.normal(size=6) * 2.0
    p = np.exp(z / temp - np.max(z / temp))
    p /= p.sum()
    best = None
    for mask in range(1, 64):
        idx = [i for i in range(6) if mask >> i & 1]
        mass = p[idx].sum()
        if mass >= top_p and (best is None or len(idx) < len(best[0]) or
                              (len(idx) == len(best[0]) and mass > best[1])):
            best = (idx, mass)
    nucleus, mass = best
    want = np.zeros(6)
    want[nucleus] = p[nucleus] / mass
    n = 20000
    got = np.zeros(6)
    for u in (np.arange(n) + 0.5) / n:
        got[orc.sample_top_p(z, temp, top_p, u)] += 1
    np.testing.assert_allclose(got / n, want, atol=2.0 / n)
