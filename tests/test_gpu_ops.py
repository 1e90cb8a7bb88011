"""Kernel-level parity: each CUDA operator vs the CPU oracle on identical bf16
inputs, including ragged tails, odd sizes and the degenerate cases."""
import numpy as np
import pytest
import torch

import bloom_decoder_token_gb300 as bg
import oracle
from parity import assert_kernel_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def gen(seed):
    return torch.Generator(device="cpu").manual_seed(seed)


def bf(shape, g, std=1.0, mean=0.0):
    return (mean + std * torch.randn(*shape, generator=g)).to(torch.bfloat16)


# ---------------------------------------------------------------- LayerNorm
@pytest.mark.parametrize("rows,h", [(1, 64), (3, 1024), (17, 4096), (2, 14336), (5, 16384),
                                    (4, 200)])
def test_layernorm(rows, h):
    g = gen(rows * 7 + h)
    x = bf((rows, h), g, 3.0, 1.0)
    gam = bf((h,), g, 0.1, 1.0)
    bet = bf((h,), g, 0.1)
    y = bg.op_layernorm(x.to(DEV), gam.to(DEV), bet.to(DEV), eps=1e-5)
    ref = oracle.layernorm(f64(x), oracle.host_bits(gam), oracle.host_bits(bet), 1e-5)
    assert_kernel_close(y, ref, what="layernorm")


def test_layernorm_constant_row_gives_beta():
    h = 1024
    x = torch.full((2, h), 7.5, dtype=torch.bfloat16)
    bet = bf((h,), gen(1), 0.5)
    y = bg.op_layernorm(x.to(DEV), None, bet.to(DEV))
    assert torch.equal(y.cpu(), torch.stack([bet, bet]))


# ---------------------------------------------------------------- linear
# The last four take the A-operand form (16-row tasks, at least a wave of them
# on 152 SMs) with 1, 2 and 4 token tiles, ragged rows and a ragged K tail.
SHAPES = [(1, 3072, 1024), (3, 100, 64), (8, 4096, 4096), (5, 13, 16384), (16, 1000, 1024),
          (33, 50, 512), (2, 4097, 256), (8, 257, 14336), (64, 600, 1040), (1, 40, 57344),
          (24, 1, 4096), (1, 12288, 4096), (3, 16000, 208), (13, 8200, 512), (24, 12300, 256)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
@pytest.mark.parametrize("epi", [bg.EPI_STORE, bg.EPI_GELU, bg.EPI_RESID],
                         ids=["store", "gelu", "resid"])
def test_linear(M, N, K, int8, epi):
    if int8 and K % 16:
        pytest.skip("int8 rows are 16-byte chunks")
    g = gen(M * 1000 + N + K + epi)
    W = bf((N, K), g, 0.02)
    x = bf((M, K), g, 1.0)
    bias = bf((N,), g, 0.5)
    y0 = bf((M, N), g, 1.0)
    kw = {}
    if int8:
        from bloom_decoder_token_gb300 import synth
        q, s = synth.quantize_rows_int8(W)
        kw = dict(q=q.to(DEV), scale=s.to(DEV))
        acc = oracle.linear(f64(x), q=oracle.host_bits(q), s_bits=oracle.host_bits(s),
                            bias_bits=oracle.host_bits(bias))
    else:
        kw = dict(w=W.to(DEV))
        acc = oracle.linear(f64(x), oracle.host_bits(W), oracle.host_bits(bias))
    y = y0.to(DEV).clone()
    bg.op_linear(x.to(DEV), bias=bias.to(DEV), epilogue=epi, y=y, **kw)
    if epi == bg.EPI_STORE:
        ref = acc
    elif epi == bg.EPI_GELU:
        ref = np.vectorize(oracle.gelu)(acc)
    else:
        ref = f64(y0) + acc
    assert_kernel_close(y, ref, what=f"linear {M}x{N}x{K}")


@pytest.mark.parametrize("N", [256, 8192], ids=["b_operand", "a_operand"])
def test_linear_int8_every_code(N):
    """Every int8 code, -128 included, at byte positions inside a lane's 16-byte
    fragment, across lanes and across chunks, is widened exactly: with unit
    scales, no bias and one-hot activations y[m][n] = q[n][p_m]."""
    K = 256
    n = torch.arange(N).unsqueeze(1)
    k = torch.arange(K).unsqueeze(0)
    q = ((n + k) % 256).to(torch.uint8).view(torch.int8)
    pos = [0, 1, 2, 3, 13, 31, 70, 255]
    x = torch.zeros(len(pos), K, dtype=torch.bfloat16)
    for m, p in enumerate(pos):
        x[m, p] = 1.0
    scale = torch.ones(N, dtype=torch.bfloat16)
    y = bg.op_linear(x.to(DEV), q=q.to(DEV), scale=scale.to(DEV))
    expect = torch.stack([q[:, p].float() for p in pos])
    assert torch.equal(y.cpu().float(), expect)


def test_linear_zero_bias_and_empty_batch():
    g = gen(5)
    W = bf((64, 128), g, 0.02)
    x = bf((2, 128), g)
    y = bg.op_linear(x.to(DEV), w=W.to(DEV))
    assert_kernel_close(y, oracle.linear(f64(x), oracle.host_bits(W)), what="no bias")
    e = bg.op_linear(torch.empty(0, 128, dtype=torch.bfloat16, device=DEV), w=W.to(DEV))
    assert e.shape == (0, 64)


# ---------------------------------------------------------------- decode attention
def make_cache(B, n, S, d, length, g, pads=0, holes=()):
    q = bf((B, n, d), g)
    k = bf((B, n, S, d), g)
    v = bf((B, n, S, d), g)
    pos = torch.full((B, S), -1, dtype=torch.int32)
    for b in range(B):
        c = 0
        for t in range(length + 1):
            if t < pads or t in holes:
                continue
            pos[b, t] = c
            c += 1
    return q, k, v, pos


def attn_ref(q, k, v, pos, slopes, length):
    B, n, S, d = k.shape
    o = np.zeros((B, n * d))
    for b in range(B):
        for j in range(n):
            oo, _ = oracle.attend(f64(q[b, j]), f64(k[b, j, :length + 1]), f64(v[b, j, :length + 1]),
                                  pos[b, :length + 1].numpy(), float(slopes[j]))
            o[b, j * d:(j + 1) * d] = oo
    return o


@pytest.mark.parametrize("B,n,d,S,length,splits,pads,holes", [
    (1, 16, 64, 40, 0, 0, 0, ()),          # one key: o = v
    (1, 32, 128, 116, 115, 0, 0, ()),      # 7b1-like
    (3, 16, 64, 140, 37, 1, 5, (9,)),
    (3, 16, 64, 140, 37, 5, 5, (9,)),      # split-KV with pads and a hole
    (2, 112, 128, 132, 131, 0, 0, ()),     # 176B-shape heads (non-power-of-two slopes)
    (2, 4, 128, 300, 299, 16, 40, (41, 100)),
    (1, 2, 64, 200, 130, 7, 64, ()),       # several splits fully masked
    (32, 32, 128, 120, 66, 1, 3, (5,)),    # 1024 CTAs: more than are resident at once
    (8, 112, 128, 140, 100, 1, 0, ()),     # 176B-shape heads, 896 CTAs
    (64, 32, 128, 140, 100, 1, 2, (7,)),   # 2048 CTAs: K / V staged by bulk copies
    (16, 112, 128, 300, 280, 2, 0, ()),    # 3584 CTAs, two splits merged by the last
])
def test_attn_decode(B, n, d, S, length, splits, pads, holes):
    g = gen(B * 31 + n + d + S + length + splits)
    q, k, v, pos = make_cache(B, n, S, d, length, g, pads, holes)
    slopes = torch.tensor(oracle.alibi_slopes(n), dtype=torch.float32)
    o = bg.op_attn_decode(q.to(DEV), k.to(DEV), v.to(DEV), pos.to(DEV), slopes.to(DEV), length,
                          splits)
    ref = attn_ref(q, k, v, pos, slopes.double().numpy(), length)
    assert_kernel_close(o, ref, atol_rms=1e-3, what="attn_decode")


def test_attn_decode_single_key_is_value():
    g = gen(77)
    q, k, v, pos = make_cache(2, 16, 8, 64, 0, g)
    slopes = torch.tensor(oracle.alibi_slopes(16), dtype=torch.float32)
    o = bg.op_attn_decode(q.to(DEV), k.to(DEV), v.to(DEV), pos.to(DEV), slopes.to(DEV), 0, 1)
    assert torch.equal(o.cpu().view(2, 16, 64), v[:, :, 0])


# ---------------------------------------------------------------- LM head + argmax
@pytest.mark.parametrize("M,V,K", [(1, 1000, 1024), (4, 250880, 1024), (8, 50000, 4096),
                                   (13, 777, 256), (130, 3000, 512)])
def test_lmhead_argmax(M, V, K):
    g = gen(M + V + K)
    E = bf((V, K), g, 0.02)
    x = bf((M, K), g)
    tok, lg = bg.op_lmhead_argmax(x.to(DEV), E.to(DEV))
    ref = oracle.linear(f64(x), oracle.host_bits(E))
    # float32 logits: accumulation error ~ sqrt(K) * 2^-24 * rms, well under 1e-4 * rms
    assert_kernel_close(lg, ref, rel=1e-5, atol_rms=1e-4, what="logits")
    lgc = lg.cpu()
    # the token is the lowest index of the maximum of the kernel's own float32 logits
    mx = lgc.max(dim=1, keepdim=True).values
    first = (lgc == mx).int().argmax(dim=1)
    assert torch.equal(tok.cpu().long(), first.long())
    # and the oracle's argmax wherever the oracle's top-2 gap clears float32 noise
    top2 = np.sort(ref, axis=1)[:, -2:]
    for b in range(M):
        if top2[b, 1] - top2[b, 0] > 1e-4:
            assert int(tok[b]) == int(np.argmax(ref[b]))


def test_lmhead_argmax_ties_pick_lowest_index():
    K, V = 256, 4096
    g = gen(9)
    E = bf((V, K), g, 0.02)
    x = bf((2, K), g)
    E[100] = (x[0].float() * 0.5).to(torch.bfloat16)   # the clear maximum of row 0 ...
    E[3000] = E[100]                                    # ... tied exactly with a later row
    E[7] = (x[1].float() * 0.5).to(torch.bfloat16)
    E[6] = E[7]
    E[4095] = E[7]
    tok, lg = bg.op_lmhead_argmax(x.to(DEV), E.to(DEV))
    assert lg[0, 100] == lg[0, 3000]
    assert tok.tolist() == [100, 6]
    tok2, none = bg.op_lmhead_argmax(x.to(DEV), E.to(DEV), logits=False)
    assert none is None and tok2.tolist() == [100, 6]
