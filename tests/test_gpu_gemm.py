"""Tensor-core (tcgen05) prefill GEMM against the oracle.

Op level: y = epilogue(x W^T + b) over shapes that span several 128 x 256
tiles, ragged M / N edges and K tails that are not a multiple of the 64-wide
k-block.  Model level: prefill batches of >= 128 tokens route their four
linear layers through this kernel; a teacher-forced layer and a whole
generation are checked against the oracle, and against the weight-streaming
path (BLOOM_FLAG_NO_TC_GEMM) for the same inputs.
"""
import gc

import numpy as np
import pytest
import torch

import bloom_decoder_token_gb300 as bg
from bloom_decoder_token_gb300 import synth
import oracle
from parity import assert_kernel_close, assert_stream_close, f64, max_abs
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


def gen(seed):
    return torch.Generator().manual_seed(seed)


def bf(shape, g, std=1.0, mean=0.0):
    return (torch.randn(shape, generator=g, dtype=torch.float64) * std + mean).to(torch.bfloat16)


# (M, N, K): one exact tile; ragged M and N with several k-blocks; K tails of
# 40 and 8 elements; the 560m QKV / up / down shapes; an N below one tile.
SHAPES = [(128, 256, 64), (130, 300, 192), (257, 520, 1000), (1, 64, 64), (200, 24, 72),
          (256, 3072, 1024), (256, 4096, 1024), (256, 1024, 4096), (384, 768, 2056)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("epi", [bg.EPI_STORE, bg.EPI_GELU, bg.EPI_RESID],
                         ids=["store", "gelu", "resid"])
def test_gemm(M, N, K, epi):
    g = gen(M * 7919 + N * 31 + K + epi)
    W = bf((N, K), g, 0.02)
    x = bf((M, K), g, 1.0)
    bias = bf((N,), g, 0.5)
    y0 = bf((M, N), g, 1.0)
    acc = oracle.linear(f64(x), oracle.host_bits(W), oracle.host_bits(bias))
    y = y0.to(DEV).clone()
    bg.op_gemm(x.to(DEV), W.to(DEV), bias=bias.to(DEV), epilogue=epi, y=y)
    if epi == bg.EPI_STORE:
        ref = acc
    elif epi == bg.EPI_GELU:
        ref = np.vectorize(oracle.gelu)(acc)
    else:
        ref = f64(y0) + acc
    assert_kernel_close(y, ref, what=f"gemm {M}x{N}x{K}")


def test_gemm_no_bias_and_empty():
    g = gen(3)
    W = bf((300, 128), g, 0.02)
    x = bf((140, 128), g)
    y = bg.op_gemm(x.to(DEV), W.to(DEV))
    assert_kernel_close(y, oracle.linear(f64(x), oracle.host_bits(W)), what="no bias")
    e = bg.op_gemm(torch.empty(0, 128, dtype=torch.bfloat16, device=DEV), W.to(DEV))
    assert e.shape == (0, 300)


def test_gemm_matches_streaming_kernel():
    """Both kernels accumulate the same products in float32: results agree to
    within a couple of bf16 ulps of the output (only the summation order differs)."""
    g = gen(11)
    W = bf((1536, 1024), g, 0.02)
    x = bf((512, 1024), g)
    b = bf((1536,), g, 0.5)
    yt = bg.op_gemm(x.to(DEV), W.to(DEV), bias=b.to(DEV)).float()
    ys = bg.op_linear(x.to(DEV), w=W.to(DEV), bias=b.to(DEV)).float()
    tol = 2.0 ** -7 * ys.abs() + 1e-3
    assert bool(((yt - ys).abs() <= tol).all())


# ---------------------------------------------------------------- model level
def prefill_shape():
    # one BLOOM-560m-width layer, 4 ragged prompts of 64 tokens: M = 256 prefill rows
    return synth.PRESETS["block"].with_(batch=4, prompt=64, new_tokens=4, ragged=True)


@pytest.mark.parametrize("flags", [0, bg.FLAG_NO_TC_GEMM], ids=["tcgen05", "streaming"])
def test_prefill_layer_teacher_forced(flags):
    shape = prefill_shape()
    w = synth.make_weights(shape, seed=4, random_affine=True)
    ids, mask = synth.make_prompts(shape, seed=4)
    B, T = ids.shape
    gm = bg.Model(w.to(DEV), max_batch=B, max_tokens=B * T, max_seq=T + 1, flags=flags)
    kv = gm.new_kv(B, T + 1)
    om = oracle.Model(w)
    seqs = om.new_seqs(B, T + 1)
    _, taps = om.prefill(seqs, ids.numpy(), mask.numpy(), taps=True)
    gm.kv_set_prompt(kv, mask.to(DEV))
    x_in = torch.from_numpy(taps[0].reshape(B * T, -1)).float()
    xt = x_in.to(DEV)
    gm.layer_prefill(kv, 0, xt, B, T)
    ref = np.concatenate([om.layer_prefill(0, f64(x_in[b * T:(b + 1) * T]), mask[b].numpy())
                          for b in range(B)])
    assert_stream_close(xt, ref, what="teacher-forced prefill layer")
    gm.check_device()
    gm.close()


@pytest.mark.parametrize("affine", [False, True], ids=["cfg", "random_affine"])
def test_prefill_generation_through_tcgen05(affine):
    shape = prefill_shape().with_(n_layer=2, vocab=4096)
    w = synth.make_weights(shape, seed=5, random_affine=affine)
    generate_parity(shape, w, steps=3, tol=2e-2)


def test_prefill_paths_agree():
    """Greedy tokens and logits of the two prefill paths for the same prompts."""
    shape = prefill_shape().with_(n_layer=2, vocab=4096)
    w = synth.make_weights(shape, seed=6).to(DEV)
    ids, mask = synth.make_prompts(shape, seed=6)
    B, T = ids.shape
    out = []
    for flags in (0, bg.FLAG_NO_TC_GEMM):
        gm = bg.Model(w, max_batch=B, max_tokens=B * T, max_seq=T + 1, flags=flags)
        kv = gm.new_kv(B, T + 1)
        lg = torch.empty(B, shape.vocab, dtype=torch.float32, device=DEV)
        tok = gm.prefill(kv, ids.to(DEV), mask.to(DEV), logits=lg)
        gm.check_device()
        out.append((tok.cpu(), lg.cpu()))
        gm.close()
    assert max_abs(out[0][1], out[1][1].double().numpy()) <= 2e-2


# ---------------------------------------------------------------- tensor-core decode linear
# (M, N, K): every token-column class (16 .. 256), split K (narrow N, long K),
# ragged N and K tails, one token.
DECODE_SHAPES = [(8, 3072, 1024), (1, 300, 192), (17, 520, 1000), (64, 4096, 4096),
                 (130, 1040, 2048), (256, 256, 16384), (16, 12288, 4096), (33, 128, 64)]


@pytest.mark.parametrize("M,N,K", DECODE_SHAPES)
@pytest.mark.parametrize("epi", [bg.EPI_STORE, bg.EPI_GELU, bg.EPI_RESID],
                         ids=["store", "gelu", "resid"])
def test_linear_tc(M, N, K, epi):
    g = gen(M * 131 + N * 7 + K + epi)
    W = bf((N, K), g, 0.02)
    x = bf((M, K), g, 1.0)
    bias = bf((N,), g, 0.5)
    y0 = bf((M, N), g, 1.0)
    acc = oracle.linear(f64(x), oracle.host_bits(W), oracle.host_bits(bias))
    y = y0.to(DEV).clone()
    bg.op_linear_tc(x.to(DEV), W.to(DEV), bias=bias.to(DEV), epilogue=epi, y=y)
    if epi == bg.EPI_STORE:
        ref = acc
    elif epi == bg.EPI_GELU:
        ref = np.vectorize(oracle.gelu)(acc)
    else:
        ref = f64(y0) + acc
    assert_kernel_close(y, ref, what=f"linear_tc {M}x{N}x{K}")


def test_linear_tc_deterministic_split_k():
    """K split over a thread-block cluster: partials summed in split order, so
    repeated runs agree bitwise."""
    g = gen(77)
    W = bf((512, 16384), g, 0.02).to(DEV)
    x = bf((24, 16384), g).to(DEV)
    y1 = bg.op_linear_tc(x, W)
    y2 = bg.op_linear_tc(x, W)
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("flags", [0, bg.FLAG_NO_TC_GEMM], ids=["tcgen05", "streaming"])
def test_decode_generation_batch16(flags):
    shape = synth.PRESETS["560m"].with_(n_layer=2, vocab=5000, batch=16)
    w = synth.make_weights(shape, seed=12, random_affine=True)
    generate_parity(shape, w, steps=4, tol=2e-2, flags=flags)


@pytest.mark.parametrize("B", [8, 16, 32])
@pytest.mark.parametrize("flags", [0, bg.FLAG_NO_TC_GEMM], ids=["tcgen05", "streaming"])
def test_decode_block_linears_through_tcgen05(B, flags):
    """An 8192-wide MLP (up: N = 8192, down: K = 8192) at 8, 16 and 32 sequences:
    the decode step runs the block linears on the tensor-core decode kernel
    (K split over a cluster, partials summed through distributed shared
    memory), against the oracle, and against the weight-streaming path for the
    same inputs."""
    shape = synth.PRESETS["560m"].with_(n_layer=2, vocab=4096, ffn=8192, batch=B, prompt=8,
                                        ragged=True)
    w = synth.make_weights(shape, seed=21, random_affine=True)
    generate_parity(shape, w, steps=3, tol=2e-2, flags=flags)


def test_decode_qkv_through_tcgen05():
    """A 2816-wide stack with 22 heads of 128 at 8 sequences: the decode QKV
    linear (8448 rows) runs on the tensor-core decode kernel with its K split
    over a cluster, the Q/K/V scatter into the cache applied by the CTA that
    sums each token group.  Against the oracle."""
    shape = synth.PRESETS["560m"].with_(n_layer=1, hidden=2816, n_head=22, ffn=11264,
                                        vocab=4096, batch=8, prompt=8, ragged=True)
    w = synth.make_weights(shape, seed=23, random_affine=True)
    generate_parity(shape, w, steps=2, tol=2e-2)


@pytest.mark.parametrize("B", [1, 2, 3])
@pytest.mark.parametrize("flags", [0, bg.FLAG_NO_TC_GEMM], ids=["tcgen05", "streaming"])
def test_decode_small_batch_through_tcgen05(B, flags):
    """One to three sequences of a stack narrow enough for the tensor-core
    decode kernel at every batch size.  Default: every block linear there
    (LayerNorm launches of their own), the head on the weight-streaming kernel
    with ln_f fused at one and two sequences and on the tensor-core kernel from
    three.  Streaming: QKV, up and the head with the LayerNorm fused at one and
    two sequences."""
    shape = synth.PRESETS["560m"].with_(n_layer=2, vocab=3000, batch=B, prompt=8, ragged=True)
    w = synth.make_weights(shape, seed=31 + B, random_affine=True)
    generate_parity(shape, w, steps=3, tol=2e-2, flags=flags)


# The 176B-layer matrices at full size (QKV 43008 x 14336, up 57344 x 14336,
# down 14336 x 57344) on the tensor-core decode kernel, compared with the oracle
# on 384 sampled output rows (the oracle computes those rows directly).
@pytest.mark.slow
@pytest.mark.parametrize("N,K", [(43008, 14336), (57344, 14336), (14336, 57344)],
                         ids=["qkv", "up", "down"])
@pytest.mark.parametrize("M", [8, 32, 256])
def test_linear_tc_176b_shapes_sampled(N, K, M):
    g = torch.Generator(device=DEV).manual_seed(N + K + M)
    W = (0.02 * torch.randn(N, K, generator=g, device=DEV)).to(torch.bfloat16)
    x = torch.randn(M, K, generator=g, device=DEV).to(torch.bfloat16)
    bias = (0.5 * torch.randn(N, generator=g, device=DEV)).to(torch.bfloat16)
    y = bg.op_linear_tc(x, W, bias=bias, epilogue=bg.EPI_GELU)
    rows = torch.randperm(N, generator=torch.Generator().manual_seed(M))[:384].sort().values
    Ws = W[rows.to(DEV)].cpu()
    acc = oracle.linear(f64(x), oracle.host_bits(Ws), oracle.host_bits(bias[rows.to(DEV)].cpu()))
    ref = np.vectorize(oracle.gelu)(acc)
    assert_kernel_close(y[:, rows.to(DEV)], ref, what=f"linear_tc {M}x{N}x{K} sampled rows")
    del W
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- int8 on the tensor-core decode kernel
# int8 codes are widened exactly into a TMEM A operand (f16 with the activations
# converted to f16 up to 32 token columns, bf16 above); ragged N, a K tail that
# is not a multiple of the 128-wide int8 k-block, split and unsplit.
INT8_TC_SHAPES = [(3, 300, 192), (8, 3072, 1024), (17, 520, 1040), (32, 4096, 4096),
                  (64, 1040, 2048), (100, 256, 16384), (128, 12288, 4096), (33, 128, 64)]


@pytest.mark.parametrize("M,N,K", INT8_TC_SHAPES)
@pytest.mark.parametrize("epi", [bg.EPI_STORE, bg.EPI_GELU, bg.EPI_RESID],
                         ids=["store", "gelu", "resid"])
def test_linear_tc_int8(M, N, K, epi):
    g = gen(M * 313 + N * 11 + K + epi)
    W = bf((N, K), g, 0.02)
    q, sc = synth.quantize_rows_int8(W)
    x = bf((M, K), g, 1.0)
    bias = bf((N,), g, 0.5)
    y0 = bf((M, N), g, 1.0)
    acc = oracle.linear(f64(x), q=oracle.host_bits(q), s_bits=oracle.host_bits(sc),
                        bias_bits=oracle.host_bits(bias))
    y = y0.to(DEV).clone()
    bg.op_linear_tc(x.to(DEV), q=q.to(DEV), scale=sc.to(DEV), bias=bias.to(DEV), epilogue=epi, y=y)
    if epi == bg.EPI_STORE:
        ref = acc
    elif epi == bg.EPI_GELU:
        ref = np.vectorize(oracle.gelu)(acc)
    else:
        ref = f64(y0) + acc
    assert_kernel_close(y, ref, what=f"linear_tc int8 {M}x{N}x{K}")


@pytest.mark.parametrize("reps", [1, 2], ids=["f16-form", "bf16-form"])
def test_linear_tc_int8_every_code(reps):
    """Every int8 code (-128 .. 127), at even and odd k, in every 16-byte chunk of
    the 128-byte swizzled rows and in both 128-wide k-blocks, comes out exactly:
    with unit scales, no bias and one-hot activations y[m][n] = q[n][p_m].  This
    pins the widening and the order of the two 16-bit values in each TMEM column
    of the A operand, in the f16 form (20 token columns) and the bf16 form (40)."""
    N, K = 512, 256
    n = torch.arange(N).unsqueeze(1)
    k = torch.arange(K).unsqueeze(0)
    q = ((3 * n + k) % 256).to(torch.uint8).view(torch.int8)
    pos = [0, 1, 2, 3, 14, 15, 16, 17, 31, 62, 63, 64, 65, 100, 127, 128, 129, 200, 254, 255] * reps
    x = torch.zeros(len(pos), K, dtype=torch.bfloat16)
    for m, p in enumerate(pos):
        x[m, p] = 1.0
    scale = torch.ones(N, dtype=torch.bfloat16)
    y = bg.op_linear_tc(x.to(DEV), q=q.to(DEV), scale=scale.to(DEV))
    expect = torch.stack([q[:, p].float() for p in pos])
    assert torch.equal(y.cpu().float(), expect)


@pytest.mark.parametrize("B", [3, 8, 32])
def test_decode_int8_through_tcgen05(B):
    """int8 block linears of decode steps on the tensor-core decode kernel
    (QKV, dense, up, down; the head stays bf16), against the oracle at the int8
    tolerance 6e-2."""
    shape = synth.PRESETS["560m"].with_(n_layer=2, vocab=3000, batch=B, prompt=8, ragged=True,
                                        int8=True)
    w = synth.make_weights(shape, seed=41 + B, random_affine=True)
    generate_parity(shape, w, steps=3, tol=6e-2)


# ---------------------------------------------------------------- prefill attention on tensor cores
def _prefill_layer_vs_oracle(shape, seed, mask, x_std=1.0, tol=2e-2):
    """One teacher-forced prefill layer of B prompts of T slots (mask [B][T]):
    GPU (tcgen05 GEMM + tensor-core attention) against the oracle layer."""
    w = synth.make_weights(shape.with_(n_layer=1), seed=seed, device=DEV, random_affine=True)
    B, T = mask.shape
    gm = bg.Model(w, max_batch=B, max_tokens=B * T, max_seq=T + 1)
    kv = gm.new_kv(B, T + 1)
    gm.kv_set_prompt(kv, mask.to(DEV))
    g = torch.Generator().manual_seed(seed + 100)
    x_in = (x_std * torch.randn(B * T, shape.hidden, generator=g)).float()
    xt = x_in.to(DEV)
    gm.layer_prefill(kv, 0, xt, B, T)
    om = oracle.Model(synth.Weights(shape, w.word_emb[:1].cpu(), w.emb_ln_g.cpu(), w.emb_ln_b.cpu(),
                                    w.lnf_g.cpu(), w.lnf_b.cpu(),
                                    [{k: v.cpu() for k, v in w.layers[0].items()}]))
    for b in range(B):
        valid = mask[b].numpy().astype(bool)
        ref = om.layer_prefill(0, f64(x_in[b * T:(b + 1) * T]), mask[b].numpy())
        assert_stream_close(f64(xt[b * T:(b + 1) * T])[valid], ref[valid], tol=tol,
                            what=f"prefill layer row {b}")
    gm.check_device()
    gm.close()
    del w
    gc.collect()
    torch.cuda.empty_cache()


def test_prefill_attention_ragged_tiles():
    """Left-padded prompts of 300 slots (5 query tiles, a ragged last tile) and
    a prompt with holes in the middle, at head width 64: every query and key
    tile edge, pads as keys, pad queries."""
    shape = synth.PRESETS["block"]
    B, T = 3, 300
    mask = torch.ones(B, T, dtype=torch.uint8)
    mask[0, :37] = 0
    mask[1, :129] = 0
    mask[2, 100:140] = 0
    _prefill_layer_vs_oracle(shape, 51, mask)


@pytest.mark.slow
def test_prefill_layer_7b1_at_2048_tokens():
    """One 7b1-width layer (32 heads x 128) over a 2048-token prompt: the prefill
    GEMM at M = 2048 and the tensor-core attention over 32 x 32 tiles."""
    shape = synth.PRESETS["7b1"]
    mask = torch.ones(1, 2048, dtype=torch.uint8)
    _prefill_layer_vs_oracle(shape, 52, mask)
