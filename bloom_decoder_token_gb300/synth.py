"""Seeded synthetic inputs: model shapes, weights and prompts.

This module holds no arithmetic of the method.  It only draws numbers (from
torch's seeded generators) in the shapes the BLOOM decoder uses, so that the
CUDA library and the CPU oracle can be fed identical bits.  Neither side's
computation lives here.

Recipe (the same for every preset):
  * draw order: word embedding, embedding LN, then per layer qkv, o, up, down
    (weight then bias) and the two LayerNorms, then the final LN;
  * weights ~ N(0, 0.02) rounded to bf16;
  * biases 0 and LayerNorm gamma 1 / beta 0, unless ``random_affine`` is set,
    in which case biases ~ N(0, 0.02) and gamma ~ 1 + N(0, 0.1),
    beta ~ N(0, 0.1) (unit tests use this so that bias and affine errors show);
  * int8 presets store per-output-row symmetric codes: s = bf16(absmax/127),
    q = clamp(round_half_even(w / s), -127, 127); a zero row has s = 0, q = 0.
    The codes and scales are inputs to both sides; the oracle widens q * s.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Shape:
    """Sizes of a BLOOM decoder stack and of one generation job."""
    name: str
    n_layer: int
    hidden: int
    n_head: int
    ffn: int
    vocab: int
    batch: int
    prompt: int          # padded prompt length T
    new_tokens: int      # tokens generated (first one comes from the prefill)
    int8: bool = False
    ragged: bool = False  # left-padded prompts with lengths uniform in [8, prompt]
    ln_eps: float = 1e-5

    @property
    def head_dim(self) -> int:
        return self.hidden // self.n_head

    @property
    def max_seq(self) -> int:
        return self.prompt + self.new_tokens

    def with_(self, **kw) -> "Shape":
        return dataclasses.replace(self, **kw)


# The five workloads: one BLOOM block; the 560m, 7b1 and 176B-layer shapes; the
# 7b1 shape with int8 weight-only block linears.
PRESETS: Dict[str, Shape] = {
    "block": Shape("block", 1, 1024, 16, 4096, 1024, 1, 8, 9),
    "560m": Shape("560m", 24, 1024, 16, 4096, 250880, 8, 32, 100, ragged=True),
    "7b1": Shape("7b1", 30, 4096, 32, 16384, 250880, 1, 16, 100),
    "176b14": Shape("176b14", 14, 14336, 112, 57344, 250880, 1, 32, 100),
    "7b1int8": Shape("7b1int8", 30, 4096, 32, 16384, 250880, 1, 16, 100, int8=True),
}


def _normal(shape, gen, device, std=0.02, chunk=1 << 28) -> torch.Tensor:
    """N(0, std) rounded to bf16, drawn in chunks to bound fp32 temporaries."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        tmp = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        flat[s:e].copy_(tmp.mul_(std))
        del tmp
    return out


def quantize_rows_int8(w: torch.Tensor):
    """Per-row symmetric absmax codes: returns (q int8 [N,K], s bf16 [N])."""
    wf = w.float()
    absmax = wf.abs().amax(dim=1)
    s = (absmax / 127.0).to(torch.bfloat16)
    sf = s.float()
    safe = torch.where(sf > 0, sf, torch.ones_like(sf))
    q = torch.round(wf / safe[:, None]).clamp_(-127, 127)
    q = torch.where(sf[:, None] > 0, q, torch.zeros_like(q)).to(torch.int8)
    return q, s


class Weights:
    """Device or host tensors of one BLOOM stack (nn.Linear layout [out, in])."""

    def __init__(self, shape: Shape, word_emb, emb_ln_g, emb_ln_b, lnf_g, lnf_b,
                 layers: List[Dict[str, torch.Tensor]]):
        self.shape = shape
        self.word_emb = word_emb
        self.emb_ln_g, self.emb_ln_b = emb_ln_g, emb_ln_b
        self.lnf_g, self.lnf_b = lnf_g, lnf_b
        self.layers = layers

    def to(self, device) -> "Weights":
        mv = lambda t: None if t is None else t.to(device)
        return Weights(self.shape, mv(self.word_emb), mv(self.emb_ln_g), mv(self.emb_ln_b),
                       mv(self.lnf_g), mv(self.lnf_b),
                       [{k: mv(v) for k, v in L.items()} for L in self.layers])

    def nbytes(self) -> int:
        tot = 0
        for t in [self.word_emb, self.emb_ln_g, self.emb_ln_b, self.lnf_g, self.lnf_b]:
            tot += t.numel() * t.element_size()
        for L in self.layers:
            for t in L.values():
                if t is not None:
                    tot += t.numel() * t.element_size()
        return tot


LINEARS = ("qkv", "o", "up", "down")


def linear_dims(shape: Shape, name: str):
    h, F = shape.hidden, shape.ffn
    return {"qkv": (3 * h, h), "o": (h, h), "up": (F, h), "down": (h, F)}[name]


def make_weights(shape: Shape, seed: int = 0, device="cpu", random_affine: bool = False,
                 n_layer: Optional[int] = None) -> Weights:
    """Draw a seeded BLOOM stack.  ``n_layer`` may limit the layers drawn
    (the first layers are identical to those of the full stack)."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    h, V = shape.hidden, shape.vocab
    L = shape.n_layer if n_layer is None else n_layer

    def ln_pair():
        if random_affine:
            g = (1.0 + _normal((h,), gen, device, std=0.1).float()).to(torch.bfloat16)
            b = _normal((h,), gen, device, std=0.1)
        else:
            g = torch.ones(h, dtype=torch.bfloat16, device=device)
            b = torch.zeros(h, dtype=torch.bfloat16, device=device)
        return g, b

    def bias(n):
        if random_affine:
            return _normal((n,), gen, device)
        return torch.zeros(n, dtype=torch.bfloat16, device=device)

    word_emb = _normal((V, h), gen, device)
    emb_ln_g, emb_ln_b = ln_pair()
    layers = []
    for _ in range(L):
        d: Dict[str, torch.Tensor] = {}
        d["ln1_g"], d["ln1_b"] = ln_pair()
        for name in LINEARS:
            N, K = linear_dims(shape, name)
            w = _normal((N, K), gen, device)
            if shape.int8:
                q, s = quantize_rows_int8(w)
                d["q_" + name], d["s_" + name] = q, s
                del w
            else:
                d["w_" + name] = w
            d["b_" + name] = bias(N)
            if name == "o":
                d["ln2_g"], d["ln2_b"] = ln_pair()
        layers.append(d)
    lnf_g, lnf_b = ln_pair()
    return Weights(shape, word_emb, emb_ln_g, emb_ln_b, lnf_g, lnf_b, layers)


def make_prompts(shape: Shape, seed: int = 0, batch: Optional[int] = None,
                 prompt: Optional[int] = None):
    """Token ids [B,T] int32 and pad mask [B,T] uint8 (1 = token), on the CPU.

    Ragged presets draw each row's length uniformly in [8, T] and left-pad it;
    the padded length T is then the longest row.  Pad slots hold token 0."""
    B = shape.batch if batch is None else batch
    T = shape.prompt if prompt is None else prompt
    gen = torch.Generator()
    gen.manual_seed(seed + 1)
    if shape.ragged:
        lens = torch.randint(min(8, T), T + 1, (B,), generator=gen)
        T = int(lens.max())
    else:
        lens = torch.full((B,), T, dtype=torch.int64)
    ids = torch.randint(0, shape.vocab, (B, T), generator=gen, dtype=torch.int64)
    mask = torch.zeros(B, T, dtype=torch.uint8)
    for b in range(B):
        mask[b, T - int(lens[b]):] = 1
    ids = torch.where(mask.bool(), ids, torch.zeros_like(ids))
    return ids.to(torch.int32), mask


def make_tokens(shape: Shape, steps: int, seed: int = 0, batch: Optional[int] = None):
    """Seeded token ids [steps, B] int32 for teacher-forced decode steps."""
    B = shape.batch if batch is None else batch
    gen = torch.Generator()
    gen.manual_seed(seed + 2)
    return torch.randint(0, shape.vocab, (steps, B), generator=gen, dtype=torch.int64).to(
        torch.int32)
