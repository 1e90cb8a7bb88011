"""Independent float64 restatement of the BLOOM forward, for pinning the oracle.

Written as dense tensor algebra with torch library routines (layer_norm,
linear, scaled_dot_product_attention with an explicit additive mask matrix,
gelu(approximate='tanh')), so it shares neither structure nor code with the
oracle's loops.  Test-only; tiny shapes.
"""
import math

import torch
import torch.nn.functional as F


def slopes_geometric(n: int) -> torch.Tensor:
    """ALiBi slopes as geometric sequences: for a power of two m, start = ratio
    = 2^(-8/m).  With n not a power of two, take the m-sequence for the largest
    power of two m <= n, then every other term (1st, 3rd, ...) of the sequence
    for 2m until n slopes are listed."""
    m = 2 ** int(math.floor(math.log2(n)))

    def geo(k):
        r = 2.0 ** (-8.0 / k)
        out, v = [], 1.0
        for _ in range(k):
            v *= r
            out.append(v)
        return out

    s = geo(m)
    if m != n:
        s += geo(2 * m)[0::2][: n - m]
    return torch.tensor(s, dtype=torch.float64)


def _dense(w):
    return w.double()


def weight(L, name, int8):
    if int8:
        return L["q_" + name].double() * L["s_" + name].double()[:, None]
    return L["w_" + name].double()


def forward(weights, tokens, mask, n_layer=None, round_bf16=False):
    """Logits [T, V] of every slot of one sequence.

    round_bf16: also round, as the GPU path does, the LayerNorm outputs, q / k /
    v, the attention output and the MLP intermediate to bf16 (the residual
    stream and the logits stay float64) -- the same method with the same
    rounding points, for telling compounding rounding from kernel error."""
    sh = weights.shape
    dev = weights.word_emb.device

    def rd(t):
        return t.to(torch.bfloat16).double() if round_bf16 else t
    h, n, d = sh.hidden, sh.n_head, sh.head_dim
    eps = sh.ln_eps
    L_ = len(weights.layers) if n_layer is None else n_layer
    tokens = torch.as_tensor(tokens).long().reshape(-1).to(dev)
    valid = torch.as_tensor(mask).bool().reshape(-1).to(dev)
    T = tokens.shape[0]
    E = _dense(weights.word_emb)
    x = F.layer_norm(E[tokens], (h,), weights.emb_ln_g.double(), weights.emb_ln_b.double(), eps)
    pos = torch.cumsum(valid.long(), 0) - 1
    slopes = slopes_geometric(n).to(dev)
    causal = torch.tril(torch.ones(T, T, dtype=torch.bool, device=dev))
    allowed = causal & valid[None, :]
    bias = slopes[:, None, None] * pos.double()[None, None, :]           # [n, 1, T]
    addmask = torch.where(allowed[None], bias.expand(n, T, T),
                          torch.tensor(-math.inf, dtype=torch.float64, device=dev))
    has_key = allowed.any(dim=1)
    # rows with no key: give them one finite entry so SDPA stays finite; zeroed below
    addmask[:, ~has_key, 0] = 0.0
    for l in range(L_):
        Lw = weights.layers[l]
        a = rd(F.layer_norm(x, (h,), Lw["ln1_g"].double(), Lw["ln1_b"].double(), eps))
        qkv = rd(F.linear(a, weight(Lw, "qkv", sh.int8), Lw["b_qkv"].double()))
        qkv = qkv.view(T, n, 3, d)
        q, k, v = (qkv[:, :, i].transpose(0, 1) for i in range(3))          # [n, T, d]
        o = F.scaled_dot_product_attention(q, k, v, attn_mask=addmask)     # scale 1/sqrt(d)
        o = rd(o.transpose(0, 1).reshape(T, h))
        o[~has_key] = 0.0
        o[~valid] = 0.0
        x = x + F.linear(o, weight(Lw, "o", sh.int8), Lw["b_o"].double())
        m = rd(F.layer_norm(x, (h,), Lw["ln2_g"].double(), Lw["ln2_b"].double(), eps))
        u = rd(F.gelu(F.linear(m, weight(Lw, "up", sh.int8), Lw["b_up"].double()),
                      approximate="tanh"))
        x = x + F.linear(u, weight(Lw, "down", sh.int8), Lw["b_down"].double())
    xf = rd(F.layer_norm(x, (h,), weights.lnf_g.double(), weights.lnf_b.double(), eps))
    return F.linear(xf, E)
