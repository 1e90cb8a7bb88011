"""ctypes front of the CPU oracle (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and has
no fallback to it.

The oracle takes the same bf16 / int8 bit patterns the GPU gets (copied to the
host) and computes in double; see ``bloom_oracle.h`` for what each call does.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import List, Optional

import numpy as np
import torch

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        _lib = C.CDLL(path)
        _declare(_lib)
    return _lib


P = C.c_void_p
I32 = C.c_int32
DBL = C.c_double


class OrcConfig(C.Structure):
    _fields_ = [("n_layer", I32), ("hidden", I32), ("n_head", I32), ("ffn", I32),
                ("vocab", I32), ("ln_eps", DBL), ("int8", I32)]


class OrcLinear(C.Structure):
    _fields_ = [("w", P), ("q", P), ("s", P), ("b", P)]


class OrcLayer(C.Structure):
    _fields_ = [("ln1_g", P), ("ln1_b", P), ("qkv", OrcLinear), ("o", OrcLinear),
                ("ln2_g", P), ("ln2_b", P), ("up", OrcLinear), ("down", OrcLinear)]


class OrcWeights(C.Structure):
    _fields_ = [("word_emb", P), ("emb_ln_g", P), ("emb_ln_b", P), ("lnf_g", P),
                ("lnf_b", P), ("layers", C.POINTER(OrcLayer))]


class OrcSeq(C.Structure):
    _fields_ = [("max_seq", I32), ("len", I32), ("next_pos", I32),
                ("pos", C.POINTER(I32)), ("k", C.POINTER(DBL)), ("v", C.POINTER(DBL))]


def _declare(L):
    L.orc_bf16_to_double.restype = DBL
    L.orc_bf16_to_double.argtypes = [C.c_uint16]
    L.orc_alibi_slopes.argtypes = [I32, P]
    L.orc_gelu.restype = DBL
    L.orc_gelu.argtypes = [DBL]
    L.orc_layernorm.argtypes = [I32, P, P, P, DBL, P]
    L.orc_linear_apply.argtypes = [C.POINTER(OrcLinear), I32, I32, I32, P, P]
    L.orc_attend.argtypes = [I32, I32, P, P, P, P, DBL, P, P]
    L.orc_argmax.restype = I32
    L.orc_argmax.argtypes = [I32, P]
    L.orc_seq_new.restype = C.POINTER(OrcSeq)
    L.orc_seq_new.argtypes = [C.POINTER(OrcConfig), I32]
    L.orc_seq_free.argtypes = [C.POINTER(OrcSeq)]
    L.orc_seq_set_prompt.argtypes = [C.POINTER(OrcSeq), I32, P]
    L.orc_seq_advance.argtypes = [C.POINTER(OrcSeq)]
    L.orc_layer_prefill.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcLayer), I32, I32, P, P,
                                    C.POINTER(OrcSeq)]
    L.orc_layer_decode.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcLayer), I32, P,
                                   C.POINTER(OrcSeq)]
    L.orc_embed.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcWeights), I32, P, P]
    L.orc_head.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcWeights), I32, P, P]
    L.orc_prefill.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcWeights), I32, I32, P, P,
                              C.POINTER(C.POINTER(OrcSeq)), P, P]
    L.orc_decode.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcWeights), I32, P,
                             C.POINTER(C.POINTER(OrcSeq)), P, P]
    L.orc_forward_full.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcWeights), I32, P, P, P]
    L.orc_num_threads.restype = I32


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else C.c_void_p(a.ctypes.data)


def host_bits(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """Host numpy copy of a tensor's raw bits (bf16 -> uint16, int8 -> int8)."""
    if t is None:
        return None
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def bf16_bits(a) -> np.ndarray:
    """bf16 bit patterns of float values (round to nearest even)."""
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def as_f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


# ---------------------------------------------------------------- building blocks
def alibi_slopes(n_head: int) -> np.ndarray:
    out = np.zeros(n_head, dtype=np.float64)
    lib().orc_alibi_slopes(n_head, _ptr(out))
    return out


def gelu(x: float) -> float:
    return lib().orc_gelu(float(x))


def layernorm(x, g_bits=None, b_bits=None, eps=1e-5) -> np.ndarray:
    x = as_f64(x)
    y = np.zeros_like(x)
    h = x.shape[-1]
    for i in range(x.size // h):
        lib().orc_layernorm(h, _ptr(x.reshape(-1, h)[i]), _ptr(g_bits), _ptr(b_bits), eps,
                            _ptr(y.reshape(-1, h)[i]))
    return y


def linear(x, w_bits=None, bias_bits=None, q=None, s_bits=None) -> np.ndarray:
    """y[M][N] = x[M][K] W^T + b with W given as bf16 bits [N][K] or int8 + scales."""
    x = as_f64(np.atleast_2d(x))
    M, K = x.shape
    N = (w_bits if w_bits is not None else q).shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    lin = OrcLinear(_ptr(w_bits), _ptr(q), _ptr(s_bits), _ptr(bias_bits))
    lib().orc_linear_apply(C.byref(lin), N, K, M, _ptr(x), _ptr(y))
    return y


def attend(q, keys, vals, pos, slope):
    """(o[d], probs[nk]) for one query of one head."""
    q, keys, vals = as_f64(q), as_f64(keys), as_f64(vals)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    d = q.shape[0]
    nk = keys.shape[0]
    o = np.zeros(d)
    p = np.zeros(max(nk, 1))
    lib().orc_attend(d, nk, _ptr(q), _ptr(keys), _ptr(vals), _ptr(pos), float(slope), _ptr(o),
                     _ptr(p))
    return o, p[:nk]


def argmax(v) -> int:
    v = as_f64(v)
    return int(lib().orc_argmax(v.shape[0], _ptr(v)))


def num_threads() -> int:
    return int(lib().orc_num_threads())


def sample_top_p(logits, temperature: float, top_p: float, u: float) -> int:
    """Per-member sampling of one row, float64, from its definition.

    "Hugging Face BLOOM Inference Optimization", Webserver Architecture and
    Request Handling: the custom generation loop applies each batch member's
    own sampling parameters (temperature, top-p).  Top-p (nucleus) sampling:
    p = softmax(logits / temperature); sort the tokens by probability, highest
    first (equal probabilities: lower index first); the nucleus is the shortest
    prefix of that order whose probabilities sum to at least top_p; the
    distribution renormalised over the nucleus is sampled by inverting its
    cumulative sum, taken in vocabulary order, at the caller's uniform number
    u in [0, 1) (the random number is an input, so both sides draw the same).
    temperature <= 0 is greedy: the argmax, lowest index on ties (so is a row
    with no finite maximum).  top_p >= 1 keeps every token.
    """
    z = as_f64(logits).ravel()
    V = z.shape[0]
    if not temperature > 0.0 or not np.isfinite(z.max()):
        return int(np.flatnonzero(z == z.max())[0])
    p = np.exp((z - z.max()) / temperature)
    p = p / p.sum()
    order = np.lexsort((np.arange(V), -p))           # probability desc, index asc
    cum = np.cumsum(p[order])
    n = V if top_p >= 1.0 else min(V, int(np.searchsorted(cum, top_p, side="left")) + 1)
    keep = np.zeros(V, dtype=bool)
    keep[order[:n]] = True
    q = np.where(keep, p, 0.0)
    c = np.cumsum(q / q.sum())                        # vocabulary order
    i = int(np.searchsorted(c, u, side="right"))      # first index with c > u
    if i >= V:                                        # u at the top of the rounding
        i = int(np.flatnonzero(keep)[-1])
    return i


# ---------------------------------------------------------------- whole model
class Model:
    """Oracle view of a ``synth.Weights`` stack (bits copied to the host)."""

    def __init__(self, weights, n_layer: Optional[int] = None):
        sh = weights.shape
        self.shape = sh
        self.n_layer = len(weights.layers) if n_layer is None else n_layer
        self.cfg = OrcConfig(self.n_layer, sh.hidden, sh.n_head, sh.ffn, sh.vocab, sh.ln_eps,
                             1 if sh.int8 else 0)
        keep: List[np.ndarray] = []

        def hb(t):
            a = host_bits(t)
            if a is not None:
                keep.append(a)
            return a

        self._emb = hb(weights.word_emb)
        self._top = [hb(weights.emb_ln_g), hb(weights.emb_ln_b), hb(weights.lnf_g),
                     hb(weights.lnf_b)]
        arr = (OrcLayer * max(self.n_layer, 1))()
        for i in range(self.n_layer):
            Lw = weights.layers[i]

            def lin(name):
                if sh.int8:
                    return OrcLinear(None, _ptr(hb(Lw["q_" + name])), _ptr(hb(Lw["s_" + name])),
                                     _ptr(hb(Lw["b_" + name])))
                return OrcLinear(_ptr(hb(Lw["w_" + name])), None, None, _ptr(hb(Lw["b_" + name])))

            arr[i] = OrcLayer(_ptr(hb(Lw["ln1_g"])), _ptr(hb(Lw["ln1_b"])), lin("qkv"), lin("o"),
                              _ptr(hb(Lw["ln2_g"])), _ptr(hb(Lw["ln2_b"])), lin("up"),
                              lin("down"))
        self._layers = arr
        self._keep = keep
        self.w = OrcWeights(_ptr(self._emb), _ptr(self._top[0]), _ptr(self._top[1]),
                            _ptr(self._top[2]), _ptr(self._top[3]),
                            C.cast(arr, C.POINTER(OrcLayer)))

    # -- sequences
    def new_seqs(self, B: int, max_seq: int):
        return Seqs(self, B, max_seq)

    def prefill(self, seqs: "Seqs", tokens, mask, taps: bool = False):
        tokens = np.ascontiguousarray(np.asarray(tokens), dtype=np.int32)
        mask = np.ascontiguousarray(np.asarray(mask), dtype=np.uint8)
        B, T = tokens.shape
        logits = np.zeros((B, self.shape.vocab))
        tp = np.zeros((self.n_layer + 1, B, T, self.shape.hidden)) if taps else None
        lib().orc_prefill(C.byref(self.cfg), C.byref(self.w), B, T, _ptr(tokens), _ptr(mask),
                          seqs.arr, _ptr(logits), _ptr(tp))
        return (logits, tp) if taps else logits

    def decode(self, seqs: "Seqs", tokens, taps: bool = False):
        tokens = np.ascontiguousarray(np.asarray(tokens).reshape(-1), dtype=np.int32)
        B = tokens.shape[0]
        logits = np.zeros((B, self.shape.vocab))
        tp = np.zeros((self.n_layer + 1, B, self.shape.hidden)) if taps else None
        lib().orc_decode(C.byref(self.cfg), C.byref(self.w), B, _ptr(tokens), seqs.arr,
                         _ptr(logits), _ptr(tp))
        return (logits, tp) if taps else logits

    def forward_full(self, tokens, mask):
        tokens = np.ascontiguousarray(np.asarray(tokens).reshape(-1), dtype=np.int32)
        mask = np.ascontiguousarray(np.asarray(mask).reshape(-1), dtype=np.uint8)
        T = tokens.shape[0]
        logits = np.zeros((T, self.shape.vocab))
        lib().orc_forward_full(C.byref(self.cfg), C.byref(self.w), T, _ptr(tokens), _ptr(mask),
                               _ptr(logits))
        return logits

    def embed(self, tokens):
        tokens = np.ascontiguousarray(np.asarray(tokens).reshape(-1), dtype=np.int32)
        x = np.zeros((tokens.shape[0], self.shape.hidden))
        lib().orc_embed(C.byref(self.cfg), C.byref(self.w), tokens.shape[0], _ptr(tokens),
                        _ptr(x))
        return x

    def head(self, x):
        x = as_f64(np.atleast_2d(x))
        logits = np.zeros((x.shape[0], self.shape.vocab))
        lib().orc_head(C.byref(self.cfg), C.byref(self.w), x.shape[0], _ptr(x), _ptr(logits))
        return logits

    def layer_prefill(self, layer: int, x, mask, seq: Optional["Seqs"] = None, b: int = 0):
        """One layer over one sequence's T slots; x[T][h] -> new x."""
        x = as_f64(x).copy()
        mask = np.ascontiguousarray(np.asarray(mask).reshape(-1), dtype=np.uint8)
        T = x.shape[0]
        pos = np.zeros(T, dtype=np.int32)
        c = 0
        for t in range(T):
            pos[t] = c if mask[t] else -1
            c += int(mask[t] != 0)
        sp = None
        if seq is not None:
            sp = seq.arr[b]
            if sp.contents.len != T:
                lib().orc_seq_set_prompt(sp, T, _ptr(mask))
        lib().orc_layer_prefill(C.byref(self.cfg), C.byref(self._layers[layer]), layer, T,
                                _ptr(pos), _ptr(x), sp)
        return x

    def layer_decode(self, layer: int, x, seqs: "Seqs", b: int):
        x = as_f64(x).copy()
        lib().orc_layer_decode(C.byref(self.cfg), C.byref(self._layers[layer]), layer, _ptr(x),
                               seqs.arr[b])
        return x


class Seqs:
    """B oracle KV caches."""

    def __init__(self, model: Model, B: int, max_seq: int):
        self.model = model
        self.B = B
        self.max_seq = max_seq
        self.arr = (C.POINTER(OrcSeq) * B)()
        for b in range(B):
            self.arr[b] = lib().orc_seq_new(C.byref(model.cfg), max_seq)

    def __del__(self):
        try:
            for b in range(self.B):
                lib().orc_seq_free(self.arr[b])
        except Exception:
            pass

    def advance(self, b: int):
        lib().orc_seq_advance(self.arr[b])

    def state(self, b: int):
        s = self.arr[b].contents
        return s.len, s.next_pos, np.ctypeslib.as_array(s.pos, shape=(self.max_seq,)).copy()

    def kv(self, b: int):
        """(K, V) views [n_layer][n_head][max_seq][d] of sequence b (writable)."""
        sh = self.model.shape
        s = self.arr[b].contents
        shp = (self.model.n_layer, sh.n_head, self.max_seq, sh.head_dim)
        return (np.ctypeslib.as_array(s.k, shape=shp), np.ctypeslib.as_array(s.v, shape=shp))
