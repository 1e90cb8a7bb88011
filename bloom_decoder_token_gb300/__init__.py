"""Python binding of the GB300 BLOOM decode engine (``libbloom.so``).

Argument marshalling only: every step of the path runs in the CUDA library
behind the C ABI of ``include/bloom.h``.  PyTorch supplies device memory and
streams.  There is no CPU fallback: if the library is missing, every entry
point raises.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import torch

from . import synth

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbloom.so")
_lib = None

BLOOM_OK = 0
STATUS = {0: "OK", 1: "E_INVALID", 2: "E_UNSUPPORTED", 3: "E_OOM", 4: "E_CAPACITY",
          5: "E_CUDA", 6: "E_DEVICE_FLAG"}
EPI_STORE, EPI_GELU, EPI_RESID = 0, 1, 2
FLAG_NO_GRAPH = 1
FLAG_NO_PDL = 2
FLAG_NO_LN_FUSION = 4
FLAG_NO_TC_GEMM = 8

OPS = ("embed", "layernorm", "qkv", "attn", "dense", "up", "down", "head")
KERNELS = ("embed_kernel", "layernorm_kernel", "linear_kernel", "gemv_tc_kernel",
           "gemm_tc_kernel", "attn_decode_kernel", "attn_prefill_kernel")

P = C.c_void_p
I32 = C.c_int32


class BloomError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"bloom {STATUS.get(status, status)}: {msg}")
        self.status = status


class Config(C.Structure):
    _fields_ = [("n_layer", I32), ("hidden", I32), ("n_head", I32), ("ffn", I32),
                ("vocab", I32), ("ln_eps", C.c_float), ("weight_dtype", I32),
                ("max_batch", I32), ("max_tokens", I32), ("max_seq", I32), ("flags", I32),
                ("wait_us", I32)]


class Linear(C.Structure):
    _fields_ = [("w", P), ("scale", P), ("bias", P)]


class LayerWeights(C.Structure):
    _fields_ = [("ln1_g", P), ("ln1_b", P), ("qkv", Linear), ("o", Linear), ("ln2_g", P),
                ("ln2_b", P), ("up", Linear), ("down", Linear)]


class WeightsC(C.Structure):
    _fields_ = [("word_emb", P), ("emb_ln_g", P), ("emb_ln_b", P), ("lnf_g", P), ("lnf_b", P),
                ("layers", C.POINTER(LayerWeights))]


MAX_BATCH = 256


class KVC(C.Structure):
    _fields_ = [("buf", P), ("bytes", C.c_size_t), ("batch", I32), ("max_seq", I32),
                ("len", I32), ("row_len", I32 * MAX_BATCH), ("row_active", C.c_uint8 * MAX_BATCH),
                ("host_buf", P), ("host_bytes", C.c_size_t), ("offload_from", I32)]


_SIGS = {
    "bloom_kv_bytes": (C.c_size_t, [C.POINTER(Config), I32, I32]),
    "bloom_create": (I32, [C.POINTER(Config), C.POINTER(WeightsC), C.POINTER(P)]),
    "bloom_kv_init": (I32, [P, C.POINTER(KVC), P, C.c_size_t, I32, I32, P]),
    "bloom_kv_bytes_offload": (I32, [C.POINTER(Config), I32, I32, I32, C.POINTER(C.c_size_t),
                                     C.POINTER(C.c_size_t)]),
    "bloom_kv_init_offload": (I32, [P, C.POINTER(KVC), P, C.c_size_t, P, C.c_size_t, I32, I32, I32,
                                    P]),
    "bloom_prefill": (I32, [P, C.POINTER(KVC), P, P, I32, I32, P, P, P]),
    "bloom_decode_step": (I32, [P, C.POINTER(KVC), P, P, P, P]),
    "bloom_decode_step_sampled": (I32, [P, C.POINTER(KVC), P, P, P, P, P, P, P]),
    "bloom_kv_admit": (I32, [P, C.POINTER(KVC), P, I32, P, P, I32, P, P, P]),
    "bloom_kv_retire": (I32, [P, C.POINTER(KVC), P, I32, P]),
    "bloom_generate": (I32, [P, C.POINTER(KVC), P, P, I32, I32, I32, P, P]),
    "bloom_check_device": (I32, [P, P]),
    "bloom_decode_profile": (I32, [P, C.POINTER(KVC), P, P, P, P, I32, P, P]),
    "bloom_destroy": (I32, [P]),
    "bloom_last_error": (C.c_char_p, []),
    "bloom_decode_launches": (I32, [P, I32]),
    "bloom_layer_decode": (I32, [P, C.POINTER(KVC), I32, P, P]),
    "bloom_kv_set_prompt": (I32, [P, C.POINTER(KVC), P, I32, I32, P]),
    "bloom_layer_prefill": (I32, [P, C.POINTER(KVC), I32, P, I32, I32, P]),
    "bloom_head": (I32, [P, P, I32, P, P, P]),
    "bloom_lm_head": (I32, [P, P, I32, P, P, P]),
    "bloom_embed": (I32, [P, P, I32, P, P]),
    "bloom_op_layernorm": (I32, [P, P, P, I32, I32, C.c_float, P, P]),
    "bloom_op_linear": (I32, [C.POINTER(Linear), I32, P, I32, I32, I32, I32, P, P]),
    "bloom_op_gemm": (I32, [C.POINTER(Linear), P, I32, I32, I32, I32, P, P]),
    "bloom_op_linear_tc": (I32, [C.POINTER(Linear), I32, P, I32, I32, I32, I32, P, P]),
    "bloom_op_attn_decode": (I32, [P, P, P, P, P, I32, I32, I32, I32, I32, I32, P, P]),
    "bloom_op_lmhead_argmax": (I32, [P, P, I32, I32, I32, P, P, P]),
    "bloom_op_sample": (I32, [P, I32, I32, C.c_int64, P, P, P, P, P]),
    "bloom_op_lmhead_argmax_noalloc": (I32, [P, P, I32, I32, I32, P, P, P]),
}
EXPORTS = tuple(_SIGS)


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def check(status: int):
    if status != BLOOM_OK:
        raise BloomError(status, lib().bloom_last_error().decode())


def _p(t: Optional[torch.Tensor]):
    return None if t is None else P(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return P(s.cuda_stream)


class KV:
    """A caller-owned KV cache (one device byte buffer) and its descriptor;
    with offload_from < n_layer the K and V of layers [offload_from, n_layer)
    live in a second, page-locked host buffer the kernels read directly."""

    def __init__(self, model: "Model", batch: int, max_seq: int, stream=None,
                 offload_from: Optional[int] = None):
        self.offload_from = model.n_layer if offload_from is None else int(offload_from)
        self.host = None
        if self.offload_from >= model.n_layer:
            n = lib().bloom_kv_bytes(C.byref(model.cfg), batch, max_seq)
            if n == 0:
                raise BloomError(1, "bloom_kv_bytes rejected the arguments")
            hn = 0
        else:
            dn, hb = C.c_size_t(), C.c_size_t()
            check(lib().bloom_kv_bytes_offload(C.byref(model.cfg), batch, max_seq,
                                               self.offload_from, C.byref(dn), C.byref(hb)))
            n, hn = dn.value, hb.value
        self.buf = torch.empty(n + 256, dtype=torch.uint8, device=model.device)
        off = (-self.buf.data_ptr()) % 256
        self.view = self.buf[off:off + n]
        self.c = KVC()
        if hn == 0:
            check(lib().bloom_kv_init(model.h, C.byref(self.c), P(self.view.data_ptr()), n, batch,
                                      max_seq, _stream(stream)))
        else:
            self.host = torch.empty(hn + 256, dtype=torch.uint8, pin_memory=True)
            hoff = (-self.host.data_ptr()) % 256
            self.host_view = self.host[hoff:hoff + hn]
            check(lib().bloom_kv_init_offload(model.h, C.byref(self.c), P(self.view.data_ptr()), n,
                                              P(self.host_view.data_ptr()), hn, batch, max_seq,
                                              self.offload_from, _stream(stream)))

    @property
    def len(self) -> int:
        return self.c.len

    @property
    def batch(self) -> int:
        return self.c.batch

    def row_len(self, b: int) -> int:
        return self.c.row_len[b]

    def row_active(self, b: int) -> bool:
        return bool(self.c.row_active[b])

    def tensors(self, model: "Model"):
        """Views of the cache regions (len, active, next_pos, pos, K, V) for inspection."""
        sh = model.shape
        B, S = self.c.batch, self.c.max_seq
        al = lambda x: (x + 255) // 256 * 256
        off_len = 256
        off_act = al(off_len + 4 * B)
        off_np = al(off_act + 4 * B)
        off_pos = al(off_np + 4 * B)
        layer = B * sh.n_head * S * sh.head_dim * 2
        nd = min(self.offload_from, model.n_layer)   # layers in the device buffer
        off_k = al(off_pos + 4 * B * S)
        off_v = al(off_k + layer * nd)
        v = self.view
        i32 = lambda a, n: v[a:a + 4 * n].view(torch.int32)
        bf = lambda buf, a, nl: buf[a:a + layer * nl].view(torch.bfloat16).view(
            nl, B, sh.n_head, S, sh.head_dim)
        out = {"len": i32(off_len, B), "active": i32(off_act, B), "next_pos": i32(off_np, B),
               "pos": i32(off_pos, B * S).view(B, S), "k": bf(v, off_k, nd), "v": bf(v, off_v, nd)}
        if self.host is not None:
            nh = model.n_layer - nd
            out["k_host"] = bf(self.host_view, 0, nh)
            out["v_host"] = bf(self.host_view, al(layer * nh), nh)
        return out


class Model:
    """A BLOOM stack on the current CUDA device, weights borrowed from torch tensors."""

    def __init__(self, weights: synth.Weights, max_batch: int, max_tokens: int, max_seq: int,
                 flags: int = 0, n_layer: Optional[int] = None, wait_us: int = 0):
        sh = weights.shape
        self.shape = sh
        self.weights = weights
        self.n_layer = len(weights.layers) if n_layer is None else n_layer
        self.device = weights.word_emb.device
        self.cfg = Config(self.n_layer, sh.hidden, sh.n_head, sh.ffn, sh.vocab, sh.ln_eps,
                          1 if sh.int8 else 0, max_batch, max_tokens, max_seq, flags, wait_us)
        arr = (LayerWeights * self.n_layer)()
        for i in range(self.n_layer):
            L = weights.layers[i]

            def lin(name):
                if sh.int8:
                    return Linear(_p(L["q_" + name]), _p(L["s_" + name]), _p(L["b_" + name]))
                return Linear(_p(L["w_" + name]), None, _p(L["b_" + name]))

            arr[i] = LayerWeights(_p(L["ln1_g"]), _p(L["ln1_b"]), lin("qkv"), lin("o"),
                                  _p(L["ln2_g"]), _p(L["ln2_b"]), lin("up"), lin("down"))
        self._arr = arr
        self._wc = WeightsC(_p(weights.word_emb), _p(weights.emb_ln_g), _p(weights.emb_ln_b),
                            _p(weights.lnf_g), _p(weights.lnf_b),
                            C.cast(arr, C.POINTER(LayerWeights)))
        h = P()
        check(lib().bloom_create(C.byref(self.cfg), C.byref(self._wc), C.byref(h)))
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            lib().bloom_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def decode_launches(self, batch: int) -> int:
        return lib().bloom_decode_launches(self.h, batch)

    def new_kv(self, batch: int, max_seq: int, stream=None, offload_from: Optional[int] = None) -> KV:
        return KV(self, batch, max_seq, stream, offload_from)

    def prefill(self, kv: KV, tokens, mask, out_tokens=None, logits=None, stream=None):
        B, T = tokens.shape
        if out_tokens is None:
            out_tokens = torch.empty(B, dtype=torch.int32, device=self.device)
        check(lib().bloom_prefill(self.h, C.byref(kv.c), _p(tokens), _p(mask), B, T,
                                  _p(out_tokens), _p(logits), _stream(stream)))
        return out_tokens

    def decode_step(self, kv: KV, next_tokens, out_tokens=None, logits=None, stream=None):
        if out_tokens is None:
            out_tokens = torch.empty(kv.batch, dtype=torch.int32, device=self.device)
        check(lib().bloom_decode_step(self.h, C.byref(kv.c), _p(next_tokens), _p(out_tokens),
                                      _p(logits), _stream(stream)))
        return out_tokens

    def decode_step_sampled(self, kv: KV, next_tokens, temperature, top_p, u, logits,
                            out_tokens=None, stream=None):
        """One decode step, then each active row's token sampled with its own
        temperature / top-p at the caller's uniform u (device float32 [B] each;
        logits: device float32 [B][V] scratch, written)."""
        if out_tokens is None:
            out_tokens = torch.empty(kv.batch, dtype=torch.int32, device=self.device)
        check(lib().bloom_decode_step_sampled(self.h, C.byref(kv.c), _p(next_tokens),
                                              _p(out_tokens), _p(logits), _p(temperature),
                                              _p(top_p), _p(u), _stream(stream)))
        return out_tokens

    def kv_admit(self, kv: KV, rows, tokens, mask, out_tokens=None, logits=None, stream=None):
        """Prefill new prompts (device tokens / mask [n][T]) into cache rows `rows`."""
        n, T = tokens.shape
        r = (C.c_int32 * n)(*[int(v) for v in rows])
        if out_tokens is None:
            out_tokens = torch.empty(n, dtype=torch.int32, device=self.device)
        check(lib().bloom_kv_admit(self.h, C.byref(kv.c), r, n, _p(tokens), _p(mask), T,
                                   _p(out_tokens), _p(logits), _stream(stream)))
        return out_tokens

    def kv_retire(self, kv: KV, rows, stream=None):
        """Rows `rows` leave the batch (decode steps skip them)."""
        r = (C.c_int32 * len(rows))(*[int(v) for v in rows])
        check(lib().bloom_kv_retire(self.h, C.byref(kv.c), r, len(rows), _stream(stream)))

    def generate(self, kv: KV, tokens_host, mask_host, n_new: int, out_host=None, stream=None):
        """Greedy generation from host buffers; returns host int32 [n_new, B]."""
        B, T = tokens_host.shape
        if out_host is None:
            out_host = torch.empty(n_new, B, dtype=torch.int32)
        check(lib().bloom_generate(self.h, C.byref(kv.c), _p(tokens_host), _p(mask_host), B, T,
                                   n_new, _p(out_host), _stream(stream)))
        return out_host

    def decode_profile(self, kv: KV, next_tokens, out_tokens=None, cap: int = 4096, stream=None):
        """One decode step launched kernel by kernel with an event after each;
        returns [(op, kernel, ms)] in launch order (names in OPS / KERNELS)."""
        if out_tokens is None:
            out_tokens = torch.empty(kv.batch, dtype=torch.int32, device=self.device)
        codes = (C.c_int32 * cap)()
        ms = (C.c_float * cap)()
        n = C.c_int32(0)
        check(lib().bloom_decode_profile(self.h, C.byref(kv.c), _p(next_tokens), _p(out_tokens),
                                         codes, ms, cap, C.byref(n), _stream(stream)))
        return [(OPS[codes[i] & 0xff], KERNELS[codes[i] >> 8], float(ms[i]))
                for i in range(n.value)]

    def check_device(self, stream=None):
        check(lib().bloom_check_device(self.h, _stream(stream)))

    def layer_decode(self, kv: KV, layer: int, x, stream=None):
        check(lib().bloom_layer_decode(self.h, C.byref(kv.c), layer, _p(x), _stream(stream)))

    def kv_set_prompt(self, kv: KV, mask, stream=None):
        B, T = mask.shape
        check(lib().bloom_kv_set_prompt(self.h, C.byref(kv.c), _p(mask), B, T, _stream(stream)))

    def layer_prefill(self, kv: KV, layer: int, x, B: int, T: int, stream=None):
        check(lib().bloom_layer_prefill(self.h, C.byref(kv.c), layer, _p(x), B, T,
                                        _stream(stream)))

    def head(self, x, out_tokens=None, logits=None, stream=None):
        B = x.shape[0]
        if out_tokens is None:
            out_tokens = torch.empty(B, dtype=torch.int32, device=self.device)
        check(lib().bloom_head(self.h, _p(x), B, _p(out_tokens), _p(logits), _stream(stream)))
        return out_tokens

    def lm_head(self, xn, out_tokens, logits=None, stream=None):
        """The tied head + argmax kernel alone on normalised rows xn [B, h]."""
        check(lib().bloom_lm_head(self.h, _p(xn), xn.shape[0], _p(out_tokens), _p(logits),
                                  _stream(stream)))
        return out_tokens

    def embed(self, tokens, x=None, stream=None):
        n = tokens.numel()
        if x is None:
            x = torch.empty(n, self.shape.hidden, dtype=torch.float32, device=self.device)
        check(lib().bloom_embed(self.h, _p(tokens), n, _p(x), _stream(stream)))
        return x


# ----------------------------------------------------------------- operators
def op_layernorm(x, g=None, b=None, eps=1e-5, y=None, stream=None):
    rows, h = x.shape
    if y is None:
        y = torch.empty_like(x)
    check(lib().bloom_op_layernorm(_p(x), _p(g), _p(b), rows, h, eps, _p(y), _stream(stream)))
    return y


def op_linear(x, w=None, bias=None, q=None, scale=None, epilogue=EPI_STORE, y=None,
              stream=None):
    M, K = x.shape
    N = (w if w is not None else q).shape[0]
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    lin = Linear(_p(w if w is not None else q), _p(scale), _p(bias))
    check(lib().bloom_op_linear(C.byref(lin), 0 if w is not None else 1, _p(x), M, N, K,
                                epilogue, _p(y), _stream(stream)))
    return y


def op_gemm(x, w, bias=None, epilogue=EPI_STORE, y=None, stream=None):
    """bf16 linear layer on the tensor-core (tcgen05) GEMM used by prefill."""
    M, K = x.shape
    N = w.shape[0]
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    lin = Linear(_p(w), None, _p(bias))
    check(lib().bloom_op_gemm(C.byref(lin), _p(x), M, N, K, epilogue, _p(y), _stream(stream)))
    return y


def op_linear_tc(x, w=None, bias=None, q=None, scale=None, epilogue=EPI_STORE, y=None,
                 stream=None):
    """Linear layer on the tensor-core decode kernel: bf16 weights w (M <= 256
    tokens) or int8 codes q with bf16 row scales (M <= 128)."""
    M, K = x.shape
    N = (w if w is not None else q).shape[0]
    if y is None:
        y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    lin = Linear(_p(w if w is not None else q), _p(scale), _p(bias))
    check(lib().bloom_op_linear_tc(C.byref(lin), 0 if w is not None else 1, _p(x), M, N, K,
                                   epilogue, _p(y), _stream(stream)))
    return y


def op_attn_decode(q, k_cache, v_cache, pos, slopes, length: int, splits: int = 0, o=None,
                   stream=None):
    B, n, S, d = k_cache.shape
    if o is None:
        o = torch.empty(B, n * d, dtype=torch.bfloat16, device=q.device)
    check(lib().bloom_op_attn_decode(_p(q), _p(k_cache), _p(v_cache), _p(pos), _p(slopes), B, n,
                                     d, S, length, splits, _p(o), _stream(stream)))
    return o


def op_lmhead_argmax(x, emb, logits: bool = True, stream=None):
    M, K = x.shape
    V = emb.shape[0]
    tok = torch.empty(M, dtype=torch.int32, device=x.device)
    lg = torch.empty(M, V, dtype=torch.float32, device=x.device) if logits else None
    check(lib().bloom_op_lmhead_argmax(_p(x), _p(emb), M, V, K, _p(tok), _p(lg),
                                       _stream(stream)))
    return tok, lg


def op_sample(logits, temperature, top_p, u, out=None, stream=None):
    """Temperature + top-p sampling of float32 logits [B][V] (rows may be
    strided) with per-row device float32 [B] temperature, top_p, u."""
    B, V = logits.shape
    if out is None:
        out = torch.empty(B, dtype=torch.int32, device=logits.device)
    check(lib().bloom_op_sample(_p(logits), B, V, logits.stride(0), _p(temperature), _p(top_p),
                                _p(u), _p(out), _stream(stream)))
    return out


def op_lmhead_argmax_noalloc(x, emb, logits: bool = True, stream=None):
    """bloom_op_lmhead_argmax without allocation (fixed in-library scratch)."""
    M, K = x.shape
    V = emb.shape[0]
    tok = torch.empty(M, dtype=torch.int32, device=x.device)
    lg = torch.empty(M, V, dtype=torch.float32, device=x.device) if logits else None
    check(lib().bloom_op_lmhead_argmax_noalloc(_p(x), _p(emb), M, V, K, _p(tok), _p(lg),
                                               _stream(stream)))
    return tok, lg
