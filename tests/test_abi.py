"""The C-ABI library loads, exports every declared entry point, and validates
its arguments on the host (no GPU needed, no compute launched)."""
import ctypes as C
import os
import re

import pytest
import torch

import bloom_decoder_token_gb300 as bg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return bg.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "bloom.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bloom_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), n
    # the binding wraps exactly the declared set
    assert sorted(bg.EXPORTS) == names


def test_no_oracle_symbols_in_product_library(lib):
    out = os.popen(f"nm -D {bg.LIB_PATH}").read()
    assert "orc_" not in out
    assert "bloom_create" in out


def _cfg(**kw):
    base = dict(n_layer=2, hidden=1024, n_head=16, ffn=4096, vocab=512, ln_eps=1e-5,
                weight_dtype=0, max_batch=4, max_tokens=64, max_seq=40, flags=0, wait_us=0)
    base.update(kw)
    return bg.Config(*[base[f] for f, _ in bg.Config._fields_])


def test_kv_bytes_layout(lib):
    c = _cfg()
    n = lib.bloom_kv_bytes(C.byref(c), 3, 40)
    # header + len + active + next_pos + pos + K + V, each 256-aligned
    al = lambda x: (x + 255) // 256 * 256
    kv = 2 * 3 * 16 * 40 * 64 * 2          # layers * B * n * S * d * 2 bytes
    off = al(256 + 4 * 3)                  # len
    off = al(off + 4 * 3)                  # active
    off = al(off + 4 * 3)                  # next_pos
    off = al(off + 4 * 3 * 40)             # pos
    assert n == al(al(off + kv) + kv)
    assert lib.bloom_kv_bytes(C.byref(c), 0, 40) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(n_head=3), 1),            # hidden % n_head
    (dict(n_head=4), 2),            # head_dim 256 unsupported
    (dict(max_batch=0), 2),
    (dict(max_batch=300), 2),
    (dict(ln_eps=0.0), 1),
    (dict(weight_dtype=7), 1),
    (dict(max_tokens=1), 1),
    (dict(ffn=1000), 2),
    (dict(wait_us=-1), 1),
])
def test_create_rejects_bad_config(lib, kw, status):
    c = _cfg(**kw)
    h = C.c_void_p()
    w = bg.WeightsC()
    st = lib.bloom_create(C.byref(c), C.byref(w), C.byref(h))
    assert st == status, lib.bloom_last_error()
    assert not h.value
    assert lib.bloom_last_error()


def test_create_rejects_null_and_misaligned_weights(lib):
    c = _cfg(n_layer=1)
    h = C.c_void_p()
    w = bg.WeightsC()
    assert lib.bloom_create(C.byref(c), C.byref(w), C.byref(h)) == 1
    arr = (bg.LayerWeights * 1)()
    fake = 0x10000
    arr[0] = bg.LayerWeights(fake, fake, bg.Linear(fake + 2, None, None), bg.Linear(fake, None, None),
                             fake, fake, bg.Linear(fake, None, None), bg.Linear(fake, None, None))
    w = bg.WeightsC(fake, fake, fake, fake, fake, C.cast(arr, C.POINTER(bg.LayerWeights)))
    assert lib.bloom_create(C.byref(c), C.byref(w), C.byref(h)) == 1
    assert "aligned" in lib.bloom_last_error().decode()
    # int8 config with bf16-style pointers (no scales) is rejected before any CUDA call
    c8 = _cfg(n_layer=1, weight_dtype=1)
    arr[0] = bg.LayerWeights(fake, fake, bg.Linear(fake, None, None), bg.Linear(fake, None, None),
                             fake, fake, bg.Linear(fake, None, None), bg.Linear(fake, None, None))
    assert lib.bloom_create(C.byref(c8), C.byref(w), C.byref(h)) == 1
    assert "scales" in lib.bloom_last_error().decode()


def test_ops_reject_bad_arguments(lib):
    assert lib.bloom_op_layernorm(None, None, None, 1, 64, 1e-5, None, None) == 1
    assert lib.bloom_op_layernorm(C.c_void_p(16), None, None, 1, 20, 1e-5, C.c_void_p(16), None) == 2
    assert lib.bloom_op_attn_decode(C.c_void_p(16), C.c_void_p(16), C.c_void_p(16), C.c_void_p(16),
                                    C.c_void_p(16), 1, 1, 96, 8, 0, 0, C.c_void_p(16), None) == 2
    # K / V read 16 bytes at a time and by bulk copies: a misaligned cache is rejected
    # on the host, before any device call
    assert lib.bloom_op_attn_decode(C.c_void_p(16), C.c_void_p(24), C.c_void_p(16), C.c_void_p(16),
                                    C.c_void_p(16), 1, 1, 128, 8, 0, 0, C.c_void_p(16), None) == 1
    assert lib.bloom_op_attn_decode(C.c_void_p(16), C.c_void_p(16), C.c_void_p(16), C.c_void_p(16),
                                    C.c_void_p(16), 1, 1, 128, 8, 0, 0, C.c_void_p(18), None) == 1
    assert lib.bloom_op_lmhead_argmax(C.c_void_p(16), C.c_void_p(16), 0, 8, 8, C.c_void_p(16),
                                      None, None) == 2
    lin = bg.Linear(C.c_void_p(16), None, None)
    assert lib.bloom_op_linear(C.byref(lin), 0, C.c_void_p(16), 1, 4, 12, 0, C.c_void_p(16), None) == 2
    assert lib.bloom_op_linear(C.byref(lin), 0, C.c_void_p(16), 1, 4, 16, 9, C.c_void_p(16), None) == 1
    lin8 = bg.Linear(C.c_void_p(16), C.c_void_p(16), None)
    assert lib.bloom_op_linear_tc(C.byref(lin8), 1, C.c_void_p(16), 129, 128, 64, 0,
                                  C.c_void_p(16), None) == 4      # int8: at most 128 tokens
    assert lib.bloom_op_linear_tc(C.byref(lin8), 1, C.c_void_p(16), 8, 128, 72, 0,
                                  C.c_void_p(16), None) == 2      # int8 rows in 16-byte chunks
    assert lib.bloom_decode_step(None, None, None, None, None, None) == 1
    assert lib.bloom_destroy(None) == 0


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(bg, "_lib", None)
    monkeypatch.setattr(bg, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        bg.lib()
