"""Host-side checks of the C ABI library (no GPU needed): it loads, exports every entry point
that include/dec.h declares, and validates model shapes on the host."""
import ctypes as C
import os
import re

import pytest

from latency_moe_decode_gb300 import build, capi, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return capi.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dec.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dec_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("dec_init", "dec_prefill_kv", "dec_step", "dec_destroy", "dec_last_error"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(capi.PROTOTYPES)


def test_status_strings(lib):
    for code in capi.STATUS:
        assert lib.dec_status_string(code)


def _cfg(**kw):
    c = synth.MOE8.replace(**kw)
    return capi.DecModelCfg(c.n_layers, c.hidden, c.n_heads, c.n_kv_heads, c.head_dim, c.n_experts, c.top_k,
                            c.moe_inter, c.n_shared, c.dense_ffn, c.vocab, c.max_ctx, c.max_batch, c.rms_eps,
                            c.rope_theta)


def test_validate_cfg(lib):
    v = lambda **kw: lib.dec_validate_cfg(C.byref(_cfg(**kw)))
    assert v() == 0
    assert lib.dec_validate_cfg(C.byref(capi.DecModelCfg(*[getattr(synth.TINY, f) for f, _ in capi.DecModelCfg._fields_]))) == 0
    assert v(n_heads=30) == -1                 # heads not a multiple of KV heads
    assert v(dense_ffn=512) == -1              # both FFN kinds
    assert v(top_k=65) == -1                   # top_k > n_experts
    assert v(n_layers=0) == -1
    assert v(head_dim=96) == -5                # not implemented
    assert v(hidden=4000) == -5
    assert v(max_batch=9) == 0                 # 9 .. 64: the wide kernels
    assert v(max_batch=64) == 0
    assert v(max_batch=65) == -5
    assert v(max_batch=16, n_experts=64, top_k=9) == -5  # the wide kernel: at most 8 experts per token
    assert v(max_batch=8, n_experts=64, top_k=9) == 0     # (8 sequences: decode_step_kernel instead)
    assert v(hidden=8192) == -5             # above the hidden sizes the kernel handles
    assert v(n_shared=2) == -5
    assert v(n_experts=200, top_k=8) == -5


def test_null_arguments_are_rejected(lib):
    out = C.c_void_p()
    assert lib.dec_init(None, None, None, C.byref(out)) == -1
    assert lib.dec_step(None, None, 1, None, None, None) == -1
    assert lib.dec_sync(None) == -1
    lib.dec_destroy(None)
