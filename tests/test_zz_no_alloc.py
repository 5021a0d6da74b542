"""dec_prefill_kv_noalloc (token-mode prefill staged in the library's static device scratch)
against dec_prefill_kv (the same prefill with a cudaMalloc'd staging buffer), on two engines
built from the same seeded weights. Kept in its own file, collected last, so it runs both alone
in a fresh process and after every other test has used the library.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from latency_moe_decode_gb300 import capi, synth

pytestmark = pytest.mark.gpu

CFG = synth.ModelCfg(n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, n_experts=8, top_k=2,
                     moe_inter=128, n_shared=1, vocab=512, max_ctx=128, max_batch=4)
MAX_IDS = 65536  # DEC_NOALLOC_PREFILL_MAX_IDS in include/dec.h
DEC_ERR_ARG = -1


def _pair():
    from latency_moe_decode_gb300.engine import Engine
    m = synth.model_to(synth.gen_model(CFG, seed=31, device="cpu"), "cuda")
    return Engine(m), Engine(m)


def _kv(eng, seq, n):
    return [tuple(t.float().cpu().numpy() for t in eng.export_kv(seq, l, 0, n)) for l in range(CFG.n_layers)]


def _step(eng, tok, seq0=0):
    b = tok.shape[0]
    logits = torch.empty(b, CFG.vocab, device="cuda")
    nxt = torch.empty(b, dtype=torch.int32, device="cuda")
    eng.step(tokens=tok, batch=b, seq0=seq0, logits=logits, next_tokens=nxt)
    eng.sync()
    return logits.cpu().numpy(), nxt.cpu().numpy()


@pytest.mark.parametrize("seq0,n_seq", [(0, 3), (1, 2)], ids=["slots0-2", "slots1-2"])
def test_noalloc_prefill_matches_allocating_prefill_on_two_calls(seq0, n_seq):
    """Both engines run the same deterministic kernels on the same ids, so the KV caches, logits
    and tokens must agree bit for bit; the second case starts at slot 1 and leaves a slot free."""
    ref, na = _pair()
    g = torch.Generator().manual_seed(5 + seq0)
    filled = 0
    for n_tok in (7, 5):  # two calls in a row, the second appending to the first
        ids = torch.randint(0, CFG.vocab, (n_seq, n_tok), generator=g, dtype=torch.int32).cuda()
        ref.prefill_tokens(ids, seq=seq0)
        na.prefill_tokens_noalloc(ids, seq=seq0)
        filled += n_tok
        for s in range(seq0, seq0 + n_seq):
            assert na.get_length(s) == ref.get_length(s) == filled
            for (kr, vr), (kn, vn) in zip(_kv(ref, s, filled), _kv(na, s, filled)):
                assert np.array_equal(kn, kr) and np.array_equal(vn, vr)
        for s in set(range(CFG.max_batch)) - set(range(seq0, seq0 + n_seq)):
            assert na.get_length(s) == ref.get_length(s) == 0
        tok = torch.randint(0, CFG.vocab, (n_seq,), generator=g, dtype=torch.int32).cuda()
        lr, tr = _step(ref, tok, seq0)
        ln, tn = _step(na, tok, seq0)
        filled += 1
        assert np.isfinite(ln).all()
        assert np.array_equal(ln, lr) and np.array_equal(tn, tr)
    ref.close()
    na.close()


def test_noalloc_prefill_rejects_oversize_and_import_mode():
    from latency_moe_decode_gb300.engine import Engine
    m = synth.model_to(synth.gen_model(CFG, seed=32, device="cpu"), "cuda")
    eng = Engine(m)
    # two slots of MAX_IDS / 2 + 1 ids each: one id over the scratch; refused before any work
    ids = torch.zeros(2, MAX_IDS // 2 + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(capi.DecError) as ei:
        eng.prefill_tokens_noalloc(ids)
    assert ei.value.status == DEC_ERR_ARG and "static scratch" in str(ei.value)
    assert eng.get_length(0) == 0 and eng.get_length(1) == 0
    k = torch.zeros(CFG.n_layers, CFG.n_kv_heads, 4, CFG.head_dim, dtype=torch.bfloat16, device="cuda")
    ctx = capi.DecCtx(0, 1, None, 4, k.data_ptr(), k.data_ptr())
    assert eng.lib.dec_prefill_kv_noalloc(eng.h, C.byref(ctx)) == DEC_ERR_ARG
    # the engine stays usable
    eng.prefill_tokens_noalloc(torch.arange(6, dtype=torch.int32, device="cuda")[None])
    assert eng.get_length(0) == 6
    eng.close()
