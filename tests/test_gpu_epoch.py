"""The engine's cross-step counters and flags restart from zero every DEC_EPOCH_LIMIT steps (a
stream-ordered memset before the step). An engine made to restart every three steps must decode
exactly as one that never restarts in the test: same kernel, same arithmetic, so the logits and
tokens agree bit for bit."""
import numpy as np
import pytest
import torch

from latency_moe_decode_gb300 import synth

pytestmark = pytest.mark.gpu

CFG = synth.ModelCfg(n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, n_experts=8, top_k=2,
                     moe_inter=128, n_shared=1, vocab=512, max_ctx=64, max_batch=2)


def _run(eng, steps):
    out = []
    tok = torch.tensor([3, 7], dtype=torch.int32, device="cuda")
    for _ in range(steps):
        logits = torch.empty(2, CFG.vocab, device="cuda")
        nxt = torch.empty(2, dtype=torch.int32, device="cuda")
        eng.step(tokens=tok, batch=2, logits=logits, next_tokens=nxt)
        eng.sync()
        out.append((logits.cpu().numpy(), nxt.cpu().numpy()))
        tok = nxt
    return out


def test_epoch_restart_is_invisible(monkeypatch):
    from latency_moe_decode_gb300.engine import Engine
    m = synth.model_to(synth.gen_model(CFG, seed=41, device="cpu"), "cuda")
    ref = Engine(m)
    monkeypatch.setenv("DEC_EPOCH_LIMIT", "3")
    short = Engine(m)
    monkeypatch.delenv("DEC_EPOCH_LIMIT")
    a, b = _run(ref, 10), _run(short, 10)
    for (la, ta), (lb, tb) in zip(a, b):
        assert np.array_equal(la, lb) and np.array_equal(ta, tb)
    ref.close()
    short.close()
