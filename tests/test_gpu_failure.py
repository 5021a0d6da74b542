"""The failure path of the decode step, made to happen without faulting the GPU.

* A wait that runs out: the engine is built with DEC_TEST_SKIP_ARRIVAL=1, so the CTA holding
  the first q/k/v tile withholds that partial sum's arrival in layer 0 (a counter that nothing
  completes; in a step of 5 tokens or more, the wide kernel, CTA 0 withholds its arrival at
  the first grid barrier), and with
  DEC_TIMEOUT_MS=20 every wait of the step is bounded by 20 ms. The step must end by itself, the
  next synchronising call must report DEC_ERR_TIMEOUT and poison the engine (later calls give
  DEC_ERR_POISONED), and the CUDA context must stay usable: a fresh engine on the same device
  then decodes exactly like one that never failed.
* A device-side bounds check: a token id beyond the vocabulary (device memory, so the host cannot
  see it) is reported by the kernel (DEC_ERR_DEVICE) instead of reading outside the embedding.
"""
import numpy as np
import pytest
import torch

from latency_moe_decode_gb300 import capi, synth

pytestmark = pytest.mark.gpu

CFG = synth.ModelCfg(n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, n_experts=8, top_k=2,
                     moe_inter=128, n_shared=1, vocab=512, max_ctx=64, max_batch=16)
BATCHES = [2, 16]  # the batch-1..8 kernel (tensor-core tiles) and the wide kernel
DEC_ERR_TIMEOUT, DEC_ERR_POISONED, DEC_ERR_DEVICE = -4, -6, -7


def _model(seed):
    return synth.model_to(synth.gen_model(CFG, seed=seed, device="cpu"), "cuda")


def _tokens(batch):
    return torch.tensor([(5 + 4 * b) % CFG.vocab for b in range(batch)], dtype=torch.int32, device="cuda")


def _decode(eng, batch, steps=3):
    out = []
    tok = _tokens(batch)
    for _ in range(steps):
        logits = torch.empty(batch, CFG.vocab, device="cuda")
        nxt = torch.empty(batch, dtype=torch.int32, device="cuda")
        eng.step(tokens=tok, batch=batch, logits=logits, next_tokens=nxt)
        eng.sync()
        out.append((logits.cpu().numpy(), nxt.cpu().numpy()))
        tok = nxt
    return out


@pytest.mark.parametrize("batch", BATCHES)
def test_withheld_arrival_times_out_and_poisons(monkeypatch, batch):
    from latency_moe_decode_gb300.engine import Engine
    m = _model(51)
    monkeypatch.setenv("DEC_TEST_SKIP_ARRIVAL", "1")
    monkeypatch.setenv("DEC_TIMEOUT_MS", "20")
    bad = Engine(m)
    monkeypatch.delenv("DEC_TEST_SKIP_ARRIVAL")
    monkeypatch.delenv("DEC_TIMEOUT_MS")
    tok = _tokens(batch)
    bad.step(tokens=tok, batch=batch)  # the launch itself succeeds; the device wait runs out
    with pytest.raises(capi.DecError) as ei:
        bad.sync()
    assert ei.value.status == DEC_ERR_TIMEOUT, str(ei.value)
    assert "timed out" in str(ei.value)
    with pytest.raises(capi.DecError) as ei:
        bad.step(tokens=tok, batch=batch)
    assert ei.value.status == DEC_ERR_POISONED
    bad.close()
    # the context is intact: two fresh engines decode, bit for bit alike
    a, b = Engine(m), Engine(m)
    ra, rb = _decode(a, batch), _decode(b, batch)
    for (la, ta), (lb, tb) in zip(ra, rb):
        assert np.isfinite(la).all() and np.array_equal(la, lb) and np.array_equal(ta, tb)
    a.close()
    b.close()


@pytest.mark.parametrize("batch", BATCHES)
def test_token_id_bounds_are_checked(batch):
    from latency_moe_decode_gb300.engine import Engine
    eng = Engine(_model(52))
    tok = _tokens(batch)
    tok[batch - 1] = CFG.vocab + 3
    eng.step(tokens=tok, batch=batch)
    with pytest.raises(capi.DecError) as ei:
        eng.sync()
    assert ei.value.status == DEC_ERR_DEVICE, str(ei.value)
    assert "device check failed" in str(ei.value)
    with pytest.raises(capi.DecError) as ei:
        eng.step(tokens=tok, batch=batch)
    assert ei.value.status == DEC_ERR_POISONED
    eng.close()
