"""Resident generation: dec_generate runs all its decode steps in one launch (each step's argmax
fed to the next step on the device), and must decode exactly like one launch per step: same
kernel arithmetic, so the tokens agree bit for bit. ("Ultra-High Interactivity on NVIDIA GPUs?
TileRT on InferenceX", section "But What Exactly is TileRT?": the host launches once.)"""
import numpy as np
import pytest
import torch

from latency_moe_decode_gb300 import synth

pytestmark = pytest.mark.gpu

TINY_MOE = synth.ModelCfg(n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, n_experts=8, top_k=2,
                          moe_inter=128, n_shared=1, vocab=512, max_ctx=96, max_batch=4)
SMALL_MOE = synth.ModelCfg(n_layers=2, hidden=512, n_heads=8, n_kv_heads=2, head_dim=128, n_experts=16, top_k=4,
                           moe_inter=256, n_shared=1, vocab=2048, max_ctx=96, max_batch=4, rope_theta=1e6)


def _per_step(eng, first, n):
    """Reference: one launch per step, chained on the device."""
    b = len(first)
    toks = torch.zeros(n + 1, b, dtype=torch.int32, device="cuda")
    toks[0] = torch.tensor(first, dtype=torch.int32, device="cuda")
    for i in range(n):
        eng.step(tokens=toks[i], batch=b, next_tokens=toks[i + 1])
    eng.sync()
    return toks[1:].cpu().numpy()


@pytest.mark.parametrize("cfg,first", [(synth.TINY.replace(max_ctx=96), [5]), (TINY_MOE, [3, 9]),
                                       (SMALL_MOE, [7, 1, 400])], ids=["dense_b1", "moe_b2", "moe_tc_b3"])
def test_resident_generation_equals_one_launch_per_step(cfg, first):
    from latency_moe_decode_gb300.engine import Engine
    m = synth.model_to(synth.gen_model(cfg, seed=61, device="cpu"), "cuda")
    prompt = torch.stack([synth.gen_tokens(20, cfg.vocab, seed=s) for s in range(len(first))]).cuda()
    a, b = Engine(m), Engine(m)
    for e in (a, b):
        for s in range(len(first)):
            e.prefill_tokens(prompt[s:s + 1], seq=s)
    n = 24
    ref = _per_step(a, first, n)
    l0 = b.info()["launches"]
    got = b.generate(first, n)
    assert b.info()["launches"] - l0 == 1  # one launch for the whole generation
    assert np.array_equal(got, ref)
    for s in range(len(first)):
        assert a.get_length(s) == b.get_length(s) == 20 + n
    # the device-buffer form continues from there, again in one launch
    out = torch.zeros(8, len(first), dtype=torch.int32, device="cuda")
    b.generate_device(torch.tensor(got[-1], dtype=torch.int32, device="cuda"), out)
    b.sync()
    assert np.array_equal(out.cpu().numpy(), _per_step(a, list(got[-1]), 8))
    a.close()
    b.close()


def test_resident_generation_across_epoch_restarts(monkeypatch):
    """With the epoch period lowered to 3 steps, a 10-step generation takes four launches (3+3+3+1),
    the counters restarting before each, and still decodes like an engine that never restarts."""
    from latency_moe_decode_gb300.engine import Engine
    m = synth.model_to(synth.gen_model(TINY_MOE, seed=62, device="cpu"), "cuda")
    ref = Engine(m)
    monkeypatch.setenv("DEC_EPOCH_LIMIT", "3")
    short = Engine(m)
    monkeypatch.delenv("DEC_EPOCH_LIMIT")
    first = [11, 22]
    l0 = short.info()["launches"]
    got = short.generate(first, 10)
    assert short.info()["launches"] - l0 == 4
    assert np.array_equal(got, ref.generate(first, 10))
    ref.close()
    short.close()


def test_resident_generation_capacity():
    from latency_moe_decode_gb300.capi import DecError
    from latency_moe_decode_gb300.engine import Engine
    m = synth.model_to(synth.gen_model(TINY_MOE, seed=63, device="cpu"), "cuda")
    eng = Engine(m)
    eng.set_length(0, TINY_MOE.max_ctx - 5)
    with pytest.raises(DecError) as e:
        eng.generate([1], 6)
    assert e.value.status == -8
    got = eng.generate([1], 5)  # exactly fills the slot
    assert got.shape == (5, 1) and eng.get_length(0) == TINY_MOE.max_ctx
    eng.close()
