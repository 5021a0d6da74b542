"""GPU parity of the wide kernel (decode steps of 9 .. 64 sequences: every GEMV on the tensor cores
with the step's tokens as N, tokens grouped per routed expert) against the CPU oracle, through
the C ABI. Each sequence has its own seeded KV history and is compared with the oracle's decode
of that sequence alone.
"""
import numpy as np
import pytest
import torch

import oracle
from latency_moe_decode_gb300 import synth
from tests.parity import GATE_ABS, StepCheck, bf16_to_f64, near_tie, rel_l2, t_bits, topk_ok
from tests.test_gpu_parity import MOE_SMALL, _engine, _gpu_step, _models, _one_layer

pytestmark = pytest.mark.gpu

MOE_WIDE = MOE_SMALL.replace(max_batch=64, max_ctx=320)
TINY_WIDE = synth.TINY.replace(max_batch=24, max_ctx=96)


@pytest.fixture(scope="module")
def moe_wide():
    return _models(MOE_WIDE, 3)


def _ragged(batch, base=5, step=37, mod=250):
    return [base + (step * b) % mod for b in range(batch)]


@pytest.mark.parametrize("batch", [9, 16, 24, 33, 64])
def test_wide_moe_small_batch_ragged(moe_wide, batch):
    """One step of `batch` sequences with ragged lengths (1 .. 4 KV tiles, several sequences
    sharing an expert, slots beyond 8): logits, argmax, final hidden state, routing and lengths of
    every sequence against the oracle."""
    m_cpu, m_gpu = moe_wide
    cfg = MOE_WIDE
    orc = oracle.Oracle(m_cpu)
    eng = _engine(m_gpu)
    lens = _ragged(batch)
    toks = synth.gen_tokens(batch, cfg.vocab, seed=50 + batch).tolist()
    kvs = []
    for b in range(batch):
        k, v = synth.gen_kv(cfg, lens[b], seed=300 + b)
        eng.prefill_import(k.cuda(), v.cuda(), seq=b)
        kv = orc.new_kv(cfg.max_ctx)
        orc.import_kv(kv, k, v, lens[b])
        kvs.append(kv)
    g_logits, g_next, g_hidden = _gpu_step(eng, tok=toks, batch=batch)
    chk = StepCheck()
    routes = [eng.routing(l) for l in range(cfg.n_layers)]
    for b in range(batch):
        o = orc.decode_step(kvs[b], lens[b], token=toks[b], want_trace=True)
        chk.add(g_logits[b], o["logits"], g_next[b], o["token"], g_hidden[b], o["hidden"])
        for l in range(cfg.n_layers):
            gi, gg = routes[l]
            assert topk_ok(gi[b], o["trace"]["topk_idx"][l], o["trace"]["router_score"][l], cfg.top_k)
            if set(gi[b]) == set(o["trace"]["topk_idx"][l]):
                assert np.allclose(gg[b], o["trace"]["topk_gate"][l], atol=GATE_ABS)
                assert abs(gg[b].sum() - 1) < 1e-5
        assert eng.get_length(b) == lens[b] + 1
    chk.assert_ok()


def test_wide_moe_small_slot_offset_and_rerun(moe_wide):
    """A wide step at slot offset 7 (slots 7 .. 22) matches the oracle, and repeating the same
    step from the same state gives bit-identical results (deterministic split-K order)."""
    m_cpu, m_gpu = moe_wide
    cfg = MOE_WIDE
    B, seq0 = 16, 7
    orc = oracle.Oracle(m_cpu)
    eng = _engine(m_gpu)
    lens = _ragged(B, base=60, step=13, mod=200)
    toks = synth.gen_tokens(B, cfg.vocab, seed=77).tolist()
    kvs = []
    for b in range(B):
        k, v = synth.gen_kv(cfg, lens[b], seed=700 + b)
        eng.prefill_import(k.cuda(), v.cuda(), seq=seq0 + b)
        kv = orc.new_kv(cfg.max_ctx)
        orc.import_kv(kv, k, v, lens[b])
        kvs.append(kv)
    a = _gpu_step(eng, tok=toks, batch=B, seq0=seq0)
    for b in range(B):
        eng.set_length(seq0 + b, lens[b])
    r = _gpu_step(eng, tok=toks, batch=B, seq0=seq0)
    assert np.array_equal(a[0], r[0]) and np.array_equal(a[1], r[1]) and np.array_equal(a[2], r[2])
    chk = StepCheck()
    for b in range(B):
        o = orc.decode_step(kvs[b], lens[b], token=toks[b])
        chk.add(a[0][b], o["logits"], a[1][b], o["token"], a[2][b], o["hidden"])
        assert eng.get_length(seq0 + b) == lens[b] + 1
    chk.assert_ok()


def test_wide_tiny_dense_prefill_and_generate():
    """The tiny dense decoder (head_dim 64, 2 query heads per KV head, dense SwiGLU FFN) with 24
    sequences: token-mode prefill of 24 slots side by side (one wide launch per position), then
    greedy generation (one wide launch per step, tokens chained on the device); every sequence's
    tokens against the oracle's greedy decode."""
    cfg = TINY_WIDE
    m_cpu, m_gpu = _models(cfg, 0)
    B, n_prompt, n_gen = 24, 20, 10
    prompts = synth.gen_tokens(B * n_prompt, cfg.vocab, seed=11).reshape(B, n_prompt)
    eng = _engine(m_gpu)
    eng.prefill_tokens(prompts.cuda())
    orc = oracle.Oracle(m_cpu)
    firsts, want = [], []
    for b in range(B):
        kv = orc.new_kv(cfg.max_ctx)
        o = orc.prefill(kv, prompts[b])
        tok = o["token"]
        firsts.append(tok)
        seq = []
        ties = 0
        for i in range(n_gen):
            o = orc.decode_step(kv, n_prompt + i, token=tok)
            ties += near_tie(o["logits"])
            tok = o["token"]
            seq.append(tok)
        want.append((seq, ties))
    for b in range(B):
        assert eng.get_length(b) == n_prompt
    got = eng.generate(firsts, n_gen)
    for b in range(B):
        seq, ties = want[b]
        if ties == 0:
            assert got[:, b].tolist() == seq, (b, got[:, b].tolist(), seq)
        assert eng.get_length(b) == n_prompt + n_gen


@pytest.mark.parametrize("batch", [16, 64])
def test_wide_moe_layer_full_size(batch):
    """One full-size MoE layer (hidden 4096, 64 experts, top-8, shared expert) at batch 16 and 64
    (at 64 nearly every expert is streamed, each for its own tokens), hidden input, each sequence
    with its own ragged KV history: final hidden state and routing against the oracle."""
    m_gpu = synth.gen_model(synth.MOE8.replace(n_layers=1), seed=0, device="cuda")
    m_cpu = synth.model_to(m_gpu, "cpu")
    cfg = synth.MOE_LAYER
    lens = [96 + (41 * b) % 160 for b in range(batch)]
    orc = oracle.Oracle(_one_layer(m_cpu))
    eng = _engine(_one_layer(m_gpu), max_ctx=320, max_batch=batch)
    x = synth.gen_hidden(batch, cfg.hidden, seed=21, device="cuda")
    outs = []
    for b in range(batch):
        k, v = synth.gen_kv(cfg, lens[b], seed=900 + b, device="cuda")
        eng.prefill_import(k, v, seq=b)
        kv = orc.new_kv(320)
        orc.import_kv(kv, k.cpu(), v.cpu(), lens[b])
        outs.append(orc.decode_step(kv, lens[b], hidden=t_bits(x)[b], want_trace=True))
    _, _, g_hidden = _gpu_step(eng, hidden=x, batch=batch)
    gi, gg = eng.routing(0)
    distinct = len(set(gi[:batch].reshape(-1).tolist()))
    assert distinct >= (40 if batch == 64 else 30)
    compared = 0
    for b, o in enumerate(outs):
        assert topk_ok(gi[b], o["trace"]["topk_idx"][0], o["trace"]["router_score"][0], 8)
        assert abs(gg[b].sum() - 1) < 1e-5
        if set(gi[b]) == set(o["trace"]["topk_idx"][0]):
            assert rel_l2(bf16_to_f64(g_hidden[b]), bf16_to_f64(o["hidden"])) <= 1e-2
            compared += 1
        assert eng.get_length(b) == lens[b] + 1
    assert compared >= batch - 2
