"""GPU parity of the wide kernel (decode steps of 5 .. 64 sequences: every GEMV on the tensor cores
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


@pytest.mark.parametrize("batch", [5, 7, 8, 9, 16, 24, 33, 64])
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


def test_wide_moe8_every_layer_teacher_forced():
    """Every layer of the full-size 8-layer stack through the wide kernel, 16 sequences side by side
    (each with its own seeded KV history at context 512), for 2 consecutive tokens: each layer's
    engine is fed every sequence's oracle input to that layer and keeps its own KV cache; per
    sequence, the layer output and sublayer delta (rel L2 <= 1e-2), the new K/V rows, the gates and
    the routing (RouteCheck) against the oracle. Then the LM head, fed each sequence's oracle final
    hidden state: logits, argmax and hidden state."""
    from tests.parity import HIDDEN_REL_L2, RouteCheck
    from tests.test_gpu_parity import _bf16
    B, ctx, n_tok = 16, 512, 2
    m_gpu = synth.gen_model(synth.MOE8, seed=0, device="cuda")
    m_cpu = synth.model_to(m_gpu, "cpu")
    cfg8 = synth.MOE8.replace(max_ctx=ctx + n_tok + 16, max_batch=B)
    kvs = [synth.gen_kv(cfg8, ctx, seed=600 + b, device="cuda") for b in range(B)]
    orc = oracle.Oracle(m_cpu)
    outs, toks, okvs = [], [], []
    for b in range(B):
        kv = orc.new_kv(cfg8.max_ctx)
        orc.import_kv(kv, kvs[b][0].cpu(), kvs[b][1].cpu(), ctx)
        tok, ob, tb = 100 + 37 * b, [], []
        for i in range(n_tok):
            tb.append(tok)
            o = orc.decode_step(kv, ctx + i, token=tok, want_trace=True)
            ob.append(o)
            tok = o["token"]
        outs.append(ob)
        toks.append(tb)
        okvs.append(kv)
    cfg1 = synth.MOE_LAYER.replace(max_ctx=cfg8.max_ctx, max_batch=B)
    rc = RouteCheck()
    compared = 0
    for l in range(8):
        eng = _engine({"cfg": cfg1, "layers": [m_gpu["layers"][l]]}, max_ctx=cfg1.max_ctx, max_batch=B)
        for b in range(B):
            eng.prefill_import(kvs[b][0][l:l + 1].contiguous(), kvs[b][1][l:l + 1].contiguous(), seq=b)
        for i in range(n_tok):
            lay_in = [bf16_to_f64(t_bits(m_cpu["embed"][toks[b][i]])) if l == 0 else outs[b][i]["trace"]["layer_out"][l - 1]
                      for b in range(B)]
            _, _, g = _gpu_step(eng, hidden=_bf16(np.stack(lay_in)).cuda(), batch=B)
            gi, gg = eng.routing(0)
            lg = eng.router_logits(0)
            for b in range(B):
                o = outs[b][i]
                where = f"sequence {b} token {i} layer {l}"
                same = rc.check(gi[b], lg[b], o["trace"]["topk_idx"][l], o["trace"]["router_score"][l], 8, where)
                assert abs(gg[b].sum() - 1) < 1e-5
                kg, vg = eng.export_kv(b, 0, ctx + i, 1)
                assert rel_l2(bf16_to_f64(t_bits(kg)), bf16_to_f64(okvs[b]["k"][l, :, ctx + i])) < 1e-2, where
                assert rel_l2(bf16_to_f64(t_bits(vg)), bf16_to_f64(okvs[b]["v"][l, :, ctx + i])) < 1e-2, where
                if same:
                    compared += 1
                    gx, ox = bf16_to_f64(g[b]), o["trace"]["layer_out"][l]
                    assert rel_l2(gx, ox) <= HIDDEN_REL_L2, where
                    assert rel_l2(gx - lay_in[b], ox - lay_in[b]) <= HIDDEN_REL_L2, f"{where} delta"
                    order = np.argsort(o["trace"]["topk_idx"][l])
                    assert np.allclose(gg[b][np.argsort(gi[b])], o["trace"]["topk_gate"][l][order], atol=GATE_ABS), where
        eng.close()
    print(f"\nwide teacher-forced layers: {compared} of {8 * n_tok * B} layer outputs compared; {rc.summary()}")
    assert compared >= 8 * n_tok * B - 8, "too few layer outputs compared"
    m_head = {"cfg": synth.MOE8.replace(n_layers=1, max_ctx=cfg8.max_ctx, max_batch=B), "layers": [m_gpu["layers"][7]],
              "embed": m_gpu["embed"], "final_norm": m_gpu["final_norm"], "lm_head": m_gpu["lm_head"]}
    eng = _engine(m_head, max_ctx=cfg8.max_ctx, max_batch=B)
    for b in range(B):
        eng.prefill_import(kvs[b][0][7:8].contiguous(), kvs[b][1][7:8].contiguous(), seq=b)
    chk = StepCheck()
    for i in range(n_tok):
        hin = _bf16(np.stack([outs[b][i]["trace"]["layer_out"][6] for b in range(B)])).cuda()
        g_logits, g_next, g_hidden = _gpu_step(eng, hidden=hin, batch=B)
        gi, _ = eng.routing(0)
        for b in range(B):
            o = outs[b][i]
            if set(gi[b].tolist()) == set(o["trace"]["topk_idx"][7].tolist()):
                chk.add(g_logits[b], o["logits"], g_next[b], o["token"], g_hidden[b], o["hidden"])
    assert chk.steps >= n_tok * B - 2
    chk.assert_ok()
