"""GPU parity: the persistent decode kernel (through the C ABI) against the CPU oracle on the same
seeded inputs. Sizes: the tiny dense decoder and a small MoE run whole workloads; the full-size
MoE stack is checked on sampled decode steps the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
from latency_moe_decode_gb300 import synth
from tests.parity import (GATE_ABS, HIDDEN_REL_L2, LOGIT_MAX_ABS, RouteCheck, StepCheck, bf16_to_f64, rel_l2,
                           t_bits, topk_ok)

pytestmark = pytest.mark.gpu

# A small MoE with the full-size head geometry (head_dim 128, 4 query heads per KV head) so that
# batch and ragged-length cases run in seconds on the oracle.
MOE_SMALL = synth.ModelCfg(n_layers=2, hidden=512, n_heads=8, n_kv_heads=2, head_dim=128, n_experts=16,
                           top_k=4, moe_inter=256, n_shared=1, vocab=2048, max_ctx=512, max_batch=8,
                           rms_eps=1e-6, rope_theta=1e6)
TINY_MOE = synth.ModelCfg(n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, n_experts=8, top_k=2,
                          moe_inter=128, n_shared=1, vocab=512, max_ctx=128, max_batch=4)


def _engine(m_gpu, **kw):
    from latency_moe_decode_gb300.engine import Engine
    return Engine(m_gpu, **kw)


def _models(cfg, seed):
    m_cpu = synth.gen_model(cfg, seed=seed, device="cpu")
    return m_cpu, synth.model_to(m_cpu, "cuda")


def _gpu_step(eng, tok=None, hidden=None, batch=1, seq0=0):
    c = eng.cfg
    logits = torch.empty(batch, max(1, c.vocab), device="cuda") if c.vocab else None
    nxt = torch.empty(batch, dtype=torch.int32, device="cuda") if c.vocab else None
    hout = torch.empty(batch, c.hidden, dtype=torch.bfloat16, device="cuda")
    t = torch.tensor(tok, dtype=torch.int32, device="cuda").reshape(batch) if tok is not None else None
    eng.step(tokens=t, hidden=hidden, batch=batch, seq0=seq0, logits=logits, next_tokens=nxt, hidden_out=hout)
    eng.sync()
    return (logits.cpu().numpy().astype(np.float64) if logits is not None else None,
            nxt.cpu().numpy() if nxt is not None else None, t_bits(hout))


# ------------------------------------------------------------------------------------------------
# tiny dense decoder: KV prefilled from 128 random tokens (seed 0), then 16 greedy steps


def test_tiny_dense_prefill_and_16_greedy_steps():
    cfg = synth.TINY
    m_cpu, m_gpu = _models(cfg, 0)
    prompt = synth.gen_tokens(128, cfg.vocab, seed=0)
    orc = oracle.Oracle(m_cpu)
    kv = orc.new_kv(cfg.max_ctx)
    first = orc.prefill(kv, prompt)
    eng = _engine(m_gpu)
    eng.prefill_tokens(prompt.cuda())
    assert eng.get_length(0) == 128
    # KV cache after prefill, every layer and position
    for l in range(cfg.n_layers):
        k, v = eng.export_kv(0, l, 0, 128)
        ko = bf16_to_f64(kv["k"][l, :, :128])
        vo = bf16_to_f64(kv["v"][l, :, :128])
        assert rel_l2(bf16_to_f64(t_bits(k)), ko) < 1e-2
        assert rel_l2(bf16_to_f64(t_bits(v)), vo) < 1e-2
    chk = StepCheck()
    tok = first["token"]
    for i in range(16):
        o = orc.decode_step(kv, 128 + i, token=tok)
        g_logits, g_next, g_hidden = _gpu_step(eng, tok=[tok])
        chk.add(g_logits[0], o["logits"], g_next[0], o["token"], g_hidden[0], o["hidden"])
        tok = o["token"]
    chk.assert_ok()
    assert eng.get_length(0) == 144


def test_tiny_moe_generate_matches_oracle_greedy():
    cfg = TINY_MOE
    m_cpu, m_gpu = _models(cfg, 1)
    prompt = synth.gen_tokens(24, cfg.vocab, seed=1)
    orc = oracle.Oracle(m_cpu)
    kv = orc.new_kv(cfg.max_ctx)
    first = orc.prefill(kv, prompt)
    eng = _engine(m_gpu)
    eng.prefill_tokens(prompt.cuda())
    toks = [first["token"]]
    for i in range(12):
        toks.append(orc.decode_step(kv, 24 + i, token=toks[-1])["token"])
    gen = eng.generate([first["token"]], 12)[:, 0]
    assert np.array_equal(gen, np.array(toks[1:]))  # free-running greedy, 12 tokens


# ------------------------------------------------------------------------------------------------
# small MoE: batches, ragged lengths, slot offsets, routing


@pytest.fixture(scope="module")
def moe_small():
    return _models(MOE_SMALL, 3)


@pytest.mark.parametrize("batch", [1, 2, 3, 5, 8])
def test_moe_small_batch_ragged(moe_small, batch):
    m_cpu, m_gpu = moe_small
    cfg = MOE_SMALL
    orc = oracle.Oracle(m_cpu)
    eng = _engine(m_gpu)
    lens = [37 + 29 * b for b in range(batch)]  # ragged, crosses 32-position tiles
    kvs = []
    toks = synth.gen_tokens(batch, cfg.vocab, seed=5 + batch).tolist()
    for b in range(batch):
        k, v = synth.gen_kv(cfg, lens[b], seed=100 + b)
        eng.prefill_import(k.cuda(), v.cuda(), seq=b)
        kv = orc.new_kv(cfg.max_ctx)
        orc.import_kv(kv, k, v, lens[b])
        kvs.append(kv)
    g_logits, g_next, g_hidden = _gpu_step(eng, tok=toks, batch=batch)
    chk = StepCheck()
    for b in range(batch):
        o = orc.decode_step(kvs[b], lens[b], token=toks[b], want_trace=True)
        chk.add(g_logits[b], o["logits"], g_next[b], o["token"], g_hidden[b], o["hidden"])
        for l in range(cfg.n_layers):
            gi, gg = eng.routing(l)
            assert topk_ok(gi[b], o["trace"]["topk_idx"][l], o["trace"]["router_score"][l], cfg.top_k)
            if set(gi[b]) == set(o["trace"]["topk_idx"][l]):
                assert np.allclose(gg[b], o["trace"]["topk_gate"][l], atol=GATE_ABS)
                assert abs(gg[b].sum() - 1) < 1e-5
        assert eng.get_length(b) == lens[b] + 1
    chk.assert_ok()


def test_moe_small_slot_offset_and_batch_invariance(moe_small):
    """Sequence results do not depend on which other sequences share the step."""
    m_cpu, m_gpu = moe_small
    cfg = MOE_SMALL
    eng = _engine(m_gpu)
    k, v = synth.gen_kv(cfg, 77, seed=9)
    for s in range(4):
        eng.prefill_import(k.cuda(), v.cuda(), seq=s)
    toks = [11, 11, 11, 11]
    lg4, nx4, h4 = _gpu_step(eng, tok=toks, batch=4)
    for s in range(4):
        eng.set_length(s, 77)
    lg1, nx1, h1 = _gpu_step(eng, tok=[11], batch=1, seq0=2)
    assert np.max(np.abs(lg4[0] - lg1[0])) < 1e-3 and nx4[0] == nx1[0]
    assert np.allclose(lg4[0], lg4[3], atol=1e-3)


def test_moe_small_deterministic_rerun(moe_small):
    m_cpu, m_gpu = moe_small
    eng = _engine(m_gpu)
    k, v = synth.gen_kv(MOE_SMALL, 300, seed=10)
    eng.prefill_import(k.cuda(), v.cuda(), seq=0)
    a = _gpu_step(eng, tok=[5])
    eng.set_length(0, 300)
    b = _gpu_step(eng, tok=[5])
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[2], b[2])


def test_argument_errors(moe_small):
    from latency_moe_decode_gb300.capi import DecError
    m_cpu, m_gpu = moe_small
    eng = _engine(m_gpu, max_batch=2, max_ctx=40)
    t = torch.zeros(3, dtype=torch.int32, device="cuda")
    with pytest.raises(DecError) as e:
        eng.step(tokens=t, batch=3)
    assert e.value.status == -1
    eng.step(tokens=t, batch=0)  # no-op
    k, v = synth.gen_kv(MOE_SMALL.replace(max_ctx=40), 40, seed=1)
    eng.prefill_import(k.cuda(), v.cuda(), seq=0)
    with pytest.raises(DecError) as e:
        eng.step(tokens=t[:1], batch=1)
    assert e.value.status == -8  # capacity
    eng.sync()


# ------------------------------------------------------------------------------------------------
# full size: one MoE layer (hidden 4096, 64 experts, top-8, shared expert), KV 8192 ~N(0,1)


@pytest.fixture(scope="module")
def moe8():
    m_gpu = synth.gen_model(synth.MOE8, seed=0, device="cuda")
    m_cpu = synth.model_to(m_gpu, "cpu")
    return m_cpu, m_gpu


def _one_layer(m):
    m1 = {"cfg": synth.MOE_LAYER, "layers": [m["layers"][0]]}
    return m1


def test_moe_layer_kv8192_hidden_input(moe8):
    m_cpu, m_gpu = moe8
    cfg = synth.MOE_LAYER
    k, v = synth.gen_kv(cfg, 8192, seed=0, device="cuda")
    x = synth.gen_hidden(1, cfg.hidden, seed=0, device="cuda")
    orc = oracle.Oracle(_one_layer(m_cpu))
    kv = orc.new_kv(8193)
    orc.import_kv(kv, k.cpu(), v.cpu(), 8192)
    o = orc.decode_step(kv, 8192, hidden=t_bits(x)[0], want_trace=True)
    eng = _engine(_one_layer(m_gpu), max_ctx=8193)
    eng.prefill_import(k, v, seq=0)
    _, _, g_hidden = _gpu_step(eng, hidden=x, batch=1)
    assert rel_l2(bf16_to_f64(g_hidden[0]), bf16_to_f64(o["hidden"])) <= 1e-2
    gi, gg = eng.routing(0)
    assert topk_ok(gi[0], o["trace"]["topk_idx"][0], o["trace"]["router_score"][0], 8)
    assert abs(gg[0].sum() - 1) < 1e-5
    # the new position's K/V landed in the cache
    kg, vg = eng.export_kv(0, 0, 8192, 1)
    assert rel_l2(bf16_to_f64(t_bits(kg)), bf16_to_f64(kv["k"][0, :, 8192])) < 1e-2
    assert rel_l2(bf16_to_f64(t_bits(vg)), bf16_to_f64(kv["v"][0, :, 8192])) < 1e-2


def test_moe_layer_batch4_expert_major_down(moe8):
    """Full-size layer at batch 4 (up to 33 active expert slots: the expert-major order of the
    down projections, and CTA-wide waits over every KV head of four sequences), each sequence
    against the oracle with its own ragged KV history."""
    m_cpu, m_gpu = moe8
    cfg = synth.MOE_LAYER
    B = 4
    lens = [1024 + 77 * b for b in range(B)]
    orc = oracle.Oracle(_one_layer(m_cpu))
    eng = _engine(_one_layer(m_gpu), max_ctx=2048, max_batch=B)
    x = synth.gen_hidden(B, cfg.hidden, seed=9, device="cuda")
    outs = []
    for b in range(B):
        k, v = synth.gen_kv(cfg, lens[b], seed=40 + b, device="cuda")
        eng.prefill_import(k, v, seq=b)
        kv = orc.new_kv(2048)
        orc.import_kv(kv, k.cpu(), v.cpu(), lens[b])
        outs.append(orc.decode_step(kv, lens[b], hidden=t_bits(x)[b], want_trace=True))
    _, _, g_hidden = _gpu_step(eng, hidden=x, batch=B)
    gi, gg = eng.routing(0)
    assert len(set(gi[:B].reshape(-1).tolist())) + 1 > 12  # the expert-major order was taken
    for b, o in enumerate(outs):
        assert topk_ok(gi[b], o["trace"]["topk_idx"][0], o["trace"]["router_score"][0], 8)
        if set(gi[b]) == set(o["trace"]["topk_idx"][0]):
            assert rel_l2(bf16_to_f64(g_hidden[b]), bf16_to_f64(o["hidden"])) <= 1e-2
        assert eng.get_length(b) == lens[b] + 1


def _bf16(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16)


def _oracle_run(m_cpu, k, v, ctx, n_tok, tok=1234, max_ctx=None):
    """The oracle decoding n_tok greedy tokens after an imported KV state, with traces."""
    orc = oracle.Oracle(m_cpu)
    kv = orc.new_kv(max_ctx or ctx + n_tok + 16)
    orc.import_kv(kv, k.cpu(), v.cpu(), ctx)
    outs, toks = [], []
    for i in range(n_tok):
        toks.append(tok)
        o = orc.decode_step(kv, ctx + i, token=tok, want_trace=True)
        outs.append(o)
        tok = o["token"]
    return orc, kv, outs, toks


@pytest.mark.parametrize("ctx,n_tok", [(1024, 8), (8192, 2)], ids=["1k", "8k"])
def test_moe8_every_layer_teacher_forced(moe8, ctx, n_tok):
    """Every layer of the 8-layer stack on the GPU, fed the oracle's own input to that layer, for
    n_tok consecutive decode tokens (each layer's engine keeps its own KV cache, which grows by the
    keys and values it computes), against the oracle's output of that layer. Strict tolerances:
    layer output and sublayer delta rel L2 <= 1e-2, new K/V rows <= 1e-2, gates, and routing
    (RouteCheck: the engine's selection is the top-k of its own logits, its logits are within
    ROUTER_LOGIT_ABS of the oracle's, and the selections are equal except at a near-tie of the
    oracle's logits, where the step's outputs are not compared). Then the LM head, fed the
    oracle's final hidden state, on every token."""
    m_cpu, m_gpu = moe8
    cfg8 = synth.MOE8.replace(max_ctx=ctx + n_tok + 16)
    k, v = synth.gen_kv(cfg8, ctx, seed=1, device="cuda")
    _, okv, outs, toks = _oracle_run(m_cpu, k, v, ctx, n_tok, max_ctx=cfg8.max_ctx)
    cfg1 = synth.MOE_LAYER.replace(max_ctx=cfg8.max_ctx)
    rc = RouteCheck()
    compared = 0
    for l in range(8):
        eng = _engine({"cfg": cfg1, "layers": [m_gpu["layers"][l]]}, max_ctx=cfg1.max_ctx)
        eng.prefill_import(k[l:l + 1].contiguous(), v[l:l + 1].contiguous())
        for i, (o, tok) in enumerate(zip(outs, toks)):
            lay_in = bf16_to_f64(t_bits(m_cpu["embed"][tok])) if l == 0 else o["trace"]["layer_out"][l - 1]
            _, _, g = _gpu_step(eng, hidden=_bf16(lay_in).reshape(1, -1).cuda())
            where = f"token {i} layer {l}"
            gi, gg = eng.routing(0)
            same = rc.check(gi[0], eng.router_logits(0)[0], o["trace"]["topk_idx"][l], o["trace"]["router_score"][l],
                            8, where)
            assert abs(gg[0].sum() - 1) < 1e-5
            kg, vg = eng.export_kv(0, 0, ctx + i, 1)
            assert rel_l2(bf16_to_f64(t_bits(kg)), bf16_to_f64(okv["k"][l, :, ctx + i])) < 1e-2, where
            assert rel_l2(bf16_to_f64(t_bits(vg)), bf16_to_f64(okv["v"][l, :, ctx + i])) < 1e-2, where
            if same:
                compared += 1
                gx, ox = bf16_to_f64(g[0]), o["trace"]["layer_out"][l]
                assert rel_l2(gx, ox) <= HIDDEN_REL_L2, where
                assert rel_l2(gx - lay_in, ox - lay_in) <= HIDDEN_REL_L2, f"{where} delta"
                order = np.argsort(o["trace"]["topk_idx"][l])
                assert np.allclose(gg[0][np.argsort(gi[0])], o["trace"]["topk_gate"][l][order], atol=GATE_ABS), where
        eng.close()
    print(f"\nteacher-forced layers ({ctx}, {n_tok} tokens): {compared} layer outputs compared; {rc.summary()}")
    assert compared >= 8 * n_tok - max(2, n_tok), "too few layer outputs compared"
    # LM head + final norm + argmax: a 1-layer model whose layer is the last one, fed its input
    m_head = {"cfg": synth.MOE8.replace(n_layers=1, max_ctx=cfg8.max_ctx), "layers": [m_gpu["layers"][7]],
              "embed": m_gpu["embed"], "final_norm": m_gpu["final_norm"], "lm_head": m_gpu["lm_head"]}
    eng = _engine(m_head, max_ctx=cfg8.max_ctx)
    eng.prefill_import(k[7:8].contiguous(), v[7:8].contiguous())
    chk = StepCheck()
    for o in outs:
        g_logits, g_next, g_hidden = _gpu_step(eng, hidden=_bf16(o["trace"]["layer_out"][6]).reshape(1, -1).cuda())
        gi, _ = eng.routing(0)
        if set(gi[0].tolist()) == set(o["trace"]["topk_idx"][7].tolist()):
            chk.add(g_logits[0], o["logits"], g_next[0], o["token"], g_hidden[0], o["hidden"])
    assert chk.steps >= n_tok - 1
    chk.assert_ok()


def test_moe8_greedy_agreement_64_tokens_teacher_forced(moe8):
    """Greedy agreement over 64 full-size decode tokens at context 1k. The oracle decodes the
    tokens; the GPU runs the last layer and the LM head fed the oracle's input to that layer
    (teacher-forced, with its own KV cache of that layer), so every token's argmax is decided by
    the engine's own final layer, norm, LM head and argmax kernels. Agreement >= 99% over the
    tokens that are not near-ties (oracle top-2 logit gap >= NEAR_TIE, routing of the layer equal);
    near-ties are left out of both counts and reported."""
    m_cpu, m_gpu = moe8
    ctx, n_tok = 1024, 64
    cfg8 = synth.MOE8.replace(max_ctx=ctx + n_tok + 16)
    k, v = synth.gen_kv(cfg8, ctx, seed=1, device="cuda")
    _, _, outs, _ = _oracle_run(m_cpu, k, v, ctx, n_tok, tok=4321, max_ctx=cfg8.max_ctx)
    m_head = {"cfg": synth.MOE8.replace(n_layers=1, max_ctx=cfg8.max_ctx), "layers": [m_gpu["layers"][7]],
              "embed": m_gpu["embed"], "final_norm": m_gpu["final_norm"], "lm_head": m_gpu["lm_head"]}
    eng = _engine(m_head, max_ctx=cfg8.max_ctx)
    eng.prefill_import(k[7:8].contiguous(), v[7:8].contiguous())
    chk, rc = StepCheck(), RouteCheck()
    for i, o in enumerate(outs):
        g_logits, g_next, g_hidden = _gpu_step(eng, hidden=_bf16(o["trace"]["layer_out"][6]).reshape(1, -1).cuda())
        gi, _ = eng.routing(0)
        if rc.check(gi[0], eng.router_logits(0)[0], o["trace"]["topk_idx"][7], o["trace"]["router_score"][7], 8,
                    f"token {i}"):
            chk.add(g_logits[0], o["logits"], g_next[0], o["token"], g_hidden[0], o["hidden"])
    print(f"\ngreedy agreement: {chk.agree}/{chk.steps - chk.near_ties} tokens ({chk.near_ties} near-tie tokens "
          f"left out, {n_tok - chk.steps} at routing near-ties); max logit err {chk.max_logit_err:.3e}, "
          f"max hidden rel {chk.max_hidden_rel:.3e}; {rc.summary()}")
    assert chk.steps >= n_tok - 4
    chk.assert_ok()


# The chained 8-layer stack cannot meet the single-layer tolerances, and no implementation that
# rounds differently from the oracle could: on this random-weight stack the oracle itself, given
# the same token with SENS_FLIPS input elements moved by one bf16 ulp, drifts by a median of ~6%
# in the final hidden state and ~0.3 in the logits, flips a router selection somewhere in the
# stack on ~40% of tokens and its own greedy token on ~1 token in 8 (measured over 64 tokens at 1k;
# the router logits of random weights put many experts within 1e-3 of the 8th, and a flipped
# expert changes a layer's output by several percent). So the chained check is statistical: over
# the steps, the engine's deviation from the oracle must not exceed the oracle's deviation from
# itself under that perturbation (medians, with a 1.5x margin), every step is compared, and the
# counts are reported.
SENS_FLIPS = 8
CHAIN_KV_REL = 5e-2


def _perturbed(orc, kv, pos, x_bits, seed):
    """The oracle's step with SENS_FLIPS input elements moved by one bf16 ulp (on a copy of the cache)."""
    kv2 = {kk: (vv.copy() if isinstance(vv, np.ndarray) else vv) for kk, vv in kv.items()}
    bits = np.array(x_bits, np.uint16)
    idx = np.random.default_rng(seed).choice(bits.size, SENS_FLIPS, replace=False)
    bits[idx] ^= 1
    return orc.decode_step(kv2, pos, hidden=bits, want_trace=True)


@pytest.mark.parametrize("ctx,steps", [(1024, 16), (8192, 4)], ids=["1k", "8k"])
def test_moe8_chained_decode_steps(moe8, ctx, steps):
    """The whole 8-layer stack chained on the GPU vs the oracle, token-forced from the oracle."""
    m_cpu, m_gpu = moe8
    cfg = synth.MOE8.replace(max_ctx=ctx + steps + 16)
    k, v = synth.gen_kv(cfg, ctx, seed=1, device="cuda")
    orc = oracle.Oracle(m_cpu)
    kv = orc.new_kv(cfg.max_ctx)
    orc.import_kv(kv, k.cpu(), v.cpu(), ctx)
    eng = _engine(m_gpu, max_ctx=cfg.max_ctx)
    eng.prefill_import(k, v, seq=0)
    embed = m_cpu["embed"].view(torch.int16).numpy().view(np.uint16)
    g_h, g_l, s_h, s_l = [], [], [], []
    g_agree = s_agree = routed_same = 0
    tok = 1234
    for i in range(steps):
        op = _perturbed(orc, kv, ctx + i, embed[tok], seed=i)
        o = orc.decode_step(kv, ctx + i, token=tok, want_trace=True)
        g_logits, g_next, g_hidden = _gpu_step(eng, tok=[tok])
        assert np.isfinite(g_logits).all()
        g_l.append(float(np.abs(g_logits[0] - o["logits"]).max()))
        g_h.append(rel_l2(bf16_to_f64(g_hidden[0]), bf16_to_f64(o["hidden"])))
        s_l.append(float(np.abs(op["logits"] - o["logits"]).max()))
        s_h.append(rel_l2(bf16_to_f64(op["hidden"]), bf16_to_f64(o["hidden"])))
        g_agree += int(g_next[0]) == int(o["token"])
        s_agree += int(op["token"]) == int(o["token"])
        routed_same += all(set(eng.routing(l)[0][0].tolist()) == set(o["trace"]["topk_idx"][l].tolist())
                           for l in range(cfg.n_layers))
        tok = o["token"]
    print(f"\nchained {ctx}: {steps} steps compared; routing identical at all layers on {routed_same}; "
          f"greedy agreement engine {g_agree}/{steps}, perturbed oracle {s_agree}/{steps}; median hidden rel "
          f"engine {np.median(g_h):.3e} vs oracle spread {np.median(s_h):.3e}; median logits err engine "
          f"{np.median(g_l):.3e} vs spread {np.median(s_l):.3e}")
    assert len(g_h) == steps
    assert np.median(g_h) <= 1.5 * max(np.median(s_h), HIDDEN_REL_L2 / 4)
    assert np.median(g_l) <= 1.5 * max(np.median(s_l), LOGIT_MAX_ABS / 4)


def test_moe8_token_prefill(moe8):
    """Token-mode prefill at full size: the KV of every layer against the oracle's, and the engine's
    own KV state carried over exactly (an engine given the exported cache by import mode decodes
    the next token bit for bit like the one that prefilled it)."""
    m_cpu, m_gpu = moe8
    cfg = synth.MOE8.replace(max_ctx=64)
    prompt = synth.gen_tokens(3, cfg.vocab, seed=7)
    orc = oracle.Oracle(m_cpu)
    kv = orc.new_kv(cfg.max_ctx)
    first = orc.prefill(kv, prompt)
    eng = _engine(m_gpu, max_ctx=cfg.max_ctx)
    eng.prefill_tokens(prompt.cuda())
    ks, vs = [], []
    for l in range(cfg.n_layers):
        kg, vg = eng.export_kv(0, l, 0, 3)
        ks.append(kg)
        vs.append(vg)
        tol = 1e-2 if l == 0 else CHAIN_KV_REL  # layer 0 sees the embeddings directly
        assert rel_l2(bf16_to_f64(t_bits(kg)), bf16_to_f64(kv["k"][l, :, :3])) < tol, l
        assert rel_l2(bf16_to_f64(t_bits(vg)), bf16_to_f64(kv["v"][l, :, :3])) < tol, l
    twin = _engine(m_gpu, max_ctx=cfg.max_ctx)
    twin.prefill_import(torch.stack(ks), torch.stack(vs), seq=0)
    assert twin.get_length(0) == eng.get_length(0) == 3
    a = _gpu_step(eng, tok=[first["token"]])
    b = _gpu_step(twin, tok=[first["token"]])
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
