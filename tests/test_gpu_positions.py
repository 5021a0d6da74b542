"""Several positions of one sequence in one launch: dec_step_positions (chunked prefill, the
verify step's compute) and dec_verify (speculative-decoding verification), against the oracle
decoding the same positions one by one ("vLLM's Kimi K3 Backend Hits 842 Tokens per Second",
section "Throughput holds across the tested range": drafts verified in one step)."""
import numpy as np
import pytest
import torch

import oracle
from latency_moe_decode_gb300 import synth
from tests.parity import HIDDEN_REL_L2, LOGIT_MAX_ABS, bf16_to_f64, near_tie, rel_l2, t_bits

pytestmark = pytest.mark.gpu

# head_dim 128 and 4 query heads per KV head like the full-size layer; small enough for the oracle
CFG = synth.ModelCfg(n_layers=2, hidden=512, n_heads=8, n_kv_heads=2, head_dim=128, n_experts=16, top_k=4,
                     moe_inter=256, n_shared=1, vocab=2048, max_ctx=256, max_batch=2, rms_eps=1e-6,
                     rope_theta=1e6)


@pytest.fixture(scope="module")
def models():
    m_cpu = synth.gen_model(CFG, seed=21, device="cpu")
    return m_cpu, synth.model_to(m_cpu, "cuda")


def _engine(m_gpu):
    from latency_moe_decode_gb300.engine import Engine
    return Engine(m_gpu)


def _setup(models, ctx, seq):
    """Both sides with the same synthetic KV state of ctx positions (slot `seq` on the GPU)."""
    m_cpu, m_gpu = models
    k, v = synth.gen_kv(CFG, ctx, seed=ctx)
    orc = oracle.Oracle(m_cpu)
    kv = orc.new_kv(CFG.max_ctx)
    orc.import_kv(kv, k, v, ctx)
    eng = _engine(m_gpu)
    eng.prefill_import(k.cuda(), v.cuda(), seq=seq)
    return orc, kv, eng


@pytest.mark.parametrize("n,ctx", [(1, 40), (5, 61), (8, 120)], ids=["n1", "n5_crosses_tile", "n8"])
def test_positions_match_oracle_one_by_one(models, n, ctx):
    orc, kv, eng = _setup(models, ctx, seq=1)
    toks = synth.gen_tokens(n, CFG.vocab, seed=n).tolist()
    logits = torch.empty(n, CFG.vocab, device="cuda")
    nxt = torch.empty(n, dtype=torch.int32, device="cuda")
    eng.step_positions(torch.tensor(toks, dtype=torch.int32, device="cuda"), seq=1, logits=logits, next_tokens=nxt)
    eng.sync()
    g_logits, g_next = logits.cpu().numpy().astype(np.float64), nxt.cpu().numpy()
    assert eng.get_length(1) == ctx + n and eng.get_length(0) == 0
    for j, t in enumerate(toks):
        o = orc.decode_step(kv, ctx + j, token=t)
        err = float(np.abs(g_logits[j] - o["logits"]).max())
        assert err <= LOGIT_MAX_ABS, f"position {j}: logits {err:.3e}"
        assert int(g_next[j]) == o["token"] or near_tie(o["logits"]), f"position {j}"
    for l in range(CFG.n_layers):  # the new keys and values landed at their positions
        kg, vg = eng.export_kv(1, l, ctx, n)
        assert rel_l2(bf16_to_f64(t_bits(kg)), bf16_to_f64(kv["k"][l, :, ctx:ctx + n])) < HIDDEN_REL_L2
        assert rel_l2(bf16_to_f64(t_bits(vg)), bf16_to_f64(kv["v"][l, :, ctx:ctx + n])) < HIDDEN_REL_L2
    eng.close()


def test_verify_accepts_the_matching_prefix_and_continues(models):
    """Drafts = the oracle's own next two greedy tokens, then a wrong one: two are accepted, the
    correction is the oracle's third token, the slot keeps ctx + 3 positions, and the next decode
    step (which overwrites the rejected draft's cache position) matches the oracle."""
    ctx, t0 = 90, 7
    orc, kv, eng = _setup(models, ctx, seq=0)
    greedy, tok = [], t0
    for j in range(4):  # the oracle's continuation (its cache then holds ctx + 4 positions)
        o = orc.decode_step(kv, ctx + j, token=tok)
        greedy.append(o["token"])
        tok = o["token"]
    wrong = (greedy[2] + 1) % CFG.vocab
    drafts = [t0, greedy[0], greedy[1], wrong, greedy[3]]
    nxt = torch.empty(len(drafts), dtype=torch.int32, device="cuda")
    m = eng.verify(torch.tensor(drafts, dtype=torch.int32, device="cuda"), seq=0, next_tokens=nxt)
    assert m == 2
    assert int(nxt[2].item()) == greedy[2]
    assert eng.get_length(0) == ctx + 3
    # continue from the correction at position ctx + 3: the oracle's step at that position is
    # the one it took with greedy[2] as input
    kv2 = orc.new_kv(CFG.max_ctx)
    kv2["k"][:], kv2["v"][:] = kv["k"], kv["v"]
    ref = orc.decode_step(kv2, ctx + 3, token=greedy[2])
    logits = torch.empty(1, CFG.vocab, device="cuda")
    eng.step(tokens=torch.tensor([greedy[2]], dtype=torch.int32, device="cuda"), batch=1, logits=logits)
    eng.sync()
    assert float(np.abs(logits.cpu().numpy()[0] - ref["logits"]).max()) <= LOGIT_MAX_ABS
    eng.close()


def test_verify_rejects_everything(models):
    ctx, t0 = 33, 11
    orc, kv, eng = _setup(models, ctx, seq=0)
    o = orc.decode_step(kv, ctx, token=t0)
    drafts = [t0, (o["token"] + 5) % CFG.vocab, 3, 4]
    nxt = torch.empty(len(drafts), dtype=torch.int32, device="cuda")
    m = eng.verify(torch.tensor(drafts, dtype=torch.int32, device="cuda"), seq=0, next_tokens=nxt)
    assert m == 0 and eng.get_length(0) == ctx + 1 and int(nxt[0].item()) == o["token"]
    eng.close()


def test_chunked_token_prefill_matches_oracle(models):
    """Token-mode prefill of one slot runs chunks of up to 8 positions per launch (21 = 8 + 8 + 5)."""
    m_cpu, m_gpu = models
    prompt = synth.gen_tokens(21, CFG.vocab, seed=4)
    orc = oracle.Oracle(m_cpu)
    kv = orc.new_kv(CFG.max_ctx)
    first = orc.prefill(kv, prompt)
    eng = _engine(m_gpu)
    launches0 = eng.info()["launches"]
    eng.prefill_tokens(prompt.cuda(), seq=1)
    assert eng.info()["launches"] - launches0 == 3 and eng.get_length(1) == 21
    for l in range(CFG.n_layers):
        kg, vg = eng.export_kv(1, l, 0, 21)
        assert rel_l2(bf16_to_f64(t_bits(kg)), bf16_to_f64(kv["k"][l, :, :21])) < HIDDEN_REL_L2
        assert rel_l2(bf16_to_f64(t_bits(vg)), bf16_to_f64(kv["v"][l, :, :21])) < HIDDEN_REL_L2
    o = orc.decode_step(kv, 21, token=first["token"])
    logits = torch.empty(1, CFG.vocab, device="cuda")
    eng.step(tokens=torch.tensor([first["token"]], dtype=torch.int32, device="cuda"), batch=1, seq0=1, logits=logits)
    eng.sync()
    assert float(np.abs(logits.cpu().numpy()[0] - o["logits"]).max()) <= LOGIT_MAX_ABS
    eng.close()


def test_positions_arguments(models):
    from latency_moe_decode_gb300.capi import DecError
    m_cpu, m_gpu = models
    eng = _engine(m_gpu)
    t = torch.zeros(9, dtype=torch.int32, device="cuda")
    with pytest.raises(DecError) as e:
        eng.step_positions(t, seq=0)  # more than DEC_MAX_STEP_TOKENS
    assert e.value.status == -1
    with pytest.raises(DecError) as e:
        eng.step_positions(t[:2], seq=2)  # slot out of range
    assert e.value.status == -1
    eng.set_length(0, CFG.max_ctx - 1)
    with pytest.raises(DecError) as e:
        eng.step_positions(t[:2], seq=0)
    assert e.value.status == -8
    eng.close()
