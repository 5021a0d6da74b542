"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties one oracle function to a library routine (torch's E4M3 and bf16 conversions,
numpy matmul/sort), to a hand-computed worked example (tests/golden/worked_examples.json), to a
closed form, or to an invariant of the definition, so that a dropped term, a wrong sign or index,
or a transposed operand fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from latency_moe_decode_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def torch_dequant(w_u8, s):
    """Dense float64 matrix from E4M3 codes + 128x128 block scales, decoded by torch."""
    w = torch.as_tensor(np.ascontiguousarray(w_u8)).view(torch.float8_e4m3fn).double().numpy()
    n, k = w.shape
    srep = np.repeat(np.repeat(np.asarray(s, np.float64), 128, 0), 128, 1)[:n, :k]
    return w * srep


def torch_bf16(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).double().numpy()


# ---------------------------------------------------------------- FP8 E4M3 codec

def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    mine = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.isnan(mine[nan]).all()  # S.1111.111 only
    assert np.array_equal(mine[~nan], ref[~nan])


def test_e4m3_named_values():
    assert oracle.e4m3_value(0x7E) == 448.0          # largest finite
    assert oracle.e4m3_value(0x01) == 2.0 ** -9      # smallest subnormal
    assert oracle.e4m3_value(0x08) == 2.0 ** -6      # smallest normal
    assert oracle.e4m3_value(0x38) == 1.0            # exponent field 7 = bias
    assert oracle.e4m3_value(0xB8) == -1.0
    assert oracle.e4m3_value(0x00) == 0.0 and math.copysign(1, oracle.e4m3_value(0x80)) < 0


def test_generator_codes_decode_back():
    """The input generator's quantiser + the oracle decoder reproduce W within half an E4M3 step."""
    w = torch.randn(256, 384, generator=torch.Generator().manual_seed(3)) * 0.02
    q, s = synth.quantize_fp8_blocks(w)
    deq = np.array([[oracle.e4m3_value(int(c)) for c in row] for row in q[:8].numpy()])
    deq *= np.repeat(s.numpy()[0], 128)[None, :]
    err = np.abs(deq - w[:8].double().numpy())
    assert err.max() <= 0.0625 * float(w[:8].abs().max()) + 1e-12


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000),
                        np.float32([1.00390625, 1.01171875, -2.00781250, 3.0e38, 1e-40, 0.0, -0.0])])
    x = x.astype(np.float32)
    ref = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = np.array([oracle.bf16_bits(float(v)) for v in x], np.uint16)
    assert np.array_equal(mine, ref)


def test_bf16_rounds_double_once():
    # 1 + 2^-8 is the midpoint between bf16 neighbours 1 and 1 + 2^-7. Slightly above it must
    # round up; rounding through float32 first would land on the midpoint and tie to even (1.0).
    assert oracle.bf16_bits(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle.bf16_bits(1.0 + 2.0 ** -8) == 0x3F80          # exact tie -> even
    assert oracle.bf16_bits(1.0 + 3 * 2.0 ** -8) == 0x3F82      # tie between 0x3F81 and 0x3F82 -> even


# ---------------------------------------------------------------- block-scaled GEMV

@pytest.mark.parametrize("n,k", [(64, 128), (128, 128), (192, 256), (256, 64), (130, 200), (1, 384)])
def test_gemv_brute_force(n, k):
    rng = np.random.default_rng(n * 1000 + k)
    w = torch.randn(n, k, generator=torch.Generator().manual_seed(n + k)) * 0.05
    q, s = synth.quantize_fp8_blocks(w)
    s = s * torch.tensor(rng.uniform(0.5, 2.0, s.shape), dtype=torch.float32)  # distinct block scales
    x = rng.standard_normal(k)
    ref = torch_dequant(q.numpy(), s.numpy()) @ x
    mine = oracle.gemv(q.numpy(), s.numpy(), x)
    assert np.allclose(mine, ref, rtol=1e-12, atol=1e-12)


def test_gemv_integer_exact():
    # codes of small integers (E4M3 represents 0..16 exactly), scale 1: exact integer result.
    rng = np.random.default_rng(7)
    ints = rng.integers(-8, 9, size=(128, 256)).astype(np.float32)
    codes = torch.tensor(ints).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    s = np.ones((1, 2), np.float32)
    x = rng.integers(-5, 6, size=256).astype(np.float64)
    assert np.array_equal(oracle.gemv(codes, s, x), ints.astype(np.int64) @ x.astype(np.int64))


def test_gemv_scale_applies_to_its_block_only():
    codes = np.full((256, 256), 0x38, np.uint8)  # all ones
    s = np.array([[1.0, 2.0], [3.0, 5.0]], np.float32)
    x = np.ones(256)
    y = oracle.gemv(codes, s, x)
    assert np.all(y[:128] == 128 * 1.0 + 128 * 2.0) and np.all(y[128:] == 128 * 3.0 + 128 * 5.0)


# ---------------------------------------------------------------- RMSNorm, RoPE

def test_rmsnorm_worked_example():
    g = json.load(open(GOLDEN))["rmsnorm"]
    w = np.full(4, 0x3F80, np.uint16)  # bf16 ones
    out = oracle.rmsnorm(np.array(g["x"], float), w, g["eps"])
    assert np.allclose(out, torch_bf16(g["out_unrounded"]), atol=0)
    assert np.allclose(out, g["out_unrounded"], rtol=4e-3)


def test_rmsnorm_weight_and_scale_invariance():
    rng = np.random.default_rng(1)
    x = torch_bf16(rng.standard_normal(256))
    w2 = np.full(256, 0x4000, np.uint16)  # bf16 2.0
    ones = np.full(256, 0x3F80, np.uint16)
    a = oracle.rmsnorm(x, ones, 0.0)
    assert np.array_equal(oracle.rmsnorm(x, w2, 0.0), 2 * a)     # scaling by a power of two is exact
    assert np.array_equal(oracle.rmsnorm(8 * x, ones, 0.0), a)     # scale invariant (eps = 0)
    assert abs(np.mean(a.astype(np.float64) ** 2) - 1.0) < 1e-2


def test_rope_worked_example_half_split():
    g = json.load(open(GOLDEN))["rope"]
    for pos, want in g["half_split"].items():
        assert np.allclose(oracle.rope(g["x"], int(pos), g["theta"]), want, atol=2e-7)
    assert not np.allclose(oracle.rope(g["x"], 1, g["theta"]), g["interleaved_pos1_for_contrast"], atol=1e-3)


def test_rope_invariants():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for p in (0, 1, 17, 8191):
        assert abs(np.linalg.norm(oracle.rope(q, p, 1e6)) - np.linalg.norm(q)) < 1e-9
    d1 = oracle.rope(q, 100, 1e4) @ oracle.rope(k, 40, 1e4)
    d2 = oracle.rope(q, 1060, 1e4) @ oracle.rope(k, 1000, 1e4)
    assert abs(d1 - d2) < 1e-9  # depends on the position difference only


# ---------------------------------------------------------------- attention

def bf16bits(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_attention_closed_forms():
    rng = np.random.default_rng(3)
    hd = 64
    q = torch_bf16(rng.standard_normal(hd))
    v1 = bf16bits(rng.standard_normal((1, hd)))
    k1 = bf16bits(rng.standard_normal((1, hd)))
    assert np.array_equal(oracle.attention_head(q, k1, v1), torch_bf16(torch.tensor(v1.view(np.int16)).view(torch.bfloat16).float().numpy()[0]))
    # equal keys -> mean of values
    K = np.repeat(k1, 5, 0)
    V = bf16bits(rng.standard_normal((5, hd)))
    Vf = torch.tensor(V.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.allclose(oracle.attention_head(q, K, V), Vf.mean(0), atol=1e-12)
    # two keys: weights sigmoid(s1 - s0) with s = q.k / sqrt(hd)
    K2 = bf16bits(rng.standard_normal((2, hd)))
    Kf = torch.tensor(K2.view(np.int16)).view(torch.bfloat16).double().numpy()
    V2 = bf16bits(rng.standard_normal((2, hd)))
    V2f = torch.tensor(V2.view(np.int16)).view(torch.bfloat16).double().numpy()
    s = Kf @ q / math.sqrt(hd)
    w1 = 1.0 / (1.0 + math.exp(s[0] - s[1]))
    assert np.allclose(oracle.attention_head(q, K2, V2), (1 - w1) * V2f[0] + w1 * V2f[1], atol=1e-12)


def test_attention_matches_torch_sdpa():
    rng = np.random.default_rng(4)
    hd, n = 128, 300
    q = torch_bf16(rng.standard_normal(hd))
    K = bf16bits(rng.standard_normal((n, hd)))
    V = bf16bits(rng.standard_normal((n, hd)))
    Kt = torch.tensor(K.view(np.int16)).view(torch.bfloat16).double()
    Vt = torch.tensor(V.view(np.int16)).view(torch.bfloat16).double()
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q)[None, None, None], Kt[None, None], Vt[None, None])[0, 0, 0].numpy()
    assert np.allclose(oracle.attention_head(q, K, V), ref, atol=1e-10)


# ---------------------------------------------------------------- router

def test_router_topk_vs_sort():
    rng = np.random.default_rng(5)
    for trial in range(50):
        r = rng.standard_normal(64) * 2
        idx, gate, score = oracle.router_topk(r, 8)
        order = np.argsort(-r, kind="stable")[:8]  # sigmoid is monotone: same order as the logits
        assert list(idx) == list(order)
        sig = 1 / (1 + np.exp(-r))
        assert np.allclose(score, sig, rtol=1e-14)
        assert np.allclose(gate, sig[order] / sig[order].sum(), rtol=1e-14)
        assert abs(gate.sum() - 1.0) < 1e-12


def test_router_ties_go_to_lower_index():
    r = np.zeros(16)
    r[[3, 9, 12]] = 1.0
    idx, gate, _ = oracle.router_topk(r, 4)
    assert list(idx) == [3, 9, 12, 0]
    assert np.allclose(gate, np.array([1, 1, 1, 0.5 / (1 / (1 + math.exp(-1)))]) / (3 + 0.5 / (1 / (1 + math.exp(-1)))))


# ---------------------------------------------------------------- SwiGLU expert

def test_swiglu_expert_brute_force():
    g = synth.fp8_matrix(128, 256, "cpu", 11, "g")
    u = synth.fp8_matrix(128, 256, "cpu", 11, "u")
    d = synth.fp8_matrix(256, 128, "cpu", 11, "d")
    xn = torch_bf16(np.random.default_rng(6).standard_normal(256))
    G, U, D = (torch_dequant(t[0].numpy(), t[1].numpy()) for t in (g, u, d))
    a, b = G @ xn, U @ xn
    h = torch_bf16(a / (1 + np.exp(-a)) * b)
    ref = D @ h
    got = oracle.swiglu_expert((g[0].numpy(), g[1].numpy()), (u[0].numpy(), u[1].numpy()),
                               (d[0].numpy(), d[1].numpy()), xn)
    assert np.allclose(got, ref, rtol=1e-6, atol=1e-9)


def test_swiglu_zero_gate_gives_zero():
    z = (np.zeros((128, 256), np.uint8), np.ones((1, 2), np.float32))
    u = synth.fp8_matrix(128, 256, "cpu", 12, "u")
    d = synth.fp8_matrix(256, 128, "cpu", 12, "d")
    y = oracle.swiglu_expert(z, (u[0].numpy(), u[1].numpy()), (d[0].numpy(), d[1].numpy()),
                             np.ones(256))
    assert np.all(y == 0)  # silu(0) = 0


# ---------------------------------------------------------------- whole decoder

TINY_MOE = synth.ModelCfg(n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64,
                          n_experts=8, top_k=2, moe_inter=128, n_shared=1, vocab=512, max_ctx=64)


@pytest.mark.parametrize("cfg", [synth.TINY.replace(max_ctx=64), TINY_MOE], ids=["dense", "moe"])
def test_full_recompute_equals_incremental(cfg):
    m = synth.gen_model(cfg, seed=1)
    orc = oracle.Oracle(m)
    toks = synth.gen_tokens(12, cfg.vocab, seed=1)
    kv = orc.new_kv(cfg.max_ctx)
    inc = orc.prefill(kv, toks)
    tok, logits = orc.full_recompute(toks)
    assert np.array_equal(inc["logits"], logits) and inc["token"] == tok


def test_zero_layers_is_lm_head_of_normed_embedding():
    cfg = synth.TINY.replace(n_layers=0)
    m = synth.gen_model(cfg, seed=2)
    orc = oracle.Oracle(m)
    kv = orc.new_kv(8)
    out = orc.decode_step(kv, 0, token=77)
    e = m["embed"][77].double().numpy()
    xn = torch_bf16(e / np.sqrt(np.mean(e * e) + cfg.rms_eps))
    ref = torch_dequant(m["lm_head"][0].numpy(), m["lm_head"][1].numpy()) @ xn
    assert np.allclose(out["logits"], ref, rtol=1e-9, atol=1e-12)
    assert out["token"] == int(np.argmax(ref))


def test_single_position_attention_returns_own_value_gqa_mapping():
    """At position 0 each query head's output is its KV head's v (head h reads h // group)."""
    cfg = synth.TINY.replace(n_layers=1, n_heads=4, n_kv_heads=2)
    m = synth.gen_model(cfg, seed=3)
    orc = oracle.Oracle(m)
    kv = orc.new_kv(8)
    out = orc.decode_step(kv, 0, token=5, want_trace=True)
    e = m["embed"][5].double().numpy()
    xn = torch_bf16(e / np.sqrt(np.mean(e * e) + cfg.rms_eps))
    Wv = torch_dequant(m["layers"][0]["wv"][0].numpy(), m["layers"][0]["wv"][1].numpy())
    v = torch_bf16(Wv @ xn).reshape(2, 64)
    o = out["trace"]["attn_out"][0].reshape(4, 64)
    for h in range(4):
        assert np.array_equal(o[h], v[h // 2])


def test_moe_with_one_expert_equals_dense_ffn():
    """top-1 of a single routed expert (gate 1) and no shared expert == the dense SwiGLU FFN."""
    dense_cfg = synth.TINY.replace(n_layers=1)
    moe_cfg = dense_cfg.replace(dense_ffn=0, n_experts=1, top_k=1, moe_inter=512, n_shared=0)
    md = synth.gen_model(dense_cfg, seed=4)
    mm = synth.gen_model(moe_cfg, seed=4)
    for k in ("embed", "final_norm", "lm_head"):
        mm[k] = md[k]
    Ld, Lm = md["layers"][0], mm["layers"][0]
    for k in ("attn_norm", "ffn_norm", "wq", "wk", "wv", "wo"):
        Lm[k] = Ld[k]
    Lm["gate"], Lm["up"], Lm["down"] = [Ld["fgate"]], [Ld["fup"]], [Ld["fdown"]]
    od, om = oracle.Oracle(md), oracle.Oracle(mm)
    kd, km = od.new_kv(8), om.new_kv(8)
    rd = od.decode_step(kd, 0, token=9)
    rm = om.decode_step(km, 0, token=9)
    assert np.array_equal(rd["logits"], rm["logits"])


def test_identical_experts_make_routing_irrelevant():
    cfg = TINY_MOE.replace(n_layers=1)
    m = synth.gen_model(cfg, seed=5)
    L = m["layers"][0]
    for k in ("gate", "up", "down"):
        L[k] = [L[k][0]] * cfg.n_experts
    orc = oracle.Oracle(m)
    kv = orc.new_kv(8)
    out = orc.decode_step(kv, 0, token=3, want_trace=True)
    # Same model with the router replaced by another random matrix: routing changes, output not.
    m2 = dict(m)
    m2["layers"] = [dict(L)]
    m2["layers"][0]["router"] = synth.fp8_matrix(cfg.n_experts, cfg.hidden, "cpu", 99, "r2")
    o2 = oracle.Oracle(m2)
    kv2 = o2.new_kv(8)
    out2 = o2.decode_step(kv2, 0, token=3, want_trace=True)
    assert not np.array_equal(out["trace"]["topk_idx"], out2["trace"]["topk_idx"])
    assert np.allclose(out["logits"], out2["logits"], rtol=0, atol=1e-12)


def test_positions_out_of_cache_are_rejected():
    m = synth.gen_model(synth.TINY.replace(n_layers=1), seed=6)
    orc = oracle.Oracle(m)
    kv = orc.new_kv(4)
    with pytest.raises(ValueError):
        orc.decode_step(kv, 4, token=1)


def test_zero_sublayers_keep_the_residual_stream():
    """With W_o = 0 and W_down = 0 every layer adds nothing: x_{l+1} = x_l, so the logits equal the
    zero-layer model's (catches a dropped or doubled residual)."""
    cfg = synth.TINY.replace(n_layers=2)
    m = synth.gen_model(cfg, seed=7)
    zero = lambda ws: (torch.zeros_like(ws[0]), ws[1])
    for L in m["layers"]:
        L["wo"], L["fdown"] = zero(L["wo"]), zero(L["fdown"])
    orc = oracle.Oracle(m)
    kv = orc.new_kv(8)
    out = orc.decode_step(kv, 0, token=11)
    m0 = dict(m)
    m0["cfg"] = cfg.replace(n_layers=0)
    m0["layers"] = []
    o0 = oracle.Oracle(m0)
    out0 = o0.decode_step(o0.new_kv(8), 0, token=11)
    assert np.array_equal(out["logits"], out0["logits"])


def test_oracle_threads_do_not_change_results():
    """The matrix-vector rows may run on several host threads; every result is bit-identical."""
    m = synth.gen_model(TINY_MOE, seed=8)
    orc = oracle.Oracle(m)
    outs = []
    for threads in (1, 3):
        oracle.set_threads(threads)
        kv = orc.new_kv(16)
        outs.append(orc.prefill(kv, synth.gen_tokens(5, TINY_MOE.vocab, seed=8)))
    oracle.set_threads(oracle.max_threads())
    assert np.array_equal(outs[0]["logits"], outs[1]["logits"])
    assert np.array_equal(outs[0]["hidden"], outs[1]["hidden"])
