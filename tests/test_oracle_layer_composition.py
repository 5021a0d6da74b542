"""Pin of the oracle's layer composition: an independent float64 restatement of whole decode steps.

The building blocks of the oracle (E4M3 decode, bf16 rounding, blocked GEMV, RMSNorm, RoPE,
attention, router, SwiGLU) are pinned one by one in test_oracle_pins.py. This file pins how they
are put together into a layer and a step, which no single-block test sees: which residual stream
the FFN norm reads, the order of the residual adds, the shared expert's weight, the gate
normalisation, the GQA head mapping, the position the new key is rotated with, and the final
norm + LM head. The restatement below is written in numpy from the definition of a pre-norm MoE
decoder (every matrix dense-dequantised by torch, every product a numpy matmul, bf16 rounding
done by its own numpy routine), sharing nothing with oracle.c but the seeded inputs.

Sources: "vLLM's Kimi K3 Backend Hits 842 Tokens per Second", section "Four changes drive the
gains" (per layer: attention input projection, output projection + residual, router scores,
shared expert with the routed experts); "Kimi K3: The Manos, The Mythos, The Legendos" (GQA; the
expert as a SwiGLU; top-k over router scores; the residual x_{l+1} = x_l + f(x_l)). The readings
the pages leave open (half-split RoPE, bf16 rounding points, sigmoid router with gates normalised
over the selection, shared expert of weight 1) are the ones listed with the oracle.

Each plausible composition mistake is planted in a copy of the restatement and must move the
outputs far beyond the restatement's agreement with the oracle, so the pin would catch the same
mistake in the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from latency_moe_decode_gb300 import synth


def bf16(x):
    """Round float64 values to bf16 (8 significant bits, round half to even), once."""
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)  # x = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)  # bf16 subnormal spacing 2^-133
    return np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)


def dq(ws):
    """Dense float64 matrix of an (E4M3 codes, 128x128 block scales) pair, decoded by torch."""
    w = ws[0].view(torch.float8_e4m3fn).double().numpy()
    n, k = w.shape
    s = np.repeat(np.repeat(ws[1].double().numpy(), 128, 0), 128, 1)[:n, :k]
    return w * s


def bfv(t):
    return t.double().numpy()


class Restated:
    """One sequence's decode on the CPU in float64, step by step from the definition.

    Mutation switches (all off = the reading the oracle implements):
      ffn_norm_pre_residual  the FFN RMSNorm reads x before the attention residual is added
      shared_gated           the shared expert is scaled by the mean routed gate
      gates_unnormalised     routed gates are the raw sigmoid scores
      rope_interleaved       RoPE pairs (2i, 2i+1) instead of (i, i + hd/2)
      kv_head_modulo         query head h reads KV head h % n_kv instead of h // group
      no_final_norm          the LM head reads x without the final RMSNorm
    """

    def __init__(self, m, **mut):
        self.m = m
        self.c = m["cfg"]
        self.mut = mut
        self.L = []
        for L in m["layers"]:
            d = {k: dq(L[k]) for k in ("wq", "wk", "wv", "wo")}
            d["attn_norm"], d["ffn_norm"] = bfv(L["attn_norm"]), bfv(L["ffn_norm"])
            if self.c.dense_ffn:
                d["ffn"] = (dq(L["fgate"]), dq(L["fup"]), dq(L["fdown"]))
            else:
                d["router"] = dq(L["router"])
                d["experts"] = [(dq(g), dq(u), dq(w)) for g, u, w in zip(L["gate"], L["up"], L["down"])]
                d["shared"] = [(dq(g), dq(u), dq(w)) for g, u, w in zip(L["sgate"], L["sup"], L["sdown"])]
            self.L.append(d)
        if self.c.vocab:
            self.embed, self.final_norm, self.lm = bfv(m["embed"]), bfv(m["final_norm"]), dq(m["lm_head"])

    def rmsnorm(self, x, w):
        return bf16(x / np.sqrt(np.mean(x * x) + self.c.rms_eps) * w)

    def rope(self, v, pos):
        hd = v.shape[-1]
        i = np.arange(hd // 2)
        ang = pos * self.c.rope_theta ** (-2.0 * i / hd)
        c, s = np.cos(ang), np.sin(ang)
        out = v.copy()
        if self.mut.get("rope_interleaved"):
            a, b = v[..., 0::2], v[..., 1::2]
            out[..., 0::2], out[..., 1::2] = a * c - b * s, b * c + a * s
        else:
            a, b = v[..., : hd // 2], v[..., hd // 2:]
            out[..., : hd // 2], out[..., hd // 2:] = a * c - b * s, b * c + a * s
        return out

    @staticmethod
    def swiglu(e, xn):
        g, u, w = e
        a, b = g @ xn, u @ xn
        return w @ bf16(a / (1.0 + np.exp(-a)) * b)

    def step(self, kv, pos, token=None, hidden=None):
        """kv: {'k','v'} float64 [L][n_kv][max_ctx][hd] (bf16 values); writes position pos."""
        c = self.c
        hd, hq, hkv = c.head_dim, c.n_heads, c.n_kv_heads
        grp = hq // hkv
        x = self.embed[token].copy() if hidden is None else np.asarray(hidden, np.float64).copy()
        tr = {"layer_out": [], "attn_out": [], "topk_idx": [], "topk_gate": []}
        for l, W in enumerate(self.L):
            xn = self.rmsnorm(x, W["attn_norm"])
            q = self.rope((W["wq"] @ xn).reshape(hq, hd), pos)
            k = self.rope((W["wk"] @ xn).reshape(hkv, hd), pos)
            v = (W["wv"] @ xn).reshape(hkv, hd)
            q, k, v = bf16(q), bf16(k), bf16(v)
            kv["k"][l, :, pos], kv["v"][l, :, pos] = k, v
            o = np.zeros((hq, hd))
            for h in range(hq):
                g = h % hkv if self.mut.get("kv_head_modulo") else h // grp
                K, V = kv["k"][l, g, : pos + 1], kv["v"][l, g, : pos + 1]
                s = K @ q[h] / np.sqrt(hd)
                p = np.exp(s - s.max())
                o[h] = (p / p.sum()) @ V
            o = bf16(o.reshape(-1))
            tr["attn_out"].append(o)
            x_pre = x
            x = bf16(x + W["wo"] @ o)
            xn2 = self.rmsnorm(x_pre if self.mut.get("ffn_norm_pre_residual") else x, W["ffn_norm"])
            if c.dense_ffn:
                y = self.swiglu(W["ffn"], xn2)
            else:
                sc = 1.0 / (1.0 + np.exp(-(W["router"] @ xn2)))
                idx = np.argsort(-sc, kind="stable")[: c.top_k]  # descending, ties to the lower index
                gate = sc[idx] if self.mut.get("gates_unnormalised") else sc[idx] / sc[idx].sum()
                tr["topk_idx"].append(idx)
                tr["topk_gate"].append(gate)
                y = np.zeros(c.hidden)
                for gi, e in zip(gate, idx):
                    y += gi * self.swiglu(W["experts"][e], xn2)
                w_sh = float(np.mean(gate)) if self.mut.get("shared_gated") else 1.0
                for e in W["shared"]:
                    y += w_sh * self.swiglu(e, xn2)
            x = bf16(x + y)
            tr["layer_out"].append(x)
        logits = None
        if c.vocab:
            xf = bf16(x) if self.mut.get("no_final_norm") else self.rmsnorm(x, self.final_norm)
            logits = self.lm @ xf
        return x, logits, tr


TINY_MOE = synth.ModelCfg(n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, n_experts=8,
                          top_k=2, moe_inter=128, n_shared=1, vocab=512, max_ctx=64)
CTX = 20  # imported KV positions before the decoded ones


def _rel(a, b):
    a, b = np.asarray(a, np.float64).ravel(), np.asarray(b, np.float64).ravel()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _run_both(cfg, seed, n_steps, **mut):
    """Decode n_steps greedy tokens after a CTX-position synthetic KV state with the oracle and the
    restatement; the restatement is fed the oracle's tokens (teacher forcing)."""
    m = synth.gen_model(cfg, seed=seed)
    orc = oracle.Oracle(m)
    k, v = synth.gen_kv(cfg, CTX, seed=seed + 1)
    okv = orc.new_kv(cfg.max_ctx)
    orc.import_kv(okv, k, v, CTX)
    ref = Restated(m, **mut)
    rkv = {"k": np.zeros((cfg.n_layers, cfg.n_kv_heads, cfg.max_ctx, cfg.head_dim)),
           "v": np.zeros((cfg.n_layers, cfg.n_kv_heads, cfg.max_ctx, cfg.head_dim))}
    rkv["k"][:, :, :CTX], rkv["v"][:, :, :CTX] = bfv(k), bfv(v)
    out = []
    tok = 7
    for i in range(n_steps):
        o = orc.decode_step(okv, CTX + i, token=tok, want_trace=True)
        x, logits, tr = ref.step(rkv, CTX + i, token=tok)
        out.append((o, x, logits, tr))
        tok = o["token"]
    # the caches the two wrote
    okv_k = (okv["k"][:, :, : CTX + n_steps].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return out, okv_k, rkv["k"][:, :, : CTX + n_steps]


@pytest.mark.parametrize("cfg", [TINY_MOE, synth.TINY.replace(max_ctx=64)], ids=["moe_shared", "dense"])
def test_restated_steps_match_oracle(cfg):
    steps, ok_k, rk = _run_both(cfg, seed=11, n_steps=3)
    assert np.array_equal(ok_k, rk), "KV cache rows differ"
    for o, x, logits, tr in steps:
        bits = o["hidden"].astype(np.uint32) << 16
        assert _rel(x, bits.view(np.float32)) <= 1e-9
        assert _rel(logits, o["logits"]) <= 1e-9
        assert int(np.argmax(logits)) == o["token"]
        for l in range(cfg.n_layers):
            assert _rel(tr["layer_out"][l], o["trace"]["layer_out"][l]) <= 1e-9
            assert _rel(tr["attn_out"][l], o["trace"]["attn_out"][l]) <= 1e-9
            if cfg.n_experts:
                assert np.array_equal(tr["topk_idx"][l], o["trace"]["topk_idx"][l])
                assert np.allclose(tr["topk_gate"][l], o["trace"]["topk_gate"][l], rtol=1e-12, atol=0)


@pytest.mark.parametrize("mutation", ["ffn_norm_pre_residual", "shared_gated", "gates_unnormalised",
                                      "rope_interleaved", "kv_head_modulo", "no_final_norm"])
def test_each_composition_mistake_is_detected(mutation):
    """A restatement with one planted composition mistake disagrees with the oracle by orders of
    magnitude more than the faithful one (<= 1e-9), in the layer outputs or the logits."""
    steps, _, _ = _run_both(TINY_MOE, seed=11, n_steps=2, **{mutation: True})
    worst = 0.0
    for o, x, logits, tr in steps:
        worst = max(worst, _rel(logits, o["logits"]))
        for l in range(TINY_MOE.n_layers):
            worst = max(worst, _rel(tr["layer_out"][l], o["trace"]["layer_out"][l]))
    assert worst > 1e-3, f"{mutation}: only {worst:.2e} away from the oracle"
