"""Host-side checks of what bench.py reports besides the timings (no GPU).

* The algorithmic bytes a decode launch must move, against the sizes of the synthetic model's own
  tensors: every FP8 weight matrix the step reads (codes plus fp32 block scales) and the KV rows
  it attends over and appends, taken from the generators' outputs rather than from a formula.
* The staleness gate of the committed DRAM-traffic record: the ncu figure is reported only while
  the kernel sources hash to the value the counters were taken at.
"""
import json
import os

import bench
from latency_moe_decode_gb300 import synth

CFG = synth.ModelCfg(n_layers=2, hidden=512, n_heads=8, n_kv_heads=2, head_dim=128, n_experts=16,
                     top_k=4, moe_inter=256, n_shared=1, vocab=2048, max_ctx=512, max_batch=8,
                     rms_eps=1e-6, rope_theta=1e6)


def _nbytes(mat):
    codes, scales = mat
    return codes.numel() * codes.element_size() + scales.numel() * scales.element_size()


def test_algorithmic_bytes_match_the_model_tensors():
    m = synth.gen_model(CFG, seed=0)
    distinct = [3, 7]  # distinct routed experts per layer of one step
    ctx = [100, 37]    # the context of each of the step's tokens (two sequences)
    expect = _nbytes(m["lm_head"])
    for l, L in enumerate(m["layers"]):
        expect += sum(_nbytes(L[k]) for k in ("wq", "wk", "wv", "wo", "router"))
        expert = _nbytes(L["gate"][0]) + _nbytes(L["up"][0]) + _nbytes(L["down"][0])
        assert all(_nbytes(L["gate"][e]) + _nbytes(L["up"][e]) + _nbytes(L["down"][e]) == expert
                   for e in range(CFG.n_experts))
        expect += distinct[l] * expert
        expect += sum(_nbytes(L[k][s]) for k in ("sgate", "sup", "sdown") for s in range(CFG.n_shared))
    # KV: every cached position of each token's sequence plus its new row is read, the new row written
    k, v = synth.gen_kv(CFG, 10, seed=1)
    row = (k.numel() * k.element_size() + v.numel() * v.element_size()) // 10  # all layers, one position
    expect += sum((t + 1) * row for t in ctx) + len(ctx) * row
    assert bench.algorithmic_bytes(CFG, distinct, ctx, len(ctx)) == expect


def test_weight_bytes_per_token_match_the_model_tensors():
    m = synth.gen_model(CFG, seed=0)
    L = m["layers"][0]
    wb = synth.weight_bytes_per_token(CFG)
    assert wb["attn"] == sum(_nbytes(L[k]) for k in ("wq", "wk", "wv", "wo"))
    assert wb["router"] == _nbytes(L["router"])
    assert wb["lm_head"] == _nbytes(m["lm_head"])


def test_traffic_record_only_on_the_sources_it_was_taken_on(monkeypatch):
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "dram_traffic_per_launch.json")))
    for workload, e in rec.items():
        if workload.startswith("_"):
            continue
        assert e["dram_bytes_per_launch"] == e["dram_bytes_read_per_launch"] + e["dram_bytes_write_per_launch"]
        monkeypatch.setattr(bench, "csrc_hash", lambda: e["csrc_hash"])
        assert bench.profile_traffic(workload) == e["dram_bytes_per_launch"]
        monkeypatch.setattr(bench, "csrc_hash", lambda: "0" * 16)
        assert bench.profile_traffic(workload) is None
    assert bench.profile_traffic("no_such_workload") is None
