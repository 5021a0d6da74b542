"""Seeded synthetic inputs for the MoE decode step: weights, prompts, KV states, hidden inputs.

This module only draws random numbers and packs them into the storage formats the decode step
consumes (FP8-E4M3 bytes with 128x128 fp32 block scales, bf16 tensors, int32 token ids). It holds
none of the decode arithmetic. Both the GPU engine (through the tests and the benchmark) and the
CPU oracle are fed from the same realised tensors.

Recipe (the model configurations of the workloads):
  * linear weights W ~ N(0, 0.02), quantised per 128x128 block: scale = amax / 448 (1 if the
    block is all zero), code = round-to-nearest-even(W / scale) in E4M3; partial edge blocks
    use the rows/columns that exist;
  * embeddings bf16 N(0, 0.02); RMSNorm weights bf16 ones;
  * prompts: token ids uniform in [0, vocab);
  * imported KV states and hidden inputs: bf16 N(0, 1).
Every tensor has its own generator seeded from (base seed, tensor name), so a tensor does not
change when another is added, and distinct layers and experts never share weights.
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Dict, List, Optional

import torch

E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class ModelCfg:
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    n_experts: int = 0
    top_k: int = 0
    moe_inter: int = 0
    n_shared: int = 0
    dense_ffn: int = 0
    vocab: int = 0
    max_ctx: int = 256
    max_batch: int = 1
    rms_eps: float = 1e-6
    rope_theta: float = 10000.0

    def replace(self, **kw) -> "ModelCfg":
        return dataclasses.replace(self, **kw)


# The workloads. "tiny": a 2-layer dense decoder (hidden 256, 4 query / 2 KV heads of 64,
# SwiGLU FFN 512, vocab 1024). "moe_layer": one MoE decoder layer (hidden 4096, 32 query / 8 KV
# heads of 128, 64 routed SwiGLU experts of 1536 with top-8 sigmoid routing and one shared
# expert), RoPE theta 1e6. "moe8": eight such layers with a 32000-token vocabulary.
TINY = ModelCfg(n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, dense_ffn=512,
                vocab=1024, max_ctx=256, max_batch=1, rms_eps=1e-6, rope_theta=10000.0)
MOE_LAYER = ModelCfg(n_layers=1, hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128,
                     n_experts=64, top_k=8, moe_inter=1536, n_shared=1, vocab=0,
                     max_ctx=8192 + 64, max_batch=1, rms_eps=1e-6, rope_theta=1e6)
MOE8 = MOE_LAYER.replace(n_layers=8, vocab=32000, max_ctx=2048 + 64)


def _seed(base: int, name: str) -> int:
    return (zlib.crc32(name.encode()) ^ (base * 0x9E3779B1)) & 0x7FFFFFFFFFFF


def _gen(device, base: int, name: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(base, name))
    return g


def quantize_fp8_blocks(w: torch.Tensor):
    """Quantise a float matrix [n, k] to E4M3 codes with one fp32 scale per 128x128 block.
    Returns (codes uint8 [n, k], scales float32 [ceil(n/128), ceil(k/128)])."""
    n, k = w.shape
    nb, kb = (n + 127) // 128, (k + 127) // 128
    wp = torch.zeros(nb * 128, kb * 128, dtype=torch.float32, device=w.device)
    wp[:n, :k] = w.float()
    blk = wp.view(nb, 128, kb, 128)
    amax = blk.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = (blk / scale[:, None, :, None]).clamp_(-E4M3_MAX, E4M3_MAX)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8).view(nb * 128, kb * 128)[:n, :k]
    return codes.contiguous(), scale.float().contiguous()


def fp8_matrix(n: int, k: int, device, base: int, name: str, std: float = 0.02):
    w = torch.randn(n, k, generator=_gen(device, base, name), device=device, dtype=torch.float32)
    return quantize_fp8_blocks(w * std)


def gen_model(cfg: ModelCfg, seed: int = 0, device="cpu") -> Dict:
    """Random-init weights of the given architecture (no trained weights exist here)."""
    dev = torch.device(device)
    d, hd = cfg.hidden, cfg.head_dim
    ones = torch.ones(d, dtype=torch.bfloat16, device=dev)
    m: Dict = {"cfg": cfg, "layers": []}
    if cfg.vocab > 0:
        m["embed"] = (torch.randn(cfg.vocab, d, generator=_gen(dev, seed, "embed"), device=dev)
                      * 0.02).to(torch.bfloat16)
        m["final_norm"] = ones.clone()
        m["lm_head"] = fp8_matrix(cfg.vocab, d, dev, seed, "lm_head")
    for l in range(cfg.n_layers):
        p = f"L{l}."
        L = {
            "attn_norm": ones.clone(),
            "ffn_norm": ones.clone(),
            "wq": fp8_matrix(cfg.n_heads * hd, d, dev, seed, p + "wq"),
            "wk": fp8_matrix(cfg.n_kv_heads * hd, d, dev, seed, p + "wk"),
            "wv": fp8_matrix(cfg.n_kv_heads * hd, d, dev, seed, p + "wv"),
            "wo": fp8_matrix(d, cfg.n_heads * hd, dev, seed, p + "wo"),
        }
        if cfg.dense_ffn > 0:
            f = cfg.dense_ffn
            L["fgate"] = fp8_matrix(f, d, dev, seed, p + "fgate")
            L["fup"] = fp8_matrix(f, d, dev, seed, p + "fup")
            L["fdown"] = fp8_matrix(d, f, dev, seed, p + "fdown")
        else:
            i = cfg.moe_inter
            L["router"] = fp8_matrix(cfg.n_experts, d, dev, seed, p + "router")
            L["gate"] = [fp8_matrix(i, d, dev, seed, p + f"e{e}.gate") for e in range(cfg.n_experts)]
            L["up"] = [fp8_matrix(i, d, dev, seed, p + f"e{e}.up") for e in range(cfg.n_experts)]
            L["down"] = [fp8_matrix(d, i, dev, seed, p + f"e{e}.down") for e in range(cfg.n_experts)]
            L["sgate"] = [fp8_matrix(i, d, dev, seed, p + f"s{s}.gate") for s in range(cfg.n_shared)]
            L["sup"] = [fp8_matrix(i, d, dev, seed, p + f"s{s}.up") for s in range(cfg.n_shared)]
            L["sdown"] = [fp8_matrix(d, i, dev, seed, p + f"s{s}.down") for s in range(cfg.n_shared)]
        m["layers"].append(L)
    return m


def model_to(m: Dict, device) -> Dict:
    """Copy every tensor of a model dict to another device (e.g. the GPU copy for the oracle)."""
    def mv(v):
        if isinstance(v, torch.Tensor):
            return v.to(device)
        if isinstance(v, tuple):
            return tuple(mv(x) for x in v)
        if isinstance(v, list):
            return [mv(x) for x in v]
        if isinstance(v, dict):
            return {k: mv(x) for k, x in v.items()}
        return v
    return mv(m)


def gen_tokens(n: int, vocab: int, seed: int, device="cpu") -> torch.Tensor:
    return torch.randint(0, vocab, (n,), generator=_gen(torch.device(device), seed, f"tokens{n}"),
                         device=device, dtype=torch.int64).to(torch.int32)


def gen_kv(cfg: ModelCfg, n_pos: int, seed: int, device="cpu"):
    """A synthetic imported KV state: K and V bf16 N(0,1), [n_layers][n_kv_heads][n_pos][head_dim]."""
    shape = (cfg.n_layers, cfg.n_kv_heads, n_pos, cfg.head_dim)
    dev = torch.device(device)
    k = torch.randn(*shape, generator=_gen(dev, seed, f"kvK{n_pos}"), device=dev).to(torch.bfloat16)
    v = torch.randn(*shape, generator=_gen(dev, seed, f"kvV{n_pos}"), device=dev).to(torch.bfloat16)
    return k, v


def gen_hidden(batch: int, hidden: int, seed: int, device="cpu") -> torch.Tensor:
    dev = torch.device(device)
    return torch.randn(batch, hidden, generator=_gen(dev, seed, f"hidden{batch}"), device=dev).to(torch.bfloat16)


def weight_bytes_per_token(cfg: ModelCfg) -> Dict[str, float]:
    """Algorithmic bytes one batch-1 decode token must stream (weights + scales), by part."""
    d, hd = cfg.hidden, cfg.head_dim

    def mat(n, k):
        return n * k + 4 * ((n + 127) // 128) * ((k + 127) // 128)

    attn = mat((cfg.n_heads + 2 * cfg.n_kv_heads) * hd, d) + mat(d, cfg.n_heads * hd)
    if cfg.dense_ffn > 0:
        ffn = 2 * mat(cfg.dense_ffn, d) + mat(d, cfg.dense_ffn)
        router = 0
    else:
        expert = 2 * mat(cfg.moe_inter, d) + mat(d, cfg.moe_inter)
        ffn = (cfg.top_k + cfg.n_shared) * expert
        router = mat(cfg.n_experts, d)
    lm = mat(cfg.vocab, d) if cfg.vocab > 0 else 0
    return {"attn": attn, "router": router, "ffn": ffn, "per_layer": attn + router + ffn,
            "lm_head": lm, "total": cfg.n_layers * (attn + router + ffn) + lm}
