"""CPU oracle of the MoE decode step (ctypes binding of oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the test suite, by the smoke check and by the benchmark's
CPU-baseline and reference legs. The GPU engine never imports it. Inputs are numpy arrays (or CPU torch tensors)
of the storage formats the decode step consumes: FP8-E4M3 codes (uint8) with fp32 block scales,
bf16 values as uint16 bit patterns, int32 token ids. All arithmetic is in oracle.c (double).
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, List, Optional

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        L.orc_e4m3_value.restype = C.c_double
        L.orc_e4m3_value.argtypes = [C.c_uint8]
        L.orc_bf16_value.restype = C.c_double
        L.orc_bf16_value.argtypes = [C.c_uint16]
        L.orc_bf16_bits.restype = C.c_uint16
        L.orc_bf16_bits.argtypes = [C.c_double]
        L.orc_bf16_round.restype = C.c_double
        L.orc_bf16_round.argtypes = [C.c_double]
        L.orc_gemv.argtypes = [C.POINTER(OrcMat), C.c_void_p, C.c_void_p]
        L.orc_rmsnorm.argtypes = [C.c_void_p, C.c_void_p, C.c_int32, C.c_double, C.c_void_p]
        L.orc_rope.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_double]
        L.orc_attention_head.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int32,
                                         C.c_void_p]
        L.orc_router_topk.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                      C.c_void_p]
        L.orc_swiglu_expert.argtypes = [C.POINTER(OrcMat)] * 3 + [C.c_void_p, C.c_void_p]
        L.orc_layer_step.restype = C.c_int32
        L.orc_layer_step.argtypes = [C.POINTER(OrcModel), C.c_int32, C.c_void_p, C.c_int32,
                                     C.POINTER(OrcKV), C.POINTER(OrcTrace)]
        L.orc_decode_step.restype = C.c_int32
        L.orc_decode_step.argtypes = [C.POINTER(OrcModel), C.c_int32, C.c_void_p, C.c_int32,
                                      C.POINTER(OrcKV), C.c_void_p, C.c_void_p, C.POINTER(OrcTrace)]
        L.orc_full_recompute.restype = C.c_int32
        L.orc_full_recompute.argtypes = [C.POINTER(OrcModel), C.c_void_p, C.c_int32, C.c_void_p]
        L.orc_argmax.restype = C.c_int32
        L.orc_argmax.argtypes = [C.c_void_p, C.c_int32]
        L.orc_set_threads.argtypes = [C.c_int32]
        L.orc_max_threads.restype = C.c_int32
        _lib = L
    return _lib


class OrcMat(C.Structure):
    _fields_ = [("w", C.c_void_p), ("s", C.c_void_p), ("n", C.c_int32), ("k", C.c_int32)]


class OrcCfg(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim",
                                         "n_experts", "top_k", "moe_inter", "n_shared", "dense_ffn",
                                         "vocab")] + [("rms_eps", C.c_double), ("rope_theta", C.c_double)]


class OrcLayer(C.Structure):
    _fields_ = [("attn_norm", C.c_void_p), ("wq", OrcMat), ("wk", OrcMat), ("wv", OrcMat),
                ("wo", OrcMat), ("ffn_norm", C.c_void_p), ("router", OrcMat),
                ("gate", C.POINTER(OrcMat)), ("up", C.POINTER(OrcMat)), ("down", C.POINTER(OrcMat)),
                ("sgate", C.POINTER(OrcMat)), ("sup", C.POINTER(OrcMat)), ("sdown", C.POINTER(OrcMat)),
                ("fgate", OrcMat), ("fup", OrcMat), ("fdown", OrcMat)]


class OrcModel(C.Structure):
    _fields_ = [("cfg", OrcCfg), ("embed", C.c_void_p), ("final_norm", C.c_void_p),
                ("lm_head", OrcMat), ("layers", C.POINTER(OrcLayer))]


class OrcKV(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("max_ctx", C.c_int32)]


class OrcTrace(C.Structure):
    _fields_ = [("layer_out", C.c_void_p), ("topk_idx", C.c_void_p), ("topk_gate", C.c_void_p),
                ("router_score", C.c_void_p), ("attn_out", C.c_void_p)]


def _np(t):
    """numpy view of a CPU array/tensor; bf16 tensors become uint16 bit patterns."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16)
            return t.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(t)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class Oracle:
    """The oracle bound to one model (a dict as produced by latency_moe_decode_gb300.synth)."""

    def __init__(self, model: Dict):
        self.cfg = model["cfg"]
        self._keep: List = []
        c = self.cfg
        self.model = OrcModel()
        m = self.model
        m.cfg = OrcCfg(c.n_layers, c.hidden, c.n_heads, c.n_kv_heads, c.head_dim, c.n_experts,
                       c.top_k, c.moe_inter, c.n_shared, c.dense_ffn, c.vocab, c.rms_eps, c.rope_theta)
        if c.vocab > 0:
            m.embed = self._arr(model["embed"])
            m.final_norm = self._arr(model["final_norm"])
            m.lm_head = self._mat(model["lm_head"])
        layers = (OrcLayer * max(1, c.n_layers))()
        for i, L in enumerate(model["layers"]):
            o = layers[i]
            o.attn_norm = self._arr(L["attn_norm"])
            o.ffn_norm = self._arr(L["ffn_norm"])
            for nm in ("wq", "wk", "wv", "wo"):
                setattr(o, nm, self._mat(L[nm]))
            if c.dense_ffn > 0:
                for nm in ("fgate", "fup", "fdown"):
                    setattr(o, nm, self._mat(L[nm]))
            else:
                o.router = self._mat(L["router"])
                for nm in ("gate", "up", "down", "sgate", "sup", "sdown"):
                    arr = (OrcMat * max(1, len(L[nm])))(*[self._mat(x) for x in L[nm]])
                    self._keep.append(arr)
                    setattr(o, nm, C.cast(arr, C.POINTER(OrcMat)))
        self._keep.append(layers)
        m.layers = C.cast(layers, C.POINTER(OrcLayer))

    def _arr(self, t) -> int:
        a = _np(t)
        self._keep.append(a)
        return _ptr(a)

    def _mat(self, ws) -> OrcMat:
        w, s = _np(ws[0]), _np(ws[1]).astype(np.float32)
        self._keep += [w, s]
        return OrcMat(_ptr(w), _ptr(s), w.shape[0], w.shape[1])

    def new_kv(self, max_ctx: int):
        c = self.cfg
        shape = (c.n_layers, c.n_kv_heads, max_ctx, c.head_dim)
        return {"k": np.zeros(shape, np.uint16), "v": np.zeros(shape, np.uint16), "max_ctx": max_ctx}

    def import_kv(self, kv, k, v, n_pos: int):
        """Copy an external bf16 KV state [n_layers][n_kv_heads][n_pos][head_dim] into positions
        0..n_pos of a cache."""
        kv["k"][:, :, :n_pos] = _np(k)
        kv["v"][:, :, :n_pos] = _np(v)

    def decode_step(self, kv, pos: int, token: int = 0, hidden=None, want_logits=True,
                    want_trace=False):
        c = self.cfg
        okv = OrcKV(_ptr(kv["k"]), _ptr(kv["v"]), kv["max_ctx"])
        logits = np.zeros(max(1, c.vocab), np.float64) if (want_logits and c.vocab > 0) else None
        hout = np.zeros(c.hidden, np.uint16)
        hin = _np(hidden).reshape(-1).astype(np.uint16) if hidden is not None else None
        tr = OrcTrace()
        trace = None
        if want_trace:
            trace = {
                "layer_out": np.zeros((c.n_layers, c.hidden)),
                "topk_idx": np.zeros((c.n_layers, max(1, c.top_k)), np.int32),
                "topk_gate": np.zeros((c.n_layers, max(1, c.top_k))),
                "router_score": np.zeros((c.n_layers, max(1, c.n_experts))),
                "attn_out": np.zeros((c.n_layers, c.n_heads * c.head_dim)),
            }
            for k2, a in trace.items():
                setattr(tr, k2, _ptr(a))
        tok = lib().orc_decode_step(C.byref(self.model), int(token),
                                    _ptr(hin) if hin is not None else None, int(pos), C.byref(okv),
                                    _ptr(logits) if logits is not None else None, _ptr(hout),
                                    C.byref(tr))
        if tok == -2:
            raise ValueError("position outside the oracle's KV cache")
        return {"token": tok, "logits": logits, "hidden": hout, "trace": trace}

    def prefill(self, kv, tokens, start_pos: int = 0):
        """Incremental prefill: one decode step per prompt token. Returns the last step's result."""
        out = None
        for i, t in enumerate(_np(tokens).reshape(-1).tolist()):
            out = self.decode_step(kv, start_pos + i, token=int(t))
        return out

    def full_recompute(self, tokens):
        t = _np(tokens).astype(np.int32).reshape(-1)
        logits = np.zeros(self.cfg.vocab, np.float64)
        tok = lib().orc_full_recompute(C.byref(self.model), _ptr(t), len(t), _ptr(logits))
        return tok, logits


def set_threads(n: int) -> None:
    """Host threads for the rows of each matrix-vector product (results do not depend on it)."""
    lib().orc_set_threads(int(n))


def max_threads() -> int:
    return int(lib().orc_max_threads())


# ---- small helpers over the building blocks (used by the pin tests) ----

def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


def bf16_bits(v: float) -> int:
    return lib().orc_bf16_bits(v)


def bf16_value(bits: int) -> float:
    return lib().orc_bf16_value(bits)


def gemv(w: np.ndarray, s: np.ndarray, x: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w, np.uint8)
    s = np.ascontiguousarray(s, np.float32)
    x = np.ascontiguousarray(x, np.float64)
    y = np.zeros(w.shape[0], np.float64)
    m = OrcMat(_ptr(w), _ptr(s), w.shape[0], w.shape[1])
    lib().orc_gemv(C.byref(m), _ptr(x), _ptr(y))
    return y


def rmsnorm(x: np.ndarray, w_bits: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    w = np.ascontiguousarray(w_bits, np.uint16)
    out = np.zeros_like(x)
    lib().orc_rmsnorm(_ptr(x), _ptr(w), len(x), eps, _ptr(out))
    return out


def rope(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    v = np.array(v, np.float64)
    lib().orc_rope(_ptr(v), len(v), pos, theta)
    return v


def attention_head(q: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, np.float64)
    k = np.ascontiguousarray(k_bits, np.uint16)
    v = np.ascontiguousarray(v_bits, np.uint16)
    o = np.zeros(q.shape[0])
    lib().orc_attention_head(_ptr(q), _ptr(k), _ptr(v), k.shape[0], q.shape[0], _ptr(o))
    return o


def router_topk(logits: np.ndarray, top_k: int):
    r = np.ascontiguousarray(logits, np.float64)
    idx = np.zeros(top_k, np.int32)
    gate = np.zeros(top_k)
    score = np.zeros(len(r))
    lib().orc_router_topk(_ptr(r), len(r), top_k, _ptr(idx), _ptr(gate), _ptr(score))
    return idx, gate, score


def swiglu_expert(g, u, d, xn: np.ndarray) -> np.ndarray:
    mats = []
    keep = []
    for ws in (g, u, d):
        w, s = np.ascontiguousarray(ws[0], np.uint8), np.ascontiguousarray(ws[1], np.float32)
        keep += [w, s]
        mats.append(OrcMat(_ptr(w), _ptr(s), w.shape[0], w.shape[1]))
    xn = np.ascontiguousarray(xn, np.float64)
    y = np.zeros(d[0].shape[0])
    lib().orc_swiglu_expert(C.byref(mats[0]), C.byref(mats[1]), C.byref(mats[2]), _ptr(xn), _ptr(y))
    return y
