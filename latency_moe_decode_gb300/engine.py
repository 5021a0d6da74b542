"""Python face of the decode engine: torch tensors in, C ABI calls out.

PyTorch only provides device memory and streams here; every step of the decode path runs in the
engine's CUDA kernels behind include/dec.h.
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, Optional

import numpy as np
import torch

from . import capi
from .capi import DecCtx, DecError, DecFp8Mat, DecInfo, DecLayerWeights, DecModelCfg, DecStepArgs, DecWeights


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


CUDA_STREAM_LEGACY = 1  # cudaStreamLegacy: the context's legacy default stream


def _stream_ptr(stream) -> Optional[int]:
    """C-ABI stream handle. torch's default stream has handle 0, which the C ABI reads as "the
    engine's own stream", so it is passed as cudaStreamLegacy instead."""
    if stream is None:
        return None
    h = stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)
    return h if h != 0 else CUDA_STREAM_LEGACY


class Engine:
    """One engine = one model's repacked weights, KV cache and workspace on the current GPU."""

    def __init__(self, model: Dict, max_ctx: Optional[int] = None, max_batch: Optional[int] = None, stream=None):
        self.lib = capi.lib()
        cfg = model["cfg"]
        if max_ctx is not None:
            cfg = cfg.replace(max_ctx=max_ctx)
        if max_batch is not None:
            cfg = cfg.replace(max_batch=max_batch)
        self.cfg = cfg
        c = DecModelCfg(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.n_experts,
                        cfg.top_k, cfg.moe_inter, cfg.n_shared, cfg.dense_ffn, cfg.vocab, cfg.max_ctx,
                        cfg.max_batch, cfg.rms_eps, cfg.rope_theta)
        keep = []

        def mat(ws) -> DecFp8Mat:
            w, s = ws
            assert w.is_cuda and w.dtype == torch.uint8 and w.is_contiguous()
            s = s.contiguous().float()
            keep.append(s)
            return DecFp8Mat(w.data_ptr(), s.data_ptr())

        def mats(lst):
            arr = (DecFp8Mat * max(1, len(lst)))(*[mat(x) for x in lst])
            keep.append(arr)
            return C.cast(arr, C.POINTER(DecFp8Mat))

        layers = (DecLayerWeights * cfg.n_layers)()
        for i, L in enumerate(model["layers"]):
            o = layers[i]
            o.attn_norm = L["attn_norm"].data_ptr()
            o.ffn_norm = L["ffn_norm"].data_ptr()
            o.wq, o.wk, o.wv, o.wo = mat(L["wq"]), mat(L["wk"]), mat(L["wv"]), mat(L["wo"])
            if cfg.dense_ffn > 0:
                o.ffn_gate, o.ffn_up, o.ffn_down = mat(L["fgate"]), mat(L["fup"]), mat(L["fdown"])
            else:
                o.router = mat(L["router"])
                o.expert_gate, o.expert_up, o.expert_down = mats(L["gate"]), mats(L["up"]), mats(L["down"])
                if cfg.n_shared:
                    o.shared_gate, o.shared_up, o.shared_down = mats(L["sgate"]), mats(L["sup"]), mats(L["sdown"])
        w = DecWeights()
        w.layers = C.cast(layers, C.POINTER(DecLayerWeights))
        if cfg.vocab > 0:
            w.embed = model["embed"].data_ptr()
            w.final_norm = model["final_norm"].data_ptr()
            w.lm_head = mat(model["lm_head"])
        h = C.c_void_p()
        if stream is None:
            stream = torch.cuda.current_stream()
        st = self.lib.dec_init(C.byref(c), C.byref(w), _stream_ptr(stream), C.byref(h))
        if st != capi.DEC_OK:
            raise DecError(st, "dec_init")
        self.h = h
        del keep

    # ---- error plumbing
    def _check(self, st: int, where: str):
        if st != capi.DEC_OK:
            raise DecError(st, where, self.lib.dec_last_error(self.h).decode())

    def close(self):
        if getattr(self, "h", None):
            self.lib.dec_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- API
    def prefill_tokens(self, tokens: torch.Tensor, seq: int = 0):
        """tokens: device int32 [n_seq, n] (or [n] for one slot)."""
        t = tokens.to(torch.int32)
        if t.dim() == 1:
            t = t[None]
        t = t.contiguous()
        ctx = DecCtx(seq, t.shape[0], t.data_ptr(), t.shape[1], None, None)
        self._check(self.lib.dec_prefill_kv(self.h, C.byref(ctx)), "dec_prefill_kv")

    def prefill_tokens_noalloc(self, tokens: torch.Tensor, seq: int = 0):
        """As prefill_tokens, through dec_prefill_kv_noalloc (ids staged in the library's static
        device scratch; at most DEC_NOALLOC_PREFILL_MAX_IDS ids per call). tokens must already be
        a contiguous device int32 tensor: this wrapper makes no copy."""
        if tokens.dtype != torch.int32 or not tokens.is_contiguous():
            raise ValueError("tokens must be a contiguous int32 device tensor")
        t = tokens if tokens.dim() == 2 else tokens[None]
        ctx = DecCtx(seq, t.shape[0], t.data_ptr(), t.shape[1], None, None)
        self._check(self.lib.dec_prefill_kv_noalloc(self.h, C.byref(ctx)), "dec_prefill_kv_noalloc")

    def prefill_import(self, k: torch.Tensor, v: torch.Tensor, seq: int = 0, n_seq: int = 1):
        """k, v: device bf16 [n_layers, n_kv_heads, n, head_dim]."""
        k, v = k.contiguous(), v.contiguous()
        ctx = DecCtx(seq, n_seq, None, k.shape[2], k.data_ptr(), v.data_ptr())
        self._check(self.lib.dec_prefill_kv(self.h, C.byref(ctx)), "dec_prefill_kv")

    def step(self, tokens: Optional[torch.Tensor] = None, hidden: Optional[torch.Tensor] = None,
             batch: Optional[int] = None, seq0: int = 0, logits: Optional[torch.Tensor] = None,
             next_tokens: Optional[torch.Tensor] = None, hidden_out: Optional[torch.Tensor] = None, stream=None):
        if batch is None:
            batch = (tokens if tokens is not None else hidden).shape[0]
        a = DecStepArgs(_ptr(tokens), _ptr(hidden), batch, seq0, _ptr(logits), _ptr(next_tokens), _ptr(hidden_out),
                        _stream_ptr(stream if stream is not None else torch.cuda.current_stream()))
        self._check(self.lib.dec_step_ex(self.h, C.byref(a)), "dec_step_ex")

    def step_positions(self, tokens: torch.Tensor, seq: int = 0, logits: Optional[torch.Tensor] = None,
                       next_tokens: Optional[torch.Tensor] = None, stream=None):
        """Consecutive positions of one sequence in one launch (device int32 tokens [n])."""
        t = tokens.to(torch.int32).contiguous()
        self._check(self.lib.dec_step_positions(self.h, seq, t.data_ptr(), t.numel(), _ptr(logits), _ptr(next_tokens),
                                                _stream_ptr(stream if stream is not None else torch.cuda.current_stream())),
                    "dec_step_positions")

    def verify(self, tokens: torch.Tensor, seq: int = 0, logits: Optional[torch.Tensor] = None,
               next_tokens: Optional[torch.Tensor] = None, stream=None) -> int:
        """Speculative verify step: tokens = [next input, drafts...]; returns the accepted count."""
        t = tokens.to(torch.int32).contiguous()
        acc = C.c_int32()
        self._check(self.lib.dec_verify(self.h, seq, t.data_ptr(), t.numel(), _ptr(logits), _ptr(next_tokens),
                                        C.byref(acc),
                                        _stream_ptr(stream if stream is not None else torch.cuda.current_stream())),
                    "dec_verify")
        return acc.value

    def generate(self, first_tokens, n_steps: int, stream=None) -> np.ndarray:
        """Greedy decode from host tokens; returns host int32 [n_steps, batch]."""
        first = np.ascontiguousarray(np.asarray(first_tokens, np.int32).reshape(-1))
        out = np.zeros((n_steps, len(first)), np.int32)
        self._check(self.lib.dec_generate(self.h, first.ctypes.data, len(first), n_steps, out.ctypes.data,
                                          _stream_ptr(stream)), "dec_generate")
        return out

    def generate_pinned(self, first: torch.Tensor, out: torch.Tensor, stream=None):
        """Same as generate() with caller-provided (pinned) host tensors: first int32 [batch],
        out int32 [n_steps, batch]."""
        self._check(self.lib.dec_generate(self.h, first.data_ptr(), first.numel(), out.shape[0], out.data_ptr(),
                                          _stream_ptr(stream)), "dec_generate")

    def generate_device(self, first: torch.Tensor, out: torch.Tensor, stream=None):
        """Resident greedy generation with device tensors: first int32 [batch], out int32
        [n_steps, batch]; one launch, queued on the stream, not synchronised."""
        self._check(self.lib.dec_generate_device(self.h, first.data_ptr(), first.numel(), out.shape[0], out.data_ptr(),
                                                 _stream_ptr(stream if stream is not None else torch.cuda.current_stream())),
                    "dec_generate_device")

    def set_length(self, seq: int, length: int):
        self._check(self.lib.dec_set_length(self.h, seq, length), "dec_set_length")

    def get_length(self, seq: int) -> int:
        n = C.c_int32()
        self._check(self.lib.dec_get_length(self.h, seq, C.byref(n)), "dec_get_length")
        return n.value

    def export_kv(self, seq: int, layer: int, pos0: int, n: int):
        c = self.cfg
        k = torch.empty(c.n_kv_heads, n, c.head_dim, dtype=torch.bfloat16, device="cuda")
        v = torch.empty_like(k)
        self._check(self.lib.dec_export_kv(self.h, seq, layer, pos0, n, k.data_ptr(), v.data_ptr()), "dec_export_kv")
        return k, v

    def sync(self):
        torch.cuda.synchronize()
        self._check(self.lib.dec_sync(self.h), "dec_sync")

    def info(self) -> Dict:
        i = DecInfo()
        self._check(self.lib.dec_get_info(self.h, C.byref(i)), "dec_get_info")
        return {f: getattr(i, f) for f, _ in DecInfo._fields_}

    @property
    def rows(self) -> int:
        """Token rows of the routing records: max(DEC_MAX_STEP_TOKENS, max_batch)."""
        return max(capi.DEC_MAX_STEP_TOKENS, self.cfg.max_batch)

    def routing(self, layer: int):
        c = self.cfg
        idx = np.zeros((self.rows, c.top_k), np.int32)
        gates = np.zeros((self.rows, c.top_k), np.float32)
        self._check(self.lib.dec_get_routing(self.h, layer, idx.ctypes.data, gates.ctypes.data), "dec_get_routing")
        return idx, gates

    def router_logits(self, layer: int) -> np.ndarray:
        c = self.cfg
        out = np.zeros((self.rows, c.n_experts), np.float32)
        self._check(self.lib.dec_get_router_logits(self.h, layer, out.ctypes.data), "dec_get_router_logits")
        return out

    def layer_times(self) -> np.ndarray:
        """Timestamps (ns) of the most recent step: input of layer l final, l = 0..n_layers, then
        the step's end (first CTA's view)."""
        n = self.cfg.n_layers + 2
        buf = (C.c_uint64 * n)()
        got = C.c_int32()
        self._check(self.lib.dec_get_layer_times(self.h, buf, n, C.byref(got)), "dec_get_layer_times")
        return np.array(buf[:got.value], dtype=np.uint64)

    def trace(self, n: int = 64) -> np.ndarray:
        buf = (C.c_uint64 * n)()
        got = C.c_int32()
        self._check(self.lib.dec_get_trace(self.h, buf, n, C.byref(got)), "dec_get_trace")
        return np.array(buf[:got.value], dtype=np.uint64)


def validate_cfg(cfg) -> int:
    c = DecModelCfg(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.n_experts, cfg.top_k,
                    cfg.moe_inter, cfg.n_shared, cfg.dense_ffn, cfg.vocab, cfg.max_ctx, cfg.max_batch, cfg.rms_eps,
                    cfg.rope_theta)
    return capi.lib().dec_validate_cfg(C.byref(c))
