"""ctypes binding of the C ABI in include/dec.h (argument marshalling only).

Every entry point of the header is bound here under the same name. The shared library is built
in-tree (latency_moe_decode_gb300/libdec.so); importing this module without it raises -- there
is no CPU path to fall back to.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdec.so")

DEC_OK = 0
DEC_MAX_STEP_TOKENS = 8  # include/dec.h
STATUS = {0: "DEC_OK", -1: "DEC_ERR_ARG", -2: "DEC_ERR_CUDA", -3: "DEC_ERR_OOM", -4: "DEC_ERR_TIMEOUT",
          -5: "DEC_ERR_UNSUPPORTED", -6: "DEC_ERR_POISONED", -7: "DEC_ERR_DEVICE", -8: "DEC_ERR_CAPACITY"}


class DecModelCfg(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("n_layers", "hidden", "n_heads", "n_kv_heads", "head_dim", "n_experts",
                                         "top_k", "moe_inter", "n_shared", "dense_ffn", "vocab", "max_ctx",
                                         "max_batch")] + [("rms_eps", C.c_float), ("rope_theta", C.c_float)]


class DecFp8Mat(C.Structure):
    _fields_ = [("w", C.c_void_p), ("scale", C.c_void_p)]


class DecLayerWeights(C.Structure):
    _fields_ = [("attn_norm", C.c_void_p), ("wq", DecFp8Mat), ("wk", DecFp8Mat), ("wv", DecFp8Mat),
                ("wo", DecFp8Mat), ("ffn_norm", C.c_void_p), ("router", DecFp8Mat),
                ("expert_gate", C.POINTER(DecFp8Mat)), ("expert_up", C.POINTER(DecFp8Mat)),
                ("expert_down", C.POINTER(DecFp8Mat)), ("shared_gate", C.POINTER(DecFp8Mat)),
                ("shared_up", C.POINTER(DecFp8Mat)), ("shared_down", C.POINTER(DecFp8Mat)),
                ("ffn_gate", DecFp8Mat), ("ffn_up", DecFp8Mat), ("ffn_down", DecFp8Mat)]


class DecWeights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("final_norm", C.c_void_p), ("lm_head", DecFp8Mat),
                ("layers", C.POINTER(DecLayerWeights))]


class DecCtx(C.Structure):
    _fields_ = [("seq", C.c_int32), ("n_seq", C.c_int32), ("token_ids", C.c_void_p), ("n_tokens", C.c_int32),
                ("k_import", C.c_void_p), ("v_import", C.c_void_p)]


class DecStepArgs(C.Structure):
    _fields_ = [("tokens", C.c_void_p), ("hidden_in", C.c_void_p), ("batch", C.c_int32), ("seq0", C.c_int32),
                ("logits", C.c_void_p), ("next_tokens", C.c_void_p), ("hidden_out", C.c_void_p),
                ("stream", C.c_void_p)]


class DecInfo(C.Structure):
    _fields_ = [("grid", C.c_int32), ("threads", C.c_int32), ("smem_bytes", C.c_int32), ("ring_slots", C.c_int32),
                ("stages_per_layer", C.c_int32), ("weight_bytes", C.c_int64), ("kv_bytes", C.c_int64),
                ("workspace_bytes", C.c_int64), ("launches", C.c_int64), ("wide_min_batch", C.c_int32)]


# name -> (restype, argtypes); the exported surface of dec.h
PROTOTYPES = {
    "dec_validate_cfg": (C.c_int, [C.POINTER(DecModelCfg)]),
    "dec_init": (C.c_int, [C.POINTER(DecModelCfg), C.POINTER(DecWeights), C.c_void_p, C.POINTER(C.c_void_p)]),
    "dec_prefill_kv": (C.c_int, [C.c_void_p, C.POINTER(DecCtx)]),
    "dec_prefill_kv_noalloc": (C.c_int, [C.c_void_p, C.POINTER(DecCtx)]),
    "dec_step_ex": (C.c_int, [C.c_void_p, C.POINTER(DecStepArgs)]),
    "dec_step": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p]),
    "dec_step_positions": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p,
                                     C.c_void_p]),
    "dec_verify": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p,
                             C.POINTER(C.c_int32), C.c_void_p]),
    "dec_generate": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]),
    "dec_generate_device": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]),
    "dec_set_length": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32]),
    "dec_get_length": (C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_int32)]),
    "dec_export_kv": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]),
    "dec_sync": (C.c_int, [C.c_void_p]),
    "dec_get_info": (C.c_int, [C.c_void_p, C.POINTER(DecInfo)]),
    "dec_get_routing": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]),
    "dec_get_router_logits": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p]),
    "dec_get_trace": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint64), C.c_int32, C.POINTER(C.c_int32)]),
    "dec_get_layer_times": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint64), C.c_int32, C.POINTER(C.c_int32)]),
    "dec_last_error": (C.c_char_p, [C.c_void_p]),
    "dec_status_string": (C.c_char_p, [C.c_int]),
    "dec_destroy": (None, [C.c_void_p]),
}

_lib = None


def lib(build_if_missing: bool = False):
    """Load libdec.so (optionally building it first). Raises if it is missing."""
    global _lib
    if _lib is None:
        if build_if_missing:
            from . import build as _build
            _build.build()
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with latency_moe_decode_gb300.build.build(); "
                               "the decode step has no CPU fallback")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in PROTOTYPES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class DecError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} {detail}".strip())
