"""ctypes binding of libdec (include/dec.h): argument marshalling only.

Every function keeps its C name and signature.  Loading fails loudly when the
library has not been built: there is no fallback of any kind.
"""

from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# DEC_DEBUG=1 in the environment loads the DEC_DEBUG build (device bounds checks) instead
LIB_PATH = os.path.join(_HERE, "libdec_debug.so" if os.environ.get("DEC_DEBUG") == "1" else "libdec.so")

DEC_OK, DEC_EINVAL, DEC_ECAPACITY, DEC_EBLOCK, DEC_ERANGE, DEC_EVOCAB, DEC_ECUDA, DEC_EDEVICE = range(8)
DEC_FP32, DEC_BF16_F16KV, DEC_INT4_F16KV = 0, 1, 2
DEC_ROWS_ALL, DEC_ROWS_LAST = 0, 1
DEC_DEV_BAD_ID, DEC_DEV_TIMEOUT, DEC_DEV_CAPACITY, DEC_DEV_BOUNDS = 1, 2, 4, 8
DEC_BUILD_DEBUG = 1
DEC_PURPOSE_SAMPLE = 4
DEC_SAMPLE_BAD_ID, DEC_SAMPLE_BAD_LOGIT, DEC_SAMPLE_NO_FINITE, DEC_SAMPLE_OVERFLOW = 1, 2, 4, 8

ERROR_NAMES = {0: "DEC_OK", 1: "DEC_EINVAL", 2: "DEC_ECAPACITY", 3: "DEC_EBLOCK", 4: "DEC_ERANGE",
               5: "DEC_EVOCAB", 6: "DEC_ECUDA", 7: "DEC_EDEVICE"}

# Every symbol include/dec.h declares (the tests check the library exports all of them).
EXPORTS = (
    "dec_last_error", "dec_config_check", "dec_weights_bytes", "dec_workspace_bytes", "dec_create", "dec_destroy",
    "dec_device_status", "dec_set_dump", "dec_pool_bytes", "dec_pool_create", "dec_pool_destroy", "dec_pool_alloc",
    "dec_pool_retain", "dec_pool_release", "dec_pool_free_blocks", "dec_pool_refcount", "dec_kv_offset",
    "dec_prefill", "dec_decode", "dec_f32_to_f16", "dec_version", "dec_profile_enable", "dec_profile_read",
    "dec_launch_count", "dec_set_graphs", "dec_set_megakernel", "dec_megakernel_available", "dec_set_step_trace",
    "dec_set_tensor_cores", "dec_debug_product", "dec_attend_scratch_bytes", "dec_attend", "dec_attend_noalloc",
    "dec_prefix_key", "dec_pool_set_fill", "dec_pool_register", "dec_pool_lookup", "dec_pool_cached_blocks",
    "dec_child_seed", "dec_rng_stream", "dec_rng_next_u32", "dec_rng_uniform", "dec_sampler_workspace_bytes",
    "dec_sampler_create", "dec_sampler_destroy", "dec_sampler_status", "dec_sample", "dec_debug_df_exp",
    "dec_quantize_int4", "dec_batch_check", "dec_attend_noalloc_status", "dec_debug_wait_timeout",
    "dec_build_flags", "dec_debug_poison_table",
)
KERNEL_CLASSES = ("embed", "qkv", "qkv_post", "attn", "attn_merge", "oproj", "gateup", "down", "lmhead", "argmax",
                  "step")


class dec_config(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("vocab", "d_model", "n_layers", "n_heads", "n_kv_heads", "head_dim",
                                         "ff_hidden", "max_positions", "block_tokens", "mode")] + [
        ("rope_base", C.c_double), ("rms_eps", C.c_double)] + [
        (n, C.c_int32) for n in ("qk_norm", "rope_split", "tied", "rope_scaling", "sliding_window", "attention_bias")]


_PP = C.POINTER(C.c_void_p)


class dec_weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("final_norm", C.c_void_p)] + [
        (n, _PP) for n in ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "mlp_norm", "w_gate", "w_up",
                           "w_down")]


_I32P = C.POINTER(C.c_int32)


class dec_batch(C.Structure):
    _fields_ = [("n_seqs", C.c_int32), ("n_tokens", C.c_int32), ("ids", _I32P), ("ids_device", C.c_void_p),
                ("positions", _I32P), ("seq_start", _I32P), ("block_table", _I32P), ("max_blocks", C.c_int32)]


class dec_sampling(C.Structure):
    _fields_ = [("temperature", C.c_double), ("top_k", C.c_int32), ("top_p", C.c_double), ("min_p", C.c_double),
                ("repetition_penalty", C.c_double), ("presence_penalty", C.c_double),
                ("frequency_penalty", C.c_double)]


class dec_rng(C.Structure):
    _fields_ = [("state", C.c_uint64), ("inc", C.c_uint64)]


_lib = None


def lib() -> C.CDLL:
    """The loaded library (raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{os.path.basename(LIB_PATH)} is not built ({LIB_PATH}); run __graft_entry__.build()"
                               " (the DEC_DEBUG build: python -m decoder_qwen3_step_gb300.build --debug)")
        L = C.CDLL(LIB_PATH)
        V, I, SZ, I64 = C.c_void_p, C.c_int, C.c_size_t, C.c_int64
        cfgp = C.POINTER(dec_config)
        sig = {
            "dec_last_error": (C.c_char_p, []),
            "dec_version": (C.c_char_p, []),
            "dec_config_check": (I, [cfgp]),
            "dec_weights_bytes": (I, [cfgp, C.POINTER(SZ)]),
            "dec_workspace_bytes": (I, [cfgp, C.c_int32, C.c_int32, C.POINTER(SZ)]),
            "dec_create": (I, [cfgp, C.POINTER(dec_weights), V, SZ, V, SZ, C.c_int32, C.c_int32, V, C.POINTER(V)]),
            "dec_destroy": (None, [V]),
            "dec_device_status": (I, [V, C.POINTER(C.c_uint32)]),
            "dec_set_dump": (I, [V, V, SZ]),
            "dec_pool_bytes": (I, [cfgp, C.c_int32, C.POINTER(SZ)]),
            "dec_pool_create": (I, [cfgp, C.c_int32, V, SZ, C.POINTER(V)]),
            "dec_pool_destroy": (None, [V]),
            "dec_pool_alloc": (I, [V, C.c_int32, _I32P]),
            "dec_pool_retain": (I, [V, C.c_int32]),
            "dec_pool_release": (I, [V, C.c_int32]),
            "dec_pool_free_blocks": (I, [V, _I32P]),
            "dec_pool_refcount": (I, [V, C.c_int32, _I32P]),
            "dec_pool_set_fill": (I, [V, C.c_int32, C.c_int32]),
            "dec_pool_register": (I, [V, C.c_int32, C.c_uint64, _I32P]),
            "dec_pool_lookup": (I, [V, C.c_uint64, _I32P]),
            "dec_pool_cached_blocks": (I, [V, _I32P]),
            "dec_prefix_key": (C.c_uint64, [C.c_uint64, _I32P, C.c_int32]),
            "dec_kv_offset": (I, [V, _I32P, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.POINTER(I64)]),
            "dec_prefill": (I, [V, V, C.POINTER(dec_batch), C.c_int32, V, V, V]),
            "dec_decode": (I, [V, V, C.POINTER(dec_batch), V, V, V]),
            "dec_f32_to_f16": (I, [V, V, I64, V]),
            "dec_profile_enable": (I, [V, C.c_int32, C.c_int32]),
            "dec_profile_read": (I, [V, C.c_int32, C.POINTER(C.c_double), C.POINTER(I64)]),
            "dec_launch_count": (I, [V, C.POINTER(I64)]),
            "dec_set_graphs": (I, [V, C.c_int32]),
            "dec_set_megakernel": (I, [V, C.c_int32]),
            "dec_set_step_trace": (I, [V, V, C.c_size_t]),
            "dec_megakernel_available": (I, [V, C.POINTER(C.c_int32)]),
            "dec_set_tensor_cores": (I, [V, C.c_int32]),
            "dec_debug_product": (I, [V, C.c_int32, C.c_int32, V, C.c_int32, V, C.c_int32, V]),
            "dec_attend_scratch_bytes": (I, [cfgp, C.c_int32, C.c_int32, C.c_int32, C.POINTER(SZ)]),
            "dec_attend": (I, [V, C.c_int32, C.c_int32, V, _I32P, _I32P, C.c_int32, V, V, SZ, V]),
            "dec_attend_noalloc": (I, [V, C.c_int32, C.c_int32, V, _I32P, _I32P, C.c_int32, V, V]),
            "dec_child_seed": (C.c_uint64, [C.c_uint64, C.c_uint64]),
            "dec_rng_stream": (None, [C.c_uint64, C.c_uint64, C.POINTER(dec_rng)]),
            "dec_rng_next_u32": (C.c_uint32, [C.POINTER(dec_rng)]),
            "dec_rng_uniform": (C.c_double, [C.POINTER(dec_rng)]),
            "dec_sampler_workspace_bytes": (I, [C.c_int32, C.c_int32, C.POINTER(SZ)]),
            "dec_sampler_create": (I, [C.c_int32, C.c_int32, V, SZ, C.POINTER(V)]),
            "dec_sampler_destroy": (None, [V]),
            "dec_sampler_status": (I, [V, C.POINTER(C.c_uint32)]),
            "dec_sample": (I, [V, V, I64, C.c_int32, C.POINTER(dec_sampling), V, _I32P, _I32P, V, V, V, V]),
            "dec_debug_df_exp": (I, [V, V, I64, V]),
            "dec_quantize_int4": (I, [V, C.c_int32, C.c_int32, V, V, V]),
            "dec_batch_check": (I, [V, C.POINTER(dec_batch), C.c_int32]),
            "dec_attend_noalloc_status": (I, [V, C.POINTER(C.c_uint32)]),
            "dec_debug_wait_timeout": (I, [V, C.c_uint32, C.c_uint64]),
            "dec_build_flags": (C.c_uint32, []),
            "dec_debug_poison_table": (I, [V, C.c_int32, C.c_int32, C.c_int32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


class DecError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = lib().dec_last_error().decode(errors="replace")
        super().__init__(f"{where}: {ERROR_NAMES.get(code, code)}: {msg}")


def check(code: int, where: str) -> None:
    if code != DEC_OK:
        raise DecError(code, where)
