"""ctypes declarations of the C ABI in include/dflash.h.

Argument marshalling only: every step of the draft cycle runs in the CUDA
library.  Loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

LIB_NAME = "libdflash_gb300.so"
_LIB = None

c_i32 = ctypes.c_int32
c_size = ctypes.c_size_t
c_ptr = ctypes.c_void_p
c_i32p = ctypes.POINTER(ctypes.c_int32)

DFLASH_OK = 0
ERRORS = {
    -1: "DFLASH_ERR_INVALID_ARG", -2: "DFLASH_ERR_SHAPE", -3: "DFLASH_ERR_CAPACITY", -4: "DFLASH_ERR_CUDA",
    -5: "DFLASH_ERR_TIMEOUT", -6: "DFLASH_ERR_UNSUPPORTED", -7: "DFLASH_ERR_WORKSPACE",
}
DTYPE_F32 = 0
DTYPE_BF16 = 1


class Config(ctypes.Structure):
    _fields_ = [("hidden", c_i32), ("layers", c_i32), ("n_q_heads", c_i32), ("n_kv_heads", c_i32),
                ("head_dim", c_i32), ("ffn", c_i32), ("vocab", c_i32), ("n_target_feats", c_i32),
                ("max_block", c_i32), ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("mask_token_id", c_i32), ("dtype", c_i32), ("qk_norm", c_i32), ("input_fusion", c_i32),
                ("kv_bf16", c_i32), ("head_bf16", c_i32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, c_ptr) for n in ("g_in", "w_q", "w_k", "w_v", "w_o", "g_post", "w_g", "w_u", "w_d", "g_q", "g_k")]


class Weights(ctypes.Structure):
    _fields_ = [("embed", c_ptr), ("lm_head", c_ptr), ("w_c", c_ptr), ("g_c", c_ptr), ("g_final", c_ptr),
                ("layers", ctypes.POINTER(LayerWeights))]


POLICY_MAX_CANDIDATES = 16


class PolicyConfig(ctypes.Structure):
    _fields_ = [("n_candidates", c_i32), ("candidates", c_i32 * POLICY_MAX_CANDIDATES),
                ("cost_fixed_ms", ctypes.c_float), ("cost_per_row_ms", ctypes.c_float),
                ("cost_per_request_ms", ctypes.c_float), ("decay", ctypes.c_float),
                ("prior_accept", ctypes.c_float), ("prior_weight", ctypes.c_float)]


# name -> (restype, argtypes)
SIGNATURES = {
    "dflash_version": (c_i32, []),
    "dflash_last_error": (ctypes.c_char_p, []),
    "dflash_model_create": (c_i32, [ctypes.POINTER(Config), ctypes.POINTER(Weights), ctypes.POINTER(c_ptr)]),
    "dflash_model_destroy": (c_i32, [c_ptr]),
    "dflash_get_status": (c_i32, [c_ptr, c_ptr, c_i32p]),
    "dflash_clear_status": (c_i32, [c_ptr, c_ptr]),
    "dflash_selftest_wait_timeout": (c_i32, [c_ptr, ctypes.c_int64, c_ptr]),
    "dflash_cache_bytes": (c_size, [ctypes.POINTER(Config), c_i32, c_i32]),
    "dflash_cache_init": (c_i32, [c_ptr, c_ptr, c_size, c_i32, c_i32, c_ptr, ctypes.POINTER(c_ptr)]),
    "dflash_cache_destroy": (c_i32, [c_ptr]),
    "dflash_cache_layout": (c_i32, [c_ptr, ctypes.POINTER(c_size), ctypes.POINTER(c_size), ctypes.POINTER(c_size)]),
    "dflash_cache_set_lengths": (c_i32, [c_ptr, c_i32p, c_ptr]),
    "dflash_workspace_bytes": (c_size, [c_ptr, c_i32, c_i32, c_i32, c_i32]),
    "dflash_inject_context": (c_i32, [c_ptr, c_ptr, c_ptr, c_ptr, c_i32p, c_i32, c_ptr, c_size, c_ptr]),
    "dflash_draft_block": (c_i32, [c_ptr, c_ptr, c_ptr, c_i32, c_ptr, c_ptr, c_ptr, c_size, c_ptr]),
    "dflash_draft_cycle": (c_i32, [c_ptr, c_ptr, c_ptr, c_ptr, c_i32p, c_i32, c_ptr, c_i32, c_ptr, c_ptr, c_ptr, c_size,
                                   c_ptr]),
    "dflash_noalloc_scratch_bytes": (c_size, []),
    "dflash_inject_context_noalloc": (c_i32, [c_ptr, c_ptr, c_ptr, c_ptr, c_i32p, c_i32, c_ptr]),
    "dflash_verify_greedy": (c_i32, [c_ptr, c_ptr, c_i32, c_i32, c_ptr, c_ptr, c_ptr, c_ptr]),
    "dflash_sampling_workspace_bytes": (c_size, [c_i32, c_i32, c_i32]),
    "dflash_verify_sampled": (c_i32, [c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_i32, c_i32, c_i32, ctypes.c_float, c_ptr,
                                      c_ptr, c_ptr, c_ptr, c_size, c_ptr]),
    "dflash_sample_tokens": (c_i32, [c_ptr, c_i32, c_i32, ctypes.c_float, c_ptr, c_ptr, c_ptr, c_size, c_ptr]),
    "dflash_block_policy_create": (c_i32, [ctypes.POINTER(PolicyConfig), ctypes.POINTER(c_ptr)]),
    "dflash_block_policy_destroy": (c_i32, [c_ptr]),
    "dflash_block_policy_observe": (c_i32, [c_ptr, c_i32, c_i32p, c_i32]),
    "dflash_block_policy_choose": (c_i32, [c_ptr, c_i32, c_i32p, ctypes.POINTER(ctypes.c_double)]),
    "dflash_block_policy_acceptance": (c_i32, [c_ptr, ctypes.POINTER(ctypes.c_double), c_i32]),
    "dflash_packed_attention_workspace_bytes": (c_size, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32]),
    "dflash_packed_block_attention": (c_i32, [c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_i32p, c_i32, c_i32, c_i32,
                                              c_i32, c_i32, c_i32, c_i32, c_ptr, c_ptr, c_size, c_ptr]),
    "dflash_packed_attention_status": (c_i32, [c_ptr, c_ptr, c_i32p]),
    "dflash_launch_count": (ctypes.c_uint64, []),
    "dflash_synthetic_target": (c_i32, [c_ptr, c_ptr, c_ptr, c_ptr, c_i32, c_ptr, c_ptr, c_ptr, c_i32, c_i32, c_i32,
                                        c_ptr, c_ptr]),
    "dflash_trace_read": (c_i32, [c_ptr, ctypes.POINTER(ctypes.c_uint64), c_size]),
    "dflash_profile_start": (c_i32, [c_ptr, c_i32]),
    "dflash_profile_stop": (c_i32, [c_ptr, c_ptr, ctypes.POINTER(ctypes.c_float), c_i32p, c_i32]),
}

STAGES = ["fuse", "inject", "qkv", "attn", "o", "gateup", "down", "lmhead", "other", "inject_persist",
          "draft_persist", "cycle_persist"]


def lib_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), LIB_NAME)


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"DFlash CUDA library {path} is not built; run __graft_entry__.build() "
                               "(there is no CPU fallback)")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


class DFlashError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = lib().dflash_last_error().decode(errors="replace")
        super().__init__(f"{where}: {ERRORS.get(code, code)}: {msg}")
        self.code = code


def check(code: int, where: str) -> None:
    if code != DFLASH_OK:
        raise DFlashError(code, where)
