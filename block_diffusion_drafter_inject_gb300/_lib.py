"""ctypes declarations of the C ABI in include/dflash.h.

Loading fails loudly (RuntimeError) when libdflash.so has not been built:
there is no other implementation to fall back to."""

import ctypes
import os

from .build import LIB

MAX_LAYERS = 16
MAX_BLOCK = 32
MAX_TOPK = 32

F32 = 0
BF16 = 1

OK = 0
ERR_NULL, ERR_DIMS, ERR_BLOCK, ERR_WORKSPACE, ERR_DTYPE, ERR_CUDA, ERR_ALIGN, ERR_DEVICE = \
    -1, -2, -3, -4, -5, -6, -7, -8
DEV_TOKEN_RANGE, DEV_PAGE_RANGE, DEV_POS_RANGE, DEV_TIMEOUT, DEV_REQ_RANGE = 1, 2, 4, 8, 16

vp = ctypes.c_void_p
i32 = ctypes.c_int32
ip = ctypes.POINTER(ctypes.c_int32)


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "d_model", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "d_ff", "vocab",
        "n_taps", "d_target", "window", "page_size", "top_k", "sel_rank", "conv_group",
        "mask_token_id", "dtype")] + [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                                      ("weight_bits", ctypes.c_int32)]


class Q4(ctypes.Structure):
    _fields_ = [("data", vp)]


# the matrices a 4-bit drafter keeps in 4 bits
Q4_LAYER = ("wqkv", "wo", "w_gate_up", "w_down")
Q4_TOP = ("fc", "lm_head")


class LayerWeights(ctypes.Structure):
    _fields_ = [("attn_norm", vp), ("mlp_norm", vp), ("wqkv", vp), ("wo", vp), ("q_norm", vp),
                ("k_norm", vp), ("w_gate_up", vp), ("w_down", vp), ("conv_w", vp * 4),
                ("conv_base", vp * 4)] + [(n + "_q4", Q4) for n in Q4_LAYER]


class Weights(ctypes.Structure):
    _fields_ = [("fc_norm", vp), ("fc", vp), ("embed", vp), ("lm_head", vp), ("final_norm", vp),
                ("sel_pu", vp), ("sel_pv", vp), ("layer", LayerWeights * MAX_LAYERS),
                ("sel_table", vp), ("sel_gate", vp)] + [(n + "_q4", Q4) for n in Q4_TOP]


class KV(ctypes.Structure):
    _fields_ = [("k", vp), ("v", vp), ("page_table", vp), ("num_pages", ctypes.c_int32),
                ("max_pages_per_req", ctypes.c_int32), ("num_rows", ctypes.c_int32)]


EXPORTS = {
    "dflash_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Config), i32, i32, i32]),
    "dflash_inject_context": (ctypes.c_int, [ctypes.POINTER(Config), ctypes.POINTER(Weights),
                                             ctypes.POINTER(KV), vp, vp, vp, i32, vp,
                                             ctypes.c_size_t, vp]),
    "dflash_draft_block": (ctypes.c_int, [ctypes.POINTER(Config), ctypes.POINTER(Weights),
                                          ctypes.POINTER(KV), vp, vp, i32, i32, vp, vp, vp, vp,
                                          ctypes.c_size_t, vp]),
    "dflash_draft_block_inject": (ctypes.c_int, [ctypes.POINTER(Config), ctypes.POINTER(Weights),
                                                 ctypes.POINTER(KV), vp, vp, vp, i32, vp, vp, i32,
                                                 i32, vp, vp, vp, vp, ctypes.c_size_t, vp]),
    "dflash_select_path": (ctypes.c_int, [ctypes.POINTER(Config), ctypes.POINTER(Weights), vp, vp,
                                          vp, i32, i32, vp, vp, vp, ctypes.c_size_t, vp]),
    "dflash_prepare_selector": (ctypes.c_int, [ctypes.POINTER(Config), ctypes.POINTER(Weights),
                                               vp, vp, ctypes.c_size_t, vp]),
    "dflash_accept_greedy": (ctypes.c_int, [vp, vp, i32, i32, i32, i32, vp, vp, vp,
                                            ctypes.c_size_t, vp]),
    "dflash_accept_greedy_noalloc": (ctypes.c_int, [vp, vp, i32, i32, i32, i32, vp, vp, vp]),
    "dflash_sample_path": (ctypes.c_int, [ctypes.POINTER(Config), ctypes.POINTER(Weights), vp,
                                          vp, vp, i32, i32, vp, vp, vp, vp, ctypes.c_size_t,
                                          vp]),
    "dflash_select_greedy": (ctypes.c_int, [ctypes.POINTER(Config), ctypes.POINTER(Weights), vp,
                                            vp, vp, vp, i32, i32, vp, vp, vp, ctypes.c_size_t,
                                            vp]),
    "dflash_draft_hidden": (ctypes.c_void_p, [ctypes.POINTER(Config), i32, i32, vp,
                                              ctypes.c_size_t]),
    "dflash_accept_sample": (ctypes.c_int, [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp,
                                            vp, ctypes.c_size_t, vp]),
    "dflash_linear": (ctypes.c_int, [i32, vp, i32, i32, vp, i32, i32, vp, vp]),
    "dflash_linear_splits": (ctypes.c_int32, [i32, i32, i32]),
    "dflash_linear_q4": (ctypes.c_int, [Q4, i32, i32, vp, i32, i32, vp, vp]),
    "dflash_test_linear_wait": (ctypes.c_int, [vp, i32, i32, vp, i32, vp, vp, ctypes.c_size_t,
                                               ctypes.c_uint32, vp]),
    "dflash_read_device_status": (ctypes.c_int, [vp, vp]),
    "dflash_clear_device_status": (ctypes.c_int, [vp, vp]),
    "dflash_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "dflash_launch_count": (ctypes.c_int64, [ctypes.c_int]),
}

_lib = None


def lib():
    """The loaded C-ABI library (built by __graft_entry__.build() / build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(
                f"libdflash.so is missing ({LIB}); build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` - there is no fallback")
        L = ctypes.CDLL(LIB)
        for name, (res, args) in EXPORTS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class DFlashError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = code
        msg = lib().dflash_status_string(code).decode()
        super().__init__(f"{what}: {msg} ({code})" if what else f"{msg} ({code})")


def check(code, what=""):
    if code != OK:
        raise DFlashError(code, what)
    return code
