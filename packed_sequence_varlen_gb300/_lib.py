"""ctypes declarations for ``libvarlen_attn.so`` (the C ABI in include/varlen_attn.h).

Argument marshalling only.  The library is loaded from this package directory;
a missing library is an error, never a fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int32, c_int64, c_size_t, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libvarlen_attn.so")

VA_OK = 0
STATUS_NAMES = {
    0: "VA_OK", 1: "VA_ERR_INVALID_ARG", 2: "VA_ERR_UNSUPPORTED", 3: "VA_ERR_WORKSPACE",
    4: "VA_ERR_CUDA", 5: "VA_ERR_BAD_SEQLENS", 6: "VA_ERR_TIMEOUT", 7: "VA_ERR_CAPACITY",
    8: "VA_ERR_BAD_TARGETS",
}

# every symbol include/varlen_attn.h declares
EXPORTS = (
    "varlen_shape_contiguous", "varlen_pack_next_fit", "varlen_pack_best_fit_decreasing",
    "varlen_build_metadata", "varlen_validate_cu_seqlens", "varlen_attn_tile_sizes",
    "varlen_attn_workspace_size", "varlen_attn_plan", "varlen_attn_fwd", "varlen_attn_bwd",
    "varlen_read_status", "varlen_clear_status", "varlen_last_error", "varlen_version",
    "varlen_profile_enable", "varlen_profile_read", "varlen_kernel_name", "varlen_launch_count",
    "varlen_attn_fwd_noalloc", "varlen_noalloc_read_status", "varlen_cu_seqlens_from_positions",
    "varlen_loss_targets", "varlen_token_ce_workspace_size", "varlen_token_ce",
    "varlen_unpad_index", "varlen_gather_rows",
    "varlen_attn_plan_window", "varlen_attn_fwd_window", "varlen_attn_bwd_window",
    "varlen_attn_workspace_size_cross", "varlen_attn_plan_cross", "varlen_attn_fwd_cross",
    "varlen_attn_bwd_cross", "varlen_test_stall_next_forward",
)


class VaShape(ctypes.Structure):
    _fields_ = [("T", c_int32), ("B", c_int32), ("Hq", c_int32), ("Hkv", c_int32),
                ("d", c_int32), ("max_seqlen", c_int32),
                ("q_row_stride", c_int64), ("q_head_stride", c_int64),
                ("k_row_stride", c_int64), ("k_head_stride", c_int64),
                ("v_row_stride", c_int64), ("v_head_stride", c_int64),
                ("o_row_stride", c_int64), ("o_head_stride", c_int64)]


class VarlenError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def _declare(lib):
    i32p = POINTER(c_int32)
    sig = {
        "varlen_shape_contiguous": (None, [POINTER(VaShape), c_int32, c_int32, c_int32, c_int32,
                                           c_int32, c_int32]),
        "varlen_pack_next_fit": (c_int32, [i32p, c_int32, c_int32, i32p, i32p, i32p]),
        "varlen_pack_best_fit_decreasing": (c_int32, [i32p, c_int32, c_int32, i32p, i32p, i32p]),
        "varlen_build_metadata": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p,
                                            c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
        "varlen_validate_cu_seqlens": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p,
                                                 c_void_p]),
        "varlen_cu_seqlens_from_positions": (c_int32, [c_void_p, c_int32, c_int32, c_int32, c_void_p,
                                                       c_int32, c_void_p, c_void_p, c_void_p, c_void_p]),
        "varlen_attn_tile_sizes": (c_int32, [c_int32, c_int32, i32p, i32p]),
        "varlen_attn_workspace_size": (c_size_t, [POINTER(VaShape), c_int32]),
        "varlen_attn_plan": (c_int32, [POINTER(VaShape), c_void_p, c_int32, c_int32, c_void_p,
                                       c_int32, c_void_p, c_void_p, c_void_p]),
        "varlen_attn_fwd": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, POINTER(VaShape),
                                      c_float, c_int32, c_void_p, c_void_p, c_void_p, c_size_t,
                                      c_void_p]),
        "varlen_attn_bwd": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_void_p, POINTER(VaShape), c_float, c_int32, c_void_p,
                                      c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
        "varlen_attn_plan_window": (c_int32, [POINTER(VaShape), c_void_p, c_int32, c_int32, c_int32,
                                              c_void_p, c_int32, c_void_p, c_void_p, c_void_p]),
        "varlen_attn_fwd_window": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, POINTER(VaShape),
                                             c_float, c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                             c_size_t, c_void_p]),
        "varlen_attn_bwd_window": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                             c_void_p, POINTER(VaShape), c_float, c_int32, c_int32,
                                             c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
        "varlen_attn_workspace_size_cross": (c_size_t, [POINTER(VaShape), c_int32, c_int32]),
        "varlen_attn_plan_cross": (c_int32, [POINTER(VaShape), c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                             c_void_p, c_int32, c_void_p, c_void_p, c_void_p]),
        "varlen_attn_fwd_cross": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, POINTER(VaShape),
                                            c_int32, c_int32, c_float, c_int32, c_void_p, c_void_p, c_void_p,
                                            c_size_t, c_void_p]),
        "varlen_attn_bwd_cross": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                            c_void_p, c_void_p, POINTER(VaShape), c_int32, c_int32, c_float,
                                            c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                            c_void_p]),
        "varlen_attn_fwd_noalloc": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p,
                                              POINTER(VaShape), c_float, c_int32, c_void_p,
                                              c_void_p, c_void_p]),
        "varlen_noalloc_read_status": (c_int32, [i32p, c_void_p]),
        "varlen_unpad_index": (c_int32, [c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_void_p]),
        "varlen_gather_rows": (c_int32, [c_void_p, c_int64, c_void_p, c_int32, c_int64, c_void_p, c_int64,
                                         c_void_p]),
        "varlen_loss_targets": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p,
                                          c_void_p]),
        "varlen_token_ce_workspace_size": (c_size_t, [c_int32]),
        "varlen_token_ce": (c_int32, [c_void_p, c_int32, c_int64, c_void_p, c_int32, c_int32, c_int32,
                                      c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_size_t,
                                      c_void_p]),
        "varlen_read_status": (c_int32, [c_void_p, i32p, c_void_p]),
        "varlen_clear_status": (c_int32, [c_void_p, c_void_p]),
        "varlen_profile_enable": (c_int32, [c_int32]),
        "varlen_profile_read": (c_int32, [i32p, POINTER(c_float), c_int32, i32p]),
        "varlen_kernel_name": (c_char_p, [c_int32]),
        "varlen_launch_count": (c_int64, []),
        "varlen_test_stall_next_forward": (c_int32, [c_int64]),
        "varlen_last_error": (c_char_p, []),
        "varlen_version": (c_char_p, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args


def load():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        _declare(lib)
        _lib = lib
    return _lib


def check(status: int):
    if status != VA_OK:
        msg = load().varlen_last_error().decode(errors="replace")
        raise VarlenError(status, msg)
