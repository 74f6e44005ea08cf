"""ctypes view of libcsa.so (the C ABI declared in include/csa.h).

Loading fails loudly if the library has not been built: there is no fallback
implementation of any step.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcsa.so")

c_int, c_float, c_ll, c_size, c_vp = ctypes.c_int, ctypes.c_float, ctypes.c_longlong, ctypes.c_size_t, ctypes.c_void_p
c_u32p = ctypes.POINTER(ctypes.c_uint32)
c_sizep = ctypes.POINTER(ctypes.c_size_t)

CSA_OK, CSA_ERR_INVALID, CSA_ERR_UNSUPPORTED, CSA_ERR_WORKSPACE, CSA_ERR_CUDA, CSA_ERR_TIMEOUT, \
    CSA_ERR_DEVICE_INDEX = range(7)
CSA_BF16, CSA_F32 = 0, 1
CSA_WS_HEADER_BYTES = 256
CSA_FLAG_TIMEOUT, CSA_FLAG_INDEX = 1, 2


class csa_layer_args(ctypes.Structure):
    _fields_ = [(n, c_int) for n in ("B", "Tq", "N", "m", "H", "d", "H_I", "d_I", "k", "W", "T", "T_raw")] + [
        ("scale", c_float),
        ("x_k", c_vp), ("x_v", c_vp), ("x_i", c_vp),
        ("g_k", c_vp), ("g_v", c_vp), ("g_i", c_vp),
        ("k_cmp", c_vp), ("v_cmp", c_vp), ("i_cmp", c_vp),
        ("k_win", c_vp), ("v_win", c_vp),
        ("raw_base", c_vp), ("q", c_vp), ("q_idx", c_vp), ("w", c_vp), ("q_pos", c_vp),
        ("idx_out", c_vp), ("out", c_vp), ("out_dtype", c_int), ("lse", c_vp),
        ("i_win", c_vp), ("gk_win", c_vp), ("gv_win", c_vp), ("gi_win", c_vp),
        ("w_stride", ctypes.c_longlong), ("i_scale", c_vp),
    ]


CSA_STACK_SWA, CSA_STACK_CSA, CSA_STACK_HCA = 0, 1, 2


class csa_stack_layer(ctypes.Structure):
    _fields_ = [("kind", c_int), ("a", csa_layer_args)]


# name -> (restype, argtypes)
SIGNATURES = {
    "csa_status_string": (ctypes.c_char_p, [c_int]),
    "csa_version": (c_int, []),
    "csa_workspace_init": (c_int, [c_vp, c_size, c_vp]),
    "csa_check_error": (c_int, [c_vp, c_u32p, c_int, c_vp]),
    "csa_compress": (c_int, [c_int, ctypes.POINTER(c_vp), ctypes.POINTER(c_vp), ctypes.POINTER(c_vp),
                             ctypes.POINTER(c_int), c_int, c_int, c_int, c_int, c_vp]),
    "csa_append": (c_int, [c_int, ctypes.POINTER(c_vp), ctypes.POINTER(c_vp), ctypes.POINTER(c_vp),
                           ctypes.POINTER(c_int), c_vp, c_vp, c_int, c_int, c_int, c_int, c_int, c_vp, c_size,
                           c_vp]),
    "csa_index_scores": (c_int, [c_vp, c_vp, c_vp, ctypes.c_int64, c_vp, c_int, c_int, c_int, c_int, c_int,
                                 c_int, c_vp, ctypes.c_int64, c_vp, c_size, c_vp]),
    "csa_quantize_fp8": (c_int, [c_vp, ctypes.c_int64, c_int, c_vp, c_vp, c_vp]),
    "csa_index_scores_fp8": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, ctypes.c_int64, c_vp, c_int, c_int, c_int, c_int,
                                     c_int, c_int, c_vp, ctypes.c_int64, c_vp, c_size, c_vp]),
    "csa_topk": (c_int, [c_vp, ctypes.c_int64, c_vp, c_int, c_int, c_int, c_int, c_int, c_vp, c_vp,
                         c_vp, c_size, c_vp]),
    "csa_topk_workspace": (c_int, [c_int, c_int, c_int, c_int, c_sizep]),
    "csa_index_topk_workspace": (c_int, [c_int, c_int, c_int, c_int, c_int, c_int, c_sizep]),
    "csa_index_topk": (c_int, [c_vp, c_vp, c_vp, ctypes.c_int64, c_vp, c_int, c_int, c_int, c_int, c_int, c_int,
                               c_int, c_vp, c_vp, c_vp, c_size, c_vp]),
    "csa_attend_workspace": (c_int, [c_int, c_int, c_int, c_int, c_int, c_int, c_sizep]),
    "csa_attend": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_int, c_int,
                           c_int, c_int, c_int, c_int, c_float, c_vp, c_int, c_vp, c_vp, c_size, c_vp]),
    "csa_attend_noalloc": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_int, c_int,
                                   c_int, c_int, c_int, c_int, c_float, c_vp, c_int, c_vp, c_vp]),
    "hca_attend_workspace": (c_int, [c_int, c_int, c_int, c_int, c_int, c_int, c_sizep]),
    "hca_attend": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_int, c_int, c_int,
                           c_int, c_int, c_int, c_float, c_vp, c_int, c_vp, c_vp, c_size, c_vp]),
    "csa_layer_workspace": (c_int, [ctypes.POINTER(csa_layer_args), c_sizep]),
    "csa_layer": (c_int, [ctypes.POINTER(csa_layer_args), c_vp, c_size, c_vp]),
    "csa_layer_host": (c_int, [ctypes.POINTER(csa_layer_args), c_vp, c_vp, c_vp, c_vp, c_size, c_vp]),
    "csa_stack_workspace": (c_int, [ctypes.POINTER(csa_stack_layer), c_int, c_sizep]),
    "csa_stack_decode": (c_int, [ctypes.POINTER(csa_stack_layer), c_int, c_vp, c_vp, c_int, c_vp, c_size, c_vp]),
    "csa_set_wait_budget": (None, [c_ll]),
    "csa_set_indexer_events": (None, [c_vp, c_vp]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m long_context_sparse_23_b300.build` (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


class CsaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {lib().csa_status_string(status).decode()}")


def check(fn: str, status: int) -> None:
    if status != CSA_OK:
        raise CsaError(fn, status)
