"""ctypes declarations of the libtq C ABI (``include/tq.h``).

Argument marshalling only: every computation runs inside libtq. Loading fails
loudly when the library has not been built; there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libtq.so")

TQ_OK = 0
TQ_ERR_INVALID_ARG = -1
TQ_ERR_UNSUPPORTED = -2
TQ_ERR_MISALIGNED = -3
TQ_ERR_WORKSPACE_TOO_SMALL = -4
TQ_ERR_CUDA = -5

TQ_PRESET_K8V4 = 0
TQ_PRESET_4BIT_NC = 1
TQ_PRESET_K3V4_NC = 2
TQ_PRESET_3BIT_NC = 3
TQ_PRESET_PROD3 = 4
PRESET_IDS = {"k8v4": TQ_PRESET_K8V4, "4bit_nc": TQ_PRESET_4BIT_NC,
              "k3v4_nc": TQ_PRESET_K3V4_NC, "3bit_nc": TQ_PRESET_3BIT_NC, "prod3": TQ_PRESET_PROD3}

TQ_DTYPE_F16 = 0
TQ_DTYPE_BF16 = 1
TQ_DTYPE_F32 = 2

TQ_DEV_SLOT_OUT_OF_RANGE = 1
TQ_DEV_BLOCK_OUT_OF_RANGE = 2
TQ_DEV_SEQ_TOO_LONG = 4
TQ_DEV_TIMEOUT = 8

# every function tq.h declares (checked by the ABI tests)
EXPORTED = ("tq_build_codebook", "tq_layout_for", "tq_store", "tq_decode_workspace_size",
            "tq_decode", "tq_decode_append", "tq_decode_partials", "tq_decode_reduce", "tq_decode_noalloc",
            "tq_dequant", "tq_prod_layout_for", "tq_prod_store", "tq_prod_scores_workspace_size",
            "tq_prod_scores", "tq_continue_workspace_size", "tq_continue", "tq_status_string", "tq_version")

TQ_DECODE_NOALLOC_SCRATCH_BYTES = 32 << 20


class tq_config(ctypes.Structure):
    _fields_ = [("preset", ctypes.c_int), ("head_dim", ctypes.c_int), ("block_size", ctypes.c_int),
                ("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("partition_tokens", ctypes.c_int), ("flags", ctypes.c_int)]


class tq_layout(ctypes.Structure):
    _fields_ = [("key_bits", ctypes.c_int), ("value_bits", ctypes.c_int), ("key_fp8", ctypes.c_int),
                ("norm_correction", ctypes.c_int), ("key_packed_bytes", ctypes.c_int),
                ("value_packed_bytes", ctypes.c_int), ("slot_bytes", ctypes.c_int),
                ("tile_tokens", ctypes.c_int), ("tile_bytes", ctypes.c_int),
                ("k_off", ctypes.c_int), ("k_row_bytes", ctypes.c_int),
                ("v_off", ctypes.c_int), ("v_row_bytes", ctypes.c_int),
                ("knorm_off", ctypes.c_int), ("vscale_off", ctypes.c_int), ("vzero_off", ctypes.c_int),
                ("block_bytes", ctypes.c_longlong)]


class tq_prod_layout(ctypes.Structure):
    _fields_ = [("mse_bits", ctypes.c_int), ("slot_bytes", ctypes.c_int), ("tile_bytes", ctypes.c_int),
                ("k_off", ctypes.c_int), ("k_row_bytes", ctypes.c_int),
                ("sign_off", ctypes.c_int), ("sign_row_bytes", ctypes.c_int),
                ("norm_off", ctypes.c_int), ("rnorm_off", ctypes.c_int), ("block_bytes", ctypes.c_longlong)]


class tq_codebook(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int), ("bits", ctypes.c_int), ("num_levels", ctypes.c_int),
                ("centroids", ctypes.c_float * 16), ("midpoints", ctypes.c_float * 15)]


_vp = ctypes.c_void_p
_i = ctypes.c_int
_ll = ctypes.c_longlong
_sz = ctypes.c_size_t
_f = ctypes.c_float

_SIGS = {
    "tq_build_codebook": (_i, [_i, _i, ctypes.POINTER(tq_codebook)]),
    "tq_layout_for": (_i, [ctypes.POINTER(tq_config), ctypes.POINTER(tq_layout)]),
    "tq_store": (_i, [ctypes.POINTER(tq_config), ctypes.POINTER(tq_codebook), _vp, _vp, _i, _ll, _vp,
                      _vp, _ll, _vp, _vp]),
    "tq_decode_workspace_size": (_sz, [ctypes.POINTER(tq_config), _i, _i]),
    "tq_decode": (_i, [ctypes.POINTER(tq_config), ctypes.POINTER(tq_codebook), _vp, _i, _vp, _ll, _vp, _i,
                       _vp, _i, _i, _f, _vp, _i, _vp, _sz, _vp, _vp]),
    "tq_decode_append": (_i, [ctypes.POINTER(tq_config), ctypes.POINTER(tq_codebook), _vp, _i, _vp, _vp, _vp,
                              _ll, _vp, _i, _vp, _i, _i, _f, _vp, _i, _vp, _sz, _vp, _vp]),
    "tq_decode_partials": (_i, [ctypes.POINTER(tq_config), ctypes.POINTER(tq_codebook), _vp, _i, _vp, _ll,
                                _vp, _i, _vp, _i, _i, _f, _vp, _sz, _vp, _vp]),
    "tq_decode_reduce": (_i, [ctypes.POINTER(tq_config), _vp, _i, _i, _i, _vp, _i, _vp, _sz, _vp]),
    "tq_decode_noalloc": (_i, [ctypes.POINTER(tq_config), ctypes.POINTER(tq_codebook), _vp, _i, _vp, _ll,
                               _vp, _i, _vp, _i, _i, _f, _vp, _i, _vp, _vp]),
    "tq_dequant": (_i, [ctypes.POINTER(tq_config), ctypes.POINTER(tq_codebook), _vp, _ll, _vp, _i, _vp, _i,
                        _i, _vp, _vp, _i, _vp, _vp]),
    "tq_prod_layout_for": (_i, [ctypes.POINTER(tq_config), ctypes.POINTER(tq_prod_layout)]),
    "tq_prod_store": (_i, [ctypes.POINTER(tq_config), ctypes.POINTER(tq_codebook), _vp, _vp, _i, _ll, _vp, _vp, _ll,
                           _vp, _vp]),
    "tq_prod_scores_workspace_size": (_sz, [ctypes.POINTER(tq_config), _i]),
    "tq_prod_scores": (_i, [ctypes.POINTER(tq_config), ctypes.POINTER(tq_codebook), _vp, _vp, _i, _vp, _ll, _vp, _i,
                            _vp, _i, _i, _f, _vp, _vp, _sz, _vp, _vp]),
    "tq_continue_workspace_size": (_sz, [ctypes.POINTER(tq_config), _i, _i]),
    "tq_continue": (_i, [ctypes.POINTER(tq_config), ctypes.POINTER(tq_codebook), _vp, _i, _vp, _i, _i, _i, _vp, _ll,
                         _vp, _i, _vp, _i, _f, _vp, _i, _vp, _sz, _vp, _vp]),
    "tq_status_string": (ctypes.c_char_p, [_i]),
    "tq_version": (_i, []),
}

_lib = None


def lib_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load libtq.so (built by ``turboquant_paged_kv_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"libtq.so is not built ({_LIB_PATH}); run "
                              "`python -m turboquant_paged_kv_gb300.build` first")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class TQError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = load().tq_status_string(status).decode()
        super().__init__(f"{fn} failed: {msg} ({status})")
        self.status = status


def check(fn: str, status: int) -> None:
    if status != TQ_OK:
        raise TQError(fn, status)
