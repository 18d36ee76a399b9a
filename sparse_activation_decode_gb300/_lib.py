"""ctypes view of the C ABI declared in include/np.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnp.so")

NP_OK, NP_ERR_ARG, NP_ERR_OOM, NP_ERR_CUDA, NP_ERR_IO, NP_ERR_TIMEOUT, NP_ERR_STATE = 0, -1, -2, -3, -4, -5, -6
NP_F32, NP_F16, NP_BF16 = 0, 1, 2
NP_COMBINE_INTERSECT, NP_COMBINE_UNION = 0, 1
NP_RES_SLOTMAP, NP_RES_WINDOW, NP_RES_FREQUENCY = 0, 1, 2
NP_PRED_SHARED_ARGMAX, NP_PRED_PERLAYER_SIGMOID = 0, 1
NP_H2D_STAGED, NP_H2D_FUSED = 0, 1
NP_SLOTS_REUSE, NP_SLOTS_COMPACT = 0, 1
KIND_NAMES = ["dense", "predictor", "set", "gather", "scatter", "ffn", "finish"]
NP_N_KINDS = len(KIND_NAMES)

READ_HOOK = ctypes.CFUNCTYPE(ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32)


class ModelDesc(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("n_dense", ctypes.c_int32), ("d_model", ctypes.c_int32),
        ("d_ff", ctypes.c_int32), ("k_max", ctypes.c_int32), ("n_centroids", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("has_gate", ctypes.c_int32), ("combine", ctypes.c_int32),
        ("residency", ctypes.c_int32), ("window", ctypes.c_int32), ("batch", ctypes.c_int32),
        ("staging_rows", ctypes.c_int32), ("pred_hidden", ctypes.c_int32), ("pred_kind", ctypes.c_int32),
        ("h2d_mode", ctypes.c_int32), ("activation", ctypes.c_int32), ("slots", ctypes.c_int32), ("lookahead", ctypes.c_int32),
        ("host_store", ctypes.c_void_p), ("dense_w", ctypes.c_void_p), ("pred_w1", ctypes.c_void_p),
        ("pred_w2", ctypes.c_void_p), ("pred_b2", ctypes.c_void_p), ("centroids", ctypes.c_void_p),
        ("main_stream", ctypes.c_void_p), ("side_stream", ctypes.c_void_p),
        ("read_hook", READ_HOOK), ("read_ctx", ctypes.c_void_p),
    ]


class DeltaView(ctypes.Structure):
    _fields_ = [
        ("n_sparse", ctypes.c_int32), ("k_max", ctypes.c_int32),
        ("counts", ctypes.c_void_p), ("active", ctypes.c_void_p), ("active_slot", ctypes.c_void_p),
        ("din_neuron", ctypes.c_void_p), ("din_slot", ctypes.c_void_p), ("dout_neuron", ctypes.c_void_p),
        ("ids", ctypes.c_void_p),
        ("move_count", ctypes.c_void_p), ("move_src", ctypes.c_void_p), ("move_dst", ctypes.c_void_p),
    ]


class Stats(ctypes.Structure):
    _fields_ = [("token", ctypes.c_int64), ("active_rows", ctypes.c_int64), ("din_rows", ctypes.c_int64),
                ("dout_rows", ctypes.c_int64), ("dropped_rows", ctypes.c_int64), ("h2d_bytes", ctypes.c_int64),
                ("moved_rows", ctypes.c_int64)]


# symbol -> (restype, argtypes)
_P, _I32, _I64, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = {
    "np_init_model": (_I32, [ctypes.POINTER(ModelDesc), ctypes.POINTER(_P)]),
    "np_free_model": (_I32, [_P]),
    "np_reset_sequence": (_I32, [_P]),
    "np_predict": (_I32, [_P, _I32, _P, _P]),
    "np_delta": (_I32, [_P, _I32, _P, ctypes.POINTER(DeltaView)]),
    "np_last_delta": (_I32, [_P, ctypes.POINTER(DeltaView)]),
    "np_scatter": (_I32, [_P, _I32]),
    "np_sparse_mlp": (_I32, [_P, _I32, _P, _P]),
    "np_dense_mlp": (_I32, [_P, _I32, _P, _P]),
    "np_ffn_layers": (_I32, [_P, _I32, _I32, _P]),
    "np_decode_token": (_I32, [_P, _P, ctypes.POINTER(Stats)]),
    "np_get_state": (_I32, [_P, _I32, _P, _P]),
    "np_resident_rows": (_I32, [_P, _I32, _I32, ctypes.POINTER(_P)]),
    "np_get_counts": (_I32, [_P, _P]),
    "np_check_error": (_I32, [_P]),
    "np_set_profiling": (_I32, [_P, _I32]),
    "np_get_profile": (_I32, [_P, _P, _P, _P]),
    "np_get_timeline": (_I32, [_P, _P, _P, _P, _I32, _P]),
    "np_host_register": (_I32, [_P, _SZ]),
    "np_host_unregister": (_I32, [_P]),
    "np_ffn_rows_noalloc": (_I32, [_P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P]),
    "np_ffn_rows_noalloc_check": (_I32, [_P]),
    "np_launch_count": (_I64, [_P]),
    "np_status_str": (ctypes.c_char_p, [_I32]),
    "np_last_error": (ctypes.c_char_p, []),
}

_lib = None


class NpError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: status {status} ({detail})")
        self.status = status


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libnp.so (built by sparse_activation_decode_gb300.build).  Raises
    ImportError when the library has not been built: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    import torch  # noqa: F401  (loads the CUDA runtime the library links against)
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"CUDA library not built: {p} is missing "
                          "(run `python -m sparse_activation_decode_gb300.build`)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(status: int, where: str) -> None:
    if status != NP_OK:
        lib = load()
        detail = f"{lib.np_status_str(status).decode()}: {lib.np_last_error().decode()}"
        raise NpError(status, where, detail)
