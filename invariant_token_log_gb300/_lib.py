"""ctypes declarations of the C ABI in include/bil.h.

Loading fails loudly: there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

# status codes and element types, as include/bil.h defines them
OK, E_INVALID_ARG, E_DTYPE, E_ALIGN, E_TARGET_RANGE, E_CUDA, E_UNSUPPORTED = range(7)
F32, BF16, F16 = 0, 1, 2
MAX_TILE_BYTES = 64 * 1024
MAX_FUSED_TILES = 2048
MAX_EXTENT_BYTES = 1 << 48
LINEAR_TILE_V = 256
LINEAR_STATIC_SCRATCH_BYTES = 8 * 1024 * 1024
LAYOUT_K_MAJOR, LAYOUT_MN_MAJOR = 0, 1

# every entry point the header declares: name -> (restype, argtypes)
_i32, _i64, _p, _u = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint
_f = ctypes.c_float
SIGNATURES = {
    "bil_contract_id": (ctypes.c_char_p, []),
    "bil_status_string": (ctypes.c_char_p, [_i32]),
    "bil_logp_fwd": (_i32, [_p, _i32, _i64, _i64, _i64, _p, _i64, ctypes.c_int32, _f, _p, _p, _p, _i32, _p]),
    "bil_logp_tile_partials": (_i32, [_p, _i32, _i64, _i64, _i64, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, _f, _p, _i64, _p, _p, _p, _i64, _p, _p]),
    "bil_logp_merge": (_i32, [_p, _p, _p, _i64, ctypes.c_int32, _i64, _p, _p, _i64, _i64, _p, _p, _p, _i32, _p]),
    "bil_logp_bwd": (_i32, [_p, _i32, _i64, _i64, _i64, _p, _i64, _f, _p, _p, _p, _p, _p, _i32, _i64, _i64,
                            _p]),
    "bil_stream_shape": (_i32, [_i32, ctypes.c_int32, _i64, _i32, _i32, ctypes.POINTER(_i32),
                                ctypes.POINTER(_i32), ctypes.POINTER(_i64)]),
    "bil_watchdog_status": (_i32, [ctypes.POINTER(_u), _i32]),
    "bil_watchdog_selftest": (_i32, [_p]),
    "bil_linear_logp_partials": (_i32, [_p, _p, _i32, _i64, _i64, _i64, _i64, _i64, ctypes.c_int32, ctypes.c_int32,
                                        _f, _p, _i64, _p, _p, _p, _i64, _p, _p, _i32, _i64, _p]),
    "bil_linear_logp_workspace_bytes": (_i32, [_i64, _i64, _i32, ctypes.POINTER(_i64)]),
    "bil_linear_logp_fwd": (_i32, [_p, _p, _i32, _i64, _i64, _i64, _i64, _i64, _f, _p, _i64, _p, _p, _p, _p, _i32,
                                   _i64, _p, _i64, _i32, _p]),
    "bil_linear_logp_bwd": (_i32, [_p, _p, _i32, _i64, _i64, _i64, _i64, _i64, ctypes.c_int32, ctypes.c_int32,
                                   _f, _p, _i64, _p, _p, _p, _p, _p, _i64, _p, _i32, _i64, _p, _i32, _i64, _p]),
    "bil_linear_logp_grad": (_i32, [_p, _p, _i32, _i64, _i64, _i64, _i64, _i64, ctypes.c_int32, ctypes.c_int32,
                                    _f, _p, _i64, _p, _p, _p, _p, _p, _i64, _p]),
    "bil_linear_gemm": (_i32, [_p, _i32, _p, _i32, _i32, _i64, _i64, _i64, _i64, _i64, _p, _i32, _i64, _p]),
    "bil_sum_f32": (_i32, [ctypes.POINTER(ctypes.c_void_p), _i32, _i64, _p, _p]),
    "bil_probe_exp_rate": (_i32, [ctypes.c_int32, ctypes.c_int32, _p, _p, _p]),
    "bil_linear_logp_fwd_static": (_i32, [_p, _p, _i32, _i64, _i64, _i64, _i64, _i64, _f, _p, _i64, _p, _p, _p, _i32,
                                          _p]),
}

_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


class BilError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _build.library_path()


def load() -> ctypes.CDLL:
    """Load libbil.so for this machine; raise if it has not been built."""
    global _lib
    lib = _lib
    if lib is not None:  # loaded: no lock on the per-call path
        return lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"the CUDA library is not built ({path} missing); run "
                "`python -m invariant_token_log_gb300.build` (there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().bil_status_string(status).decode()


def contract_id() -> str:
    return load().bil_contract_id().decode()


def stream_shape(dtype: int, tile_v: int, num_tiles: int, fused: bool, entropy: bool = False) -> tuple[int, int, int]:
    """(stages, consumer warps, shared-memory bytes) of the forward kernels' pipeline."""
    st, cw, sm = _i32(0), _i32(0), _i64(0)
    check("bil_stream_shape", load().bil_stream_shape(dtype, tile_v, num_tiles, int(fused), int(entropy),
                                                      ctypes.byref(st), ctypes.byref(cw), ctypes.byref(sm)))
    return st.value, cw.value, sm.value


def check(fn: str, status: int) -> None:
    if status != OK:
        raise BilError(fn, status)
