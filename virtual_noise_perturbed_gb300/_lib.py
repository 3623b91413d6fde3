"""ctypes loader for ``libvn.so`` (the C ABI in ``include/vn.h``).

Only argument marshalling lives in Python: every step of the computation runs
in the library's CUDA kernels. There is no fallback: if the library has not
been built, every entry point raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libvn.so")

# vn_status
VN_OK = 0
STATUS_NAMES = {
    0: "VN_OK", 1: "VN_ERR_NULL", 2: "VN_ERR_SHAPE", 3: "VN_ERR_DTYPE", 4: "VN_ERR_VALUE",
    5: "VN_ERR_ALIGN", 6: "VN_ERR_OVERFLOW", 7: "VN_ERR_TIMEOUT", 8: "VN_ERR_CUDA",
    9: "VN_ERR_DEVICE", 10: "VN_ERR_PATH",
}
# vn_dtype
VN_F32, VN_BF16 = 0, 1
# vn_path
VN_PATH_AUTO, VN_PATH_FFMA, VN_PATH_TC = 0, 1, 2
# vn_act
VN_ACT_NONE, VN_ACT_TANH = 0, 1
# vn_noise
VN_NOISE_UNIFORM, VN_NOISE_GAUSSIAN = 0, 1

#: Every symbol the header declares, with (restype, argtypes).
_P, _I64, _U64, _I, _D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_double
SIGNATURES = {
    "vn_perturbed_linear": (_I, [_P, _I, _I, _P, _I, _P, _I, _P, _I64, _I64, _I64, _I64, _D, _U64,
                                 _P, _I, _P]),
    "vn_perturbed_linear_ex": (_I, [_P, _I, _I, _P, _I, _P, _I, _P, _I64, _I64, _I64, _I64, _D,
                                    _U64, _P, _I, _I, _I, _P]),
    "vn_perturbed_linear_kind": (_I, [_P, _I, _I, _P, _I, _P, _I, _P, _I64, _I64, _I64, _I64, _D,
                                      _U64, _P, _I, _I, _I, _I, _P]),
    "vn_weight_gradient": (_I, [_P, _P, _I64, _I64, _I64, _D, _U64, _P, _P]),
    "vn_bias_gradient": (_I, [_P, _P, _I64, _I64, _D, _U64, _P, _P]),
    "vn_noise_dump": (_I, [_P, _I64, _I64, _U64, _P, _P]),
    "vn_reduce_metric": (_I, [_P, _P, _I64, _I64, _D, _U64, _P, _P]),
    "vn_perturbed_mlp": (_I, [_P, _I, _I, _I64, _P, _P, _P, _P, _P, _I64, _I64, _D, _I, _P, _P]),
    "vn_perturbed_mlp_ex": (_I, [_P, _I, _I, _I64, _P, _P, _P, _P, _P, _I64, _I64, _D, _I, _I, _P,
                                 _P]),
    "vn_centered_ranks": (_I, [_P, _I64, _P, _P]),
    "vn_es_update": (_I, [_P, _P, _I64, _D, _P]),
    "vn_noise_dump_ex": (_I, [_P, _I64, _I64, _U64, _I, _P, _P]),
    "vn_gradient_ex": (_I, [_P, _P, _I64, _I64, _D, _U64, _I, _P, _P]),
    "vn_gradient_update": (_I, [_P, _P, _I64, _I64, _D, _U64, _I, _D, _P, _P, _P]),
    "vn_device_status": (_I, [_P]),
    "vn_hash_probe": (_I, [_I64, _U64, _I64, _I64, _P, _P]),
    "vn_testhook_linear_tc_withhold": (_I, [_P, _I, _I, _P, _I, _P, _I, _P, _I64, _I64, _I64, _I64,
                                           _D, _U64, _P, _I, _I64, _D, _P]),
    "vn_status_string": (ctypes.c_char_p, [_I]),
    "vn_last_error_message": (ctypes.c_char_p, []),
    "vn_perturbed_linear_path": (_I, [_P, _I, _I, _P, _I, _I64, _I64, _I64]),
    "vn_version": (_I, []),
}

_lock = threading.Lock()
_lib = None


class VNError(RuntimeError):
    """A non-VN_OK status from the library."""

    def __init__(self, status: int, where: str):
        lib = _lib
        text = lib.vn_status_string(status).decode() if lib else STATUS_NAMES.get(status, "?")
        if status == 8 and lib is not None:
            text += f" ({lib.vn_last_error_message().decode()})"
        super().__init__(f"{where}: {text}")
        self.status = status


def load() -> ctypes.CDLL:
    """Load libvn.so once; raise if it is missing (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; build it with "
                    "`python -m virtual_noise_perturbed_gb300.build` (needs nvcc)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def check(status: int, where: str) -> None:
    if status != VN_OK:
        raise VNError(status, where)
