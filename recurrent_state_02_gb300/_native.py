"""ctypes binding of liblinattn.so: the C ABI of include/linattn.h, same names,
argument marshalling only.  Loading fails loudly when the library has not been
built; there is no other implementation to fall back to."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblinattn.so")

LA_OK, LA_ERR_NULL, LA_ERR_SHAPE, LA_ERR_DTYPE, LA_ERR_ALIGN = 0, 1, 2, 3, 4
LA_ERR_UNSUPPORTED, LA_ERR_CUDA, LA_ERR_TIMEOUT, LA_ERR_WORKSPACE = 5, 6, 7, 8
LA_DTYPE_BF16, LA_DTYPE_FP32 = 0, 1

# Every function the header declares, with its ctypes signature.
_vp, _fp, _i, _f, _sz, _u64 = (ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                               ctypes.c_ulonglong)
SIGNATURES = {
    "la_state_init": (_i, [_fp, _fp, _i, _i, _i, _i, _vp]),
    "la_prefill_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "la_prefill_chunked": (_i, [_vp, _vp, _vp, _i, _fp, _fp, _fp, _i, _i, _i, _i, _i, _i, _f, _vp, _fp, _fp,
                                _vp, _sz, _vp]),
    "la_prefill_varlen_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "la_prefill_varlen": (_i, [_vp, _vp, _vp, _i, _fp, _fp, _fp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _fp, _fp,
                               _vp, _sz, _vp]),
    "la_prefill_chunked_noalloc": (_i, [_vp, _vp, _vp, _i, _fp, _fp, _fp, _i, _i, _i, _i, _i, _i, _f, _vp, _fp,
                                        _fp, _vp]),
    "la_decode_step": (_i, [_vp, _vp, _vp, _i, _fp, _fp, _fp, _i, _i, _i, _i, _f, _vp, _vp]),
    "la_delta_rule": (_i, [_vp, _vp, _vp, _i, _fp, _fp, _i, _i, _i, _i, _i, _vp, _fp, _vp]),
    "la_delta_chunked_workspace_bytes": (_sz, [_i, _i, _i]),
    "la_delta_rule_chunked": (_i, [_vp, _vp, _vp, _i, _fp, _fp, _i, _i, _i, _i, _i, _vp, _fp, _vp, _sz, _vp]),
    "la_backward_workspace_bytes": (_sz, [_i, _i, _i]),
    "la_prefill_backward": (_i, [_vp, _vp, _vp, _i, _fp, _fp, _fp, _i, _i, _i, _i, _i, _f, _vp, _vp, _fp, _fp,
                                 _vp, _vp, _vp, _fp, _fp, _fp, _vp, _sz, _vp]),
    "la_backward_states_bytes": (_sz, [_i, _i, _i]),
    "la_prefill_chunked_save": (_i, [_vp, _vp, _vp, _i, _fp, _fp, _fp, _i, _i, _i, _i, _i, _i, _f, _vp, _fp, _fp,
                                     _fp, _fp, _vp, _sz, _vp]),
    "la_prefill_backward_saved": (_i, [_vp, _vp, _vp, _i, _fp, _fp, _fp, _i, _i, _i, _i, _i, _vp, _vp, _fp, _fp,
                                       _fp, _fp, _vp, _vp, _vp, _fp, _fp, _fp, _vp, _sz, _vp]),
    "la_last_device_status": (_i, [_vp]),
    "la_status_string": (ctypes.c_char_p, [_i]),
    "la_debug_wait_probe": (_i, [_u64, _vp]),
}


class LinAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


_lib = None


def lib():
    """The loaded library (raises if liblinattn.so is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                "(the CUDA library is the only implementation of this package)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().la_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != LA_OK:
        raise LinAttnError(status, where)
