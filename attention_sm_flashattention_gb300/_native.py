"""ctypes binding to libfa.so: argument marshalling only.

Every step of the attention path runs in the library's CUDA kernels; this
module only turns torch tensors into pointers, sizes and a stream handle.
There is no fallback: if the library is missing or was built for another
machine, the first call raises.
"""

from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_WORKSPACE = -3
FA_ERR_CUDA = -4
FA_ERR_DEVICE = -5
FA_ERR_TIMEOUT = -6
FA_ERR_SCRATCH_LIMIT = -7
FA_NOALLOC_SCRATCH_BYTES = 64 << 20  # fa_bwd_noalloc's static device buffer (include/fa.h)

FA_DTYPE_F16 = 0
FA_DTYPE_BF16 = 1

# Every symbol include/fa.h declares, with its ctypes signature.
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_fwd_bf16": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_bwd_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "fa_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_bwd_bf16": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_fwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "fa_reshape_and_cache": (_i, [_vp] * 5 + [_i] * 5 + [_vp]),
    "fa_fwd_sparse": (_i, [_vp] * 9 + [_i] * 9 + [_f, _i, _vp]),
    "fa_fwd_paged": (_i, [_vp] * 7 + [_i] * 9 + [_f, _i, _vp]),
    "fa_fwd_paged_split": (_i, [_vp] * 8 + [_sz] + [_i] * 10 + [_f, _i, _vp]),
    "fa_fwd_paged_split_workspace_size": (_sz, [_i] * 5),
    "fa_fwd_paged_split_count": (_i, [_i] * 8),
    "fa_bwd_ex_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i]),
    "fa_bwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "fa_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_device_status": (_i, [_vp]),
    "fa_device_status_raw": (_i, [_vp, ctypes.POINTER(ctypes.c_int)]),
    "fa_error_string": (ctypes.c_char_p, [_i]),
    "fa_selftest_wait_timeout": (_i, [_vp]),
    "fa_fwd_tile_count": (ctypes.c_longlong, [_i, _i, _i]),
    "fa_fwd_flops": (ctypes.c_double, [_i, _i, _i, _i, _i]),
    "fa_bwd_flops": (ctypes.c_double, [_i, _i, _i, _i, _i]),
    "fa_fwd_ex_flops": (ctypes.c_double, [_i, _i, _i, _i, _i, _i]),
    "fa_bwd_ex_flops": (ctypes.c_double, [_i, _i, _i, _i, _i, _i]),
}

_lib = None


class FaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {error_string(code)} (code {code})")


def lib() -> ctypes.CDLL:
    """Load libfa.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc, sm_103a)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def error_string(code: int) -> str:
    return lib().fa_error_string(code).decode()


def check(code: int, where: str) -> None:
    if code != FA_OK:
        raise FaError(code, where)
