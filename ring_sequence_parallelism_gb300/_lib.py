"""ctypes binding of libringattn.so (the C ABI in include/ringattn.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  Loading fails loudly when the library has not been built; there is
no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_HERE, "libringattn.so")

RING_OK = 0
RING_ERR_INVALID_ARG = -1
RING_ERR_UNSUPPORTED = -2
RING_ERR_CUDA = -3
RING_ERR_TIMEOUT = -4
RING_ERR_OOM = -5
STATUS_NAMES = {0: "RING_OK", -1: "RING_ERR_INVALID_ARG", -2: "RING_ERR_UNSUPPORTED", -3: "RING_ERR_CUDA",
                -4: "RING_ERR_TIMEOUT", -5: "RING_ERR_OOM"}

RING_LAYOUT_CONTIGUOUS = 0
RING_LAYOUT_STRIPED = 1
RING_LAYOUT_ZIGZAG = 2
RING_BLOCK_SKIP, RING_BLOCK_FULL, RING_BLOCK_DIAG, RING_BLOCK_PARTIAL = 0, 1, 2, 3
(RING_OPT_ROTATION, RING_OPT_TIMING, RING_OPT_WAIT_LIMIT_NS, RING_OPT_DEBUG_DROP_V_LOADS, RING_OPT_WINDOW,
 RING_OPT_BWD_LAP, RING_OPT_FWD_LAP) = 0, 1, 2, 3, 4, 5, 6

# Every symbol include/ringattn.h declares, with (restype, argtypes).
_vp = ctypes.c_void_p
_i = ctypes.c_int
_ll = ctypes.c_longlong
_pll = ctypes.POINTER(ctypes.c_longlong)
_pi = ctypes.POINTER(ctypes.c_int)
_pf = ctypes.POINTER(ctypes.c_float)


class RingState(ctypes.Structure):
    _fields_ = [("m", _vp), ("l", _vp), ("o", _vp)]


SIGNATURES = {
    "ring_attn_create": (_i, [ctypes.POINTER(_vp), _i, _i, _ll, _i, _i, _i, _i]),
    "ring_attn_create_gqa": (_i, [ctypes.POINTER(_vp), _i, _i, _i, _ll, _i, _i, _i, _i]),
    "ring_attn_decode_workspace_size": (_i, [_vp, _ll, ctypes.POINTER(ctypes.c_size_t)]),
    "ring_attn_decode": (_i, [_vp, _vp, _vp, _vp, _ll, _vp, _vp, _vp, _vp]),
    "ring_attn_destroy": (_i, [_vp]),
    "ring_attn_last_error": (ctypes.c_char_p, []),
    "ring_attn_workspace_size": (_i, [_vp, ctypes.POINTER(ctypes.c_size_t)]),
    "ring_attn_plan_block": (_i, [_vp, _i, _i, _pi, _pi, _pll]),
    "ring_attn_plan_mask": (_i, [_vp, _i, _i, ctypes.c_longlong, _pll, _pll]),
    "ring_attn_plan_key_range": (_i, [_vp, _i, _i, ctypes.c_longlong, _pll, _pll]),
    "ring_attn_shard_work": (_i, [_vp, _pll, _pll]),
    "ring_attn_step_work": (_i, [_vp, _i, _pll, _pll]),
    "ring_attn_state_init": (_i, [_vp, RingState, _vp]),
    "ring_attn_block_partial": (_i, [_vp, _i, _i, _vp, _vp, _vp, RingState, _i, _vp]),
    "ring_attn_merge": (_i, [_vp, RingState, RingState, _vp]),
    "ring_attn_finalize": (_i, [_vp, _i, RingState, _vp, _vp, _vp]),
    "ring_attn_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ring_attn_fwd_host": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ring_attn_set_option": (_i, [_vp, _i, _ll]),
    "ring_attn_set_segments": (_i, [_vp, _pll, _i]),
    "ring_attn_get_timing": (_i, [_vp, _pf, _pf, _pf, _pf]),
    "ring_attn_get_release_wait": (_i, [_vp, _pf]),
    "ring_attn_check": (_i, [_vp, _vp]),
    "ring_attn_fwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ring_attn_bwd_workspace_size": (_i, [_vp, ctypes.POINTER(ctypes.c_size_t)]),
    "ring_attn_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ring_attn_get_bwd_timing": (_i, [_vp, _pf, _pf, _pf]),
}

_LIB = None


class RingAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def load(path: str = LIBRARY):
    """Load the CUDA library (built in-tree by ``build.build()``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()'). "
            "There is no CPU fallback.")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def check(status: int):
    if status != RING_OK:
        msg = load().ring_attn_last_error()
        raise RingAttnError(status, msg.decode() if msg else "")
    return status
