"""ctypes loader for ``libcpattn.so`` (the C ABI declared in include/cpattn.h).

The library is built in-tree by ``build.py``.  There is no fallback: if the
shared object is missing or does not export a symbol, loading raises.
"""

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcpattn.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_CUDA = -3
ERR_TIMEOUT = -4
ERR_ALIGNMENT = -5
ERR_RANGE = -6
ERR_TOO_LARGE = -7
NOALLOC_SCRATCH_BYTES = 64 << 20
PASS_KV = 0
PASS_Q = 1
SELECT_MESSAGE = 0
SELECT_FITTED = 1

DEBUG_WAIT_LIMIT_NS = 1
DEBUG_WITHHOLD_Q = 2
DEBUG_NVTX = 3

ZIGZAG = 0
INTERLEAVE = 1
TILE_ROWS = 128

c_i32p = ctypes.POINTER(ctypes.c_int32)
vp = ctypes.c_void_p
i32 = ctypes.c_int
i64 = ctypes.c_int64

# name -> (restype, argtypes); must match include/cpattn.h
SIGNATURES = {
    "cp_shard_plan_sizes": (i32, [c_i32p, c_i32p, i32, i32, i32, c_i32p, c_i32p, c_i32p]),
    "cp_shard_plan": (i32, [vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp,
                            vp, vp]),
    "cp_attn_partial": (i32, [vp, i32, vp, i32, vp, i32, vp, i64, i64, vp, i64, i64, i32, i32,
                              i32, i32, i32, ctypes.c_float, i32, i32, vp, i32, vp, i32, i32,
                              vp, vp]),
    "cp_attn_prefill": (i32, [vp, i32, vp, i32, vp, i32, vp, i64, i64, vp, i64, i64, i32, i32,
                              i32, i32, i32, ctypes.c_float, vp, i32, vp, vp, vp]),
    "cp_attn_partial_restore": (i32, [vp, i32, vp, i32, vp, i32, vp, i64, i64, vp, i64, i64,
                                      i32, i32, i32, i32, i32, ctypes.c_float, i32, i32, vp, vp,
                                      i32, vp, i32, vp, vp]),
    "cp_attn_partial_accumulate": (i32, [vp, i32, vp, i32, vp, i32, vp, i64, i64, vp, i64, i64,
                                         i32, i32, i32, i32, i32, ctypes.c_float, i32, i32, vp,
                                         vp, vp, vp, i32, i32, vp, vp]),
    "cp_select_pass": (i32, [ctypes.c_int64, ctypes.c_int64, i32, i32, i32,
                             ctypes.POINTER(ctypes.c_double)]),
    "cp_select_pass_cost": (i32, [ctypes.c_int64, ctypes.c_int64, i32, i32, i32, i32,
                                  ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                  ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_double)]),
    "cp_lse_merge": (i32, [vp, vp, i32, i64, i64, i32, i32, i32, vp, vp, i32, vp, i32, vp, vp]),
    "cp_restore": (i32, [vp, i32, vp, i32, i64, vp, vp, vp]),
    "cp_partial_kv_workspace_size": (i32, [c_i32p, c_i32p, i32, i32, i32, i32, i32, i32,
                                           ctypes.POINTER(ctypes.c_int64), c_i32p, c_i32p]),
    "cp_partial_kv_workspace_size_segs": (i32, [vp, i32, i32, i32, i32,
                                                ctypes.POINTER(ctypes.c_int64), c_i32p, c_i32p]),
    "cp_pass_q_schedule_size": (i32, [c_i32p, c_i32p, i32, i32, i32, c_i32p, c_i32p]),
    "cp_pass_q_schedule": (i32, [c_i32p, c_i32p, i32, i32, i32, c_i32p, c_i32p, c_i32p, vp,
                                 c_i32p, c_i32p]),
    "cp_attn_pass_q": (i32, [vp, vp, c_i32p, i32, vp, i32, vp, i64, i64, vp, i64, i64, i32, i32,
                             i32, i32, i32, ctypes.c_float, vp, vp, vp, vp, vp]),
    "cp_prefill_host_workspace_size": (i32, [c_i32p, c_i32p, i32, i32, i32, i32, i32, i32, i32,
                                             i32, ctypes.POINTER(ctypes.c_int64)]),
    "cp_prefill_host": (i32, [c_i32p, c_i32p, i32, i32, i32, i32, i32, i32, i32, ctypes.c_float,
                              i32, i32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                              ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp), vp,
                              i64, vp, vp, vp, vp]),
    "cp_attn_partial_kv": (i32, [vp, i32, vp, i32, vp, i32, vp, i64, i64, vp, i64, i64, i32,
                                 i32, i32, i32, i32, ctypes.c_float, i32, i32, i32, vp, vp, i32,
                                 vp, i32, vp, i64, vp, vp]),
    "cp_attn_partial_kv_noalloc": (i32, [vp, i32, vp, i32, vp, i32, vp, i64, i64, vp, i64, i64,
                                         i32, i32, i32, i32, i32, ctypes.c_float, i32, i32, i32,
                                         vp, vp, i32, vp, i32, i64, vp, vp]),
    "cp_attn_debug": (i32, [i32, ctypes.c_longlong]),
    "cp_status_string": (ctypes.c_char_p, [i32]),
}

_lib = None


class CpAttnError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


def load():
    """Load the shared library (once).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m context_causal_attention_cp_gb300.build` (there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(code):
    try:
        return load().cp_status_string(int(code)).decode()
    except Exception:  # noqa: BLE001 - only used for messages
        return "status"


def check(code, where):
    if code != OK:
        raise CpAttnError(code, where)
