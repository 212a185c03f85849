"""ctypes declarations of the C ABI in include/pa.h (libpa.so, built in-tree).

Loading fails loudly: there is no Python or CPU fallback for any call.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(HERE, "libpa.so")

PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_CUDA = -3
PA_ERR_NO_BLOCKS = -4
PA_ERR_DEVICE_BOUNDS = -5
PA_ERR_DEVICE_TIMEOUT = -6
PA_ERR_WORKSPACE = -7
PA_ERR_DEVICE_PLAN = -8
PA_ERR_HOST_MEMORY = -9

PA_F32 = 0
PA_BF16 = 1

PA_NO_ALLOC_SCRATCH_BYTES = 16 << 20  # include/pa.h

PA_KERNEL_AUTO = 0
PA_KERNEL_SIMT = 1
PA_KERNEL_MMA = 2


PA_LAYOUT_ROW = 0
PA_LAYOUT_SPLIT = 1


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("layout", ctypes.c_int32)]


class SimConfig(ctypes.Structure):
    _fields_ = [("policy", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("max_new_tokens", ctypes.c_int32), ("max_steps", ctypes.c_int32),
                ("total_slots", ctypes.c_int64)]


class SimResult(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("steps", "admitted", "completed", "preemptions", "blocked_steps",
                                              "peak_running", "sum_used", "sum_held", "sum_running")] + \
               [("utilization", ctypes.c_double)]


class DecodeOpts(ctypes.Structure):
    _fields_ = [("num_splits", ctypes.c_int32), ("kernel", ctypes.c_int32),
                ("ev_partial_begin", ctypes.c_void_p), ("ev_partial_end", ctypes.c_void_p),
                ("shared_plan", ctypes.c_void_p), ("host_seq_lens", ctypes.c_void_p)]


class SharedPlanInfo(ctypes.Structure):
    _fields_ = [("num_groups", ctypes.c_int32), ("num_members", ctypes.c_int32),
                ("shared_blocks", ctypes.c_int64), ("saved_blocks", ctypes.c_int64)]


# symbol -> (restype, argtypes)
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_PI32 = ctypes.POINTER(ctypes.c_int32)
_PI64 = ctypes.POINTER(ctypes.c_int64)
_DESC = ctypes.POINTER(CacheDesc)
_OPTS = ctypes.POINTER(DecodeOpts)

SIGNATURES = {
    "pa_status_string": (ctypes.c_char_p, [_I32]),
    "pa_shared_plan_ints": (ctypes.c_size_t, [_I32]),
    "pa_shared_plan_build": (_I32, [_PI32, _I32, _PI32, _I32, _I32, _I32, _I32, _I32, _PI32, ctypes.c_size_t,
                                    ctypes.POINTER(SharedPlanInfo)]),
    "pa_version": (ctypes.c_char_p, []),
    "pa_reshape_and_cache": (_I32, [_P, _P, _P, _I32, _P, _P, _DESC, _P]),
    "pa_copy_blocks": (_I32, [_P, _P, _DESC, _P, _I32, _P]),
    "pa_decode_workspace_bytes": (ctypes.c_size_t, [_DESC, _I32, _I32, _OPTS]),
    "pa_decode": (_I32, [_P, _P, _P, _P, _DESC, _P, _I32, _P, _I32, _I32, ctypes.c_float, _P,
                         ctypes.c_size_t, _OPTS, _P]),
    "pa_decode_default_splits": (_I32, [_DESC, _I32, _OPTS]),
    "pa_decode_shared_tc": (_I32, [_DESC, _I32, _I32, _OPTS]),
    "pa_decode_launch_count": (_I32, [_DESC, _I32, _I32, _I32, _OPTS]),
    "pa_decode_no_alloc": (_I32, [_P, _P, _P, _P, _DESC, _P, _I32, _P, _I32, _I32, ctypes.c_float, _OPTS, _P]),
    "pa_split_range": (None, [_I64, _I32, _I32, _PI64, _PI64]),
    "pa_split_owner": (_I32, [_I64, _I32, _I64]),
    "pa_get_device_error": (_I32, [_P]),
    "pa_selftest_wait_timeout": (_I32, [_I64, _P]),
    "pa_bm_create": (_P, [_I32, _I32, _PI32]),
    "pa_bm_destroy": (None, [_P]),
    "pa_bm_new_seq": (_I32, [_P, _I32, _PI32]),
    "pa_bm_fork": (_I32, [_P, _I32, _PI32]),
    "pa_bm_free_seq": (_I32, [_P, _I32]),
    "pa_bm_append_token": (_I32, [_P, _I32, _PI32, _PI32, _PI32]),
    "pa_bm_append_tokens": (_I32, [_P, _I32, _I32, _PI32, _PI32, _PI32]),
    "pa_bm_seq_len": (_I32, [_P, _I32, _PI32, _PI32]),
    "pa_bm_block_table": (_I32, [_P, _I32, _PI32, _I32, _PI32]),
    "pa_bm_physical_index": (_I32, [_P, _I32, _I32, _PI32]),
    "pa_bm_refcount": (_I32, [_P, _I32, _PI32]),
    "pa_bm_stats": (_I32, [_P, _PI32, _PI32, _PI32]),
    "pa_bm_export": (_I32, [_P, _PI32, _I32, _I32, _PI32, _PI32]),
    "pa_bm_new_seq_cached": (_I32, [_P, _PI32, _I32, _PI32, _PI32]),
    "pa_bm_slots": (_I32, [_P, _I32, _I32, _I32, _PI32]),
    "pa_bm_cache_stats": (_I32, [_P, _PI32, _PI64, _PI64]),
    "pa_bm_set_prefix_retention": (_I32, [_P, _I32]),
    "pa_bm_evictable": (_I32, [_P, _PI32]),
    "pa_sim_run": (_I32, [ctypes.POINTER(SimConfig), _PI32, _PI32, _PI32, _I32, ctypes.POINTER(SimResult)]),
}

_lib = None


def load():
    """The loaded libpa.so with argument types set.  Raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY):
            raise RuntimeError(
                "libpa.so is not built (%s). Run `python -c \"import __graft_entry__ as g; g.build()\"` "
                "or `python paged_kv_cache_150_gb300/build.py`; there is no fallback path." % LIBRARY)
        lib = ctypes.CDLL(LIBRARY)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class PagedAttentionError(RuntimeError):
    def __init__(self, call, status):
        self.status = int(status)
        msg = load().pa_status_string(int(status))
        super().__init__("%s failed: %s (%d)" % (call, msg.decode() if msg else "?", status))


def check(call, status):
    if status != PA_OK:
        raise PagedAttentionError(call, status)
