"""ctypes binding of libkvc.so: argument marshalling only.

Every computation happens in the CUDA library; this module converts torch
tensors to ``kvc_tensor`` descriptors, passes host int32 arrays and the
current CUDA stream, and turns non-zero status codes into ``KVCError``.  There
is no fallback: if libkvc.so is missing the import fails.
"""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
# KVC_LIB=debug loads the build whose kernels check every length and slot index
# against the capacity (bit 32 of the device error word; see include/kvc.h)
VARIANT = "debug" if os.environ.get("KVC_LIB", "") == "debug" else "release"
LIB_PATH = os.path.join(PKG, "libkvc_debug.so" if VARIANT == "debug" else "libkvc.so")

STATUS = {
    0: "KVC_OK", 1: "KVC_ERR_NULL", 2: "KVC_ERR_ZERO_BATCH", 3: "KVC_ERR_ZERO_CAPACITY",
    4: "KVC_ERR_CAPACITY_EXCEEDS_POSITIONS", 5: "KVC_ERR_ELEMENT_OVERFLOW", 6: "KVC_ERR_ALLOC",
    7: "KVC_ERR_FULL", 8: "KVC_ERR_KEY_SHAPE", 9: "KVC_ERR_VALUE_SHAPE", 10: "KVC_ERR_QUERY_SHAPE",
    11: "KVC_ERR_OUTPUT_SHAPE", 12: "KVC_ERR_DTYPE", 13: "KVC_ERR_LAYER", 14: "KVC_ERR_NONFINITE_KEY",
    15: "KVC_ERR_NONFINITE_VALUE", 16: "KVC_ERR_CUT", 17: "KVC_ERR_EMPTY_QUERY", 18: "KVC_ERR_POSITION",
    19: "KVC_ERR_CONFIG", 20: "KVC_ERR_CUDA", 21: "KVC_ERR_DEVICE", 22: "KVC_ERR_TICKET",
}
CODE = {v: k for k, v in STATUS.items()}

DTYPES = {"bf16": 0, "f32": 1, "f64": 2}
OPT_DECODE_SPLIT_ROWS, OPT_FORCE_GENERIC, OPT_SUFFIX_KERNEL, OPT_TIMING, OPT_DECODE_FUSED = 1, 2, 3, 4, 5
OPT_TEST_STALL = 6
OPT_DEVICE_LENGTHS = 7
OPT_DECODE_PDL = 8
OPT_TEST_POISON = 9
OPT_TEST_PLANT_LENGTH = 10
OPT_DECODE_TC = 11
OPT_DECODE_LANES = 12
OPT_DECODE_STREAMK = 13
KERNELS = {"rope_append": 0, "decode": 1, "decode_combine": 2, "suffix": 3, "generic_attend": 4,
           "bookkeeping": 5}

# Every entry point declared in include/kvc.h.
EXPORTS = ("kvc_abi_version", "kvc_status_string", "kvc_last_error", "kvc_create", "kvc_create_ex",
           "kvc_destroy", "kvc_append_attend", "kvc_prepare_attend", "kvc_commit", "kvc_prefill_suffix", "kvc_prefill_suffix_host", "kvc_reset", "kvc_truncate",
           "kvc_lcp", "kvc_lcp_window", "kvc_share_prefix", "kvc_block_table", "kvc_get_lengths", "kvc_get_len",
           "kvc_read_rows", "kvc_sync_lengths", "kvc_get_config", "kvc_storage", "kvc_check", "kvc_set_option",
           "kvc_kernel_stats", "kvc_reset_stats", "kvc_decode_attend_noalloc", "kvc_noalloc_check")


class KVCError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{self.name}: {message}")


class kvc_config(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("heads_q", ctypes.c_int32), ("heads_kv", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("layers", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("rope_max_positions", ctypes.c_int32), ("rope_base", ctypes.c_double),
                ("checked", ctypes.c_int32), ("device", ctypes.c_int32), ("window", ctypes.c_int32),
                ("block_rows", ctypes.c_int32), ("blocks", ctypes.c_int32)]


class kvc_tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4)]


class kvc_ticket(ctypes.Structure):
    _fields_ = [("handle", ctypes.c_void_p), ("layer", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("version", ctypes.c_uint64)]


_P = ctypes.c_void_p
_I32P = ctypes.POINTER(ctypes.c_int32)
_TP = ctypes.POINTER(kvc_tensor)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run kv_cache_append_rope_gb300.build.build() "
                          "(nvcc for sm_103a) -- there is no CPU fallback")
    lib = ctypes.CDLL(LIB_PATH)
    sig = {
        "kvc_abi_version": (ctypes.c_int32, []),
        "kvc_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "kvc_last_error": (ctypes.c_char_p, [_P]),
        "kvc_create": (ctypes.c_int, [ctypes.c_int32] * 5 + [ctypes.POINTER(_P)]),
        "kvc_create_ex": (ctypes.c_int, [ctypes.POINTER(kvc_config), ctypes.POINTER(_P)]),
        "kvc_destroy": (None, [_P]),
        "kvc_append_attend": (ctypes.c_int, [_P, ctypes.c_int32, _TP, _TP, _TP, _TP, _P]),
        "kvc_prepare_attend": (ctypes.c_int, [_P, ctypes.c_int32, _TP, _TP, _TP, _TP,
                                              ctypes.POINTER(kvc_ticket), _P]),
        "kvc_commit": (ctypes.c_int, [_P, ctypes.POINTER(kvc_ticket), ctypes.c_int32, _P]),
        "kvc_prefill_suffix": (ctypes.c_int, [_P, ctypes.c_int32, _TP, _TP, _TP, _I32P, _I32P, _TP, _P]),
        "kvc_prefill_suffix_host": (ctypes.c_int, [_P, ctypes.c_int32, _TP, _TP, _TP, _I32P, _I32P, _TP,
                                                    ctypes.c_int32, _P]),
        "kvc_reset": (ctypes.c_int, [_P, _P]),
        "kvc_truncate": (ctypes.c_int, [_P, _I32P, _P]),
        "kvc_lcp": (ctypes.c_int, [_I32P, ctypes.c_int64, _I32P, ctypes.c_int64, _I32P]),
        "kvc_lcp_window": (ctypes.c_int, [_I32P, ctypes.c_int64, _I32P, ctypes.c_int64, ctypes.c_int32, _I32P]),
        "kvc_share_prefix": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P]),
        "kvc_block_table": (ctypes.c_int, [_P, _I32P, _I32P]),
        "kvc_get_lengths": (ctypes.c_int, [_P, ctypes.c_int32, _I32P, _I32P]),
        "kvc_get_len": (ctypes.c_int, [_P, ctypes.c_int32, _I32P]),
        "kvc_read_rows": (ctypes.c_int, [_P, ctypes.c_int32, _TP, _TP, _P, _P]),
        "kvc_sync_lengths": (ctypes.c_int, [_P]),
        "kvc_get_config": (ctypes.c_int, [_P, ctypes.POINTER(kvc_config)]),
        "kvc_storage": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.POINTER(_P), ctypes.POINTER(_P),
                                       ctypes.POINTER(_P)]),
        "kvc_check": (ctypes.c_int, [_P, _P]),
        "kvc_set_option": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int64]),
        "kvc_kernel_stats": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.POINTER(ctypes.c_double),
                                            ctypes.POINTER(ctypes.c_int64)]),
        "kvc_reset_stats": (ctypes.c_int, [_P]),
        "kvc_decode_attend_noalloc": (ctypes.c_int, [_P, _P, _P, _I32P, _P, ctypes.c_int32, ctypes.c_int32,
                                                     ctypes.c_int32, ctypes.c_int32, _P]),
        "kvc_noalloc_check": (ctypes.c_int, [_P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(code):
    return lib.kvc_status_string(code).decode()


def last_error(handle=None):
    return lib.kvc_last_error(handle).decode("utf-8", "replace")


def check(status, handle=None):
    if status != 0:
        raise KVCError(status, last_error(handle) or status_string(status))


def int_array(values):
    arr = (ctypes.c_int32 * len(values))(*[int(v) for v in values])
    return arr
