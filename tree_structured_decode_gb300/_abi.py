"""ctypes declarations mirroring include/tree_attn.h."""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libtreeattn.so")

TA_OK = 0
STATUS_NAMES = {
    0: "TA_OK", 1: "TA_ERR_INVALID_ARG", 2: "TA_ERR_NOT_A_TREE", 3: "TA_ERR_PAGE_RANGE",
    4: "TA_ERR_UNSUPPORTED", 5: "TA_ERR_ALIGNMENT", 6: "TA_ERR_CUDA", 7: "TA_ERR_OOM",
    8: "TA_ERR_DEVICE", 9: "TA_ERR_HOST_ONLY_PLAN", 10: "TA_ERR_BUFFER_TOO_SMALL",
}
DEVERR_NONE, DEVERR_TIMEOUT, DEVERR_BOUNDS = 0, 1, 2

# Every symbol the header declares (checked by the ABI test).
EXPORTS = (
    "tree_attn_options_init", "tree_attn_plan", "tree_attn_run", "tree_attn_device_status",
    "tree_attn_plan_describe", "tree_attn_plan_get_stats", "tree_attn_plan_destroy",
    "tree_attn_status_string", "tree_attn_last_error", "tree_attn_profile_enable",
    "tree_attn_profile_read", "tree_attn_run_static", "tree_attn_append_kv",
    "tree_attn_plan_describe_schedule",
)
STATIC_SCRATCH_BYTES = 32 << 20


class TreeAttnError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))


class Options(ctypes.Structure):
    _fields_ = [
        ("gamma", ctypes.c_int64),
        ("beta", ctypes.c_int64),
        ("ts_q_set", ctypes.c_int32 * 4),
        ("ts_c", ctypes.c_int32),
        ("mma_min_rows", ctypes.c_int32),
        ("split_tokens", ctypes.c_int32),
        ("min_split_tokens", ctypes.c_int32),
        ("split_waves", ctypes.c_int32),
        ("num_sms", ctypes.c_int32),
        ("force_path", ctypes.c_int32),
        ("host_only", ctypes.c_int32),
        ("wait_timeout_us", ctypes.c_int32),
        ("force_edges", ctypes.POINTER(ctypes.c_int8)),
        ("debug_stuck_wait", ctypes.c_int32),
        ("merge_mode", ctypes.c_int32),
        ("no_pack", ctypes.c_int32),
        ("cost_model", ctypes.c_int32),
    ]


class PlanStats(ctypes.Structure):
    _fields_ = [
        ("n_nodes", ctypes.c_int32), ("n_query_tokens", ctypes.c_int32),
        ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("n_groups", ctypes.c_int32),
        ("n_groups_mma", ctypes.c_int32), ("n_units", ctypes.c_int32),
        ("grid", ctypes.c_int32), ("n_merge_tokens", ctypes.c_int32),
        ("n_partials", ctypes.c_int64), ("chunk_tokens", ctypes.c_int64),
        ("group_kv_tokens", ctypes.c_int64), ("unique_kv_tokens", ctypes.c_int64),
        ("visible_pairs", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64),
        ("metadata_bytes", ctypes.c_int64), ("plan_ms", ctypes.c_double),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_lib = None
_I32P = ctypes.POINTER(ctypes.c_int32)


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libtreeattn.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or os.environ.get("TREE_ATTN_LIB", LIB_PATH)
    if not os.path.exists(p):
        raise ImportError(
            f"libtreeattn.so not found at {p}: build it with "
            "`python -m tree_structured_decode_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(p)
    lib.tree_attn_options_init.argtypes = [ctypes.POINTER(Options)]
    lib.tree_attn_options_init.restype = None
    lib.tree_attn_plan.argtypes = [
        _I32P, ctypes.c_int32, _I32P, _I32P, _I32P, ctypes.c_int32, ctypes.c_int32,
        _I32P, _I32P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_float, ctypes.POINTER(Options), ctypes.POINTER(ctypes.c_void_p)]
    lib.tree_attn_plan.restype = ctypes.c_int
    lib.tree_attn_run.argtypes = [ctypes.c_void_p] * 7
    lib.tree_attn_run.restype = ctypes.c_int
    lib.tree_attn_run_static.argtypes = [ctypes.c_void_p] * 7
    lib.tree_attn_run_static.restype = ctypes.c_int
    lib.tree_attn_append_kv.argtypes = [ctypes.c_void_p] * 6
    lib.tree_attn_append_kv.restype = ctypes.c_int
    lib.tree_attn_device_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p, _I32P]
    lib.tree_attn_device_status.restype = ctypes.c_int
    lib.tree_attn_profile_enable.argtypes = [ctypes.c_void_p, ctypes.c_int32]
    lib.tree_attn_profile_enable.restype = ctypes.c_int
    lib.tree_attn_profile_read.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_float),
                                           ctypes.POINTER(ctypes.c_float)]
    lib.tree_attn_profile_read.restype = ctypes.c_int
    lib.tree_attn_plan_describe.argtypes = [ctypes.c_void_p, ctypes.c_char_p, ctypes.c_size_t,
                                            ctypes.POINTER(ctypes.c_size_t)]
    lib.tree_attn_plan_describe.restype = ctypes.c_int
    lib.tree_attn_plan_describe_schedule.argtypes = [ctypes.c_void_p, ctypes.c_char_p,
                                                     ctypes.c_size_t,
                                                     ctypes.POINTER(ctypes.c_size_t)]
    lib.tree_attn_plan_describe_schedule.restype = ctypes.c_int
    lib.tree_attn_plan_get_stats.argtypes = [ctypes.c_void_p, ctypes.POINTER(PlanStats)]
    lib.tree_attn_plan_get_stats.restype = ctypes.c_int
    lib.tree_attn_plan_destroy.argtypes = [ctypes.c_void_p]
    lib.tree_attn_plan_destroy.restype = None
    lib.tree_attn_status_string.argtypes = [ctypes.c_int]
    lib.tree_attn_status_string.restype = ctypes.c_char_p
    lib.tree_attn_last_error.argtypes = []
    lib.tree_attn_last_error.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().tree_attn_status_string(status).decode()


def check(status: int, where: str):
    if status != TA_OK:
        detail = load_library().tree_attn_last_error().decode(errors="replace")
        raise TreeAttnError(status, where, detail)
