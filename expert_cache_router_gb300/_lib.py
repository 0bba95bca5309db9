"""ctypes declarations of libmoe_offload.so (the C ABI in include/moe_offload.h)."""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoe_offload.so")

MOE_OK, MOE_ERR_INVALID, MOE_ERR_CUDA, MOE_ERR_OOM, MOE_ERR_CAPTURE, MOE_ERR_DEVICE_STATUS = range(6)
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID", 2: "MOE_ERR_CUDA", 3: "MOE_ERR_OOM",
                4: "MOE_ERR_CAPTURE", 5: "MOE_ERR_DEVICE_STATUS"}
MOE_DTYPE_BF16, MOE_DTYPE_FP8_E4M3_B128 = 0, 1
MOE_DEV_BAD_EXPERT_ID, MOE_DEV_BAD_SLOT_ID, MOE_DEV_AUDIT_FAILED, MOE_DEV_BAD_COUNT, MOE_DEV_TIMEOUT = 1, 2, 4, 8, 16
MOE_TRACE_FIELDS = 16
# decode trace record fields (moe_offload_trace_read), in order
TRACE_FIELD_NAMES = ("head_wait", "head_logits", "head_topk", "head_done", "gate_first", "host_first",
                     "host_done", "copy_done", "gate_done", "down_first", "down_waits", "down_done", "down_out")
TRACE_MIN_FIELDS = ("gate_first", "host_first", "down_first")

# Every symbol the header declares, in declaration order.
EXPORTS = [
    "moe_offload_slots_for_fraction", "moe_offload_slots_auto", "moe_offload_create", "moe_offload_route_topk",
    "moe_offload_slot_ensure", "moe_offload_miss_copy", "moe_offload_grouped_ffn",
    "moe_offload_decode_layer", "moe_offload_audit", "moe_offload_get_stats",
    "moe_offload_read_table", "moe_offload_debug_write_table", "moe_offload_profile_read", "moe_offload_read_misses", "moe_offload_prefetch",
    "moe_offload_read_route_counts", "moe_offload_plan_static", "moe_offload_set_placement",
    "moe_offload_read_prefetch", "moe_offload_read_slot",
    "moe_offload_read_slot_scales", "moe_offload_set_shared_expert", "moe_offload_reset",
    "moe_offload_host_alloc", "moe_offload_host_free", "moe_offload_prefill_times", "moe_offload_prefill_gemm_ms",
    "moe_offload_device_bytes", "moe_offload_get_config", "moe_offload_read_routing",
    "moe_offload_host_read_gbs", "moe_offload_debug_wait", "moe_offload_trace_enable", "moe_offload_trace_read",
    "moe_offload_graph_create", "moe_offload_graph_launch",
    "moe_offload_graph_launch_host", "moe_offload_graph_times", "moe_offload_graph_kernel_count",
    "moe_offload_graph_destroy", "moe_offload_grouped_ffn_noalloc", "moe_offload_last_error",
    "moe_offload_destroy",
]


class Config(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int), ("num_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("hidden", ctypes.c_int), ("inter", ctypes.c_int), ("num_slots", ctypes.c_int),
                ("dtype", ctypes.c_int), ("renormalize", ctypes.c_int),
                ("max_tokens_graph", ctypes.c_int), ("shared_expert", ctypes.c_int),
                ("prefetch_n", ctypes.c_int), ("auto_reserve_bytes", ctypes.c_ulonglong)]


class Stats(ctypes.Structure):
    _fields_ = [("calls", ctypes.c_uint64), ("hits", ctypes.c_uint64), ("misses", ctypes.c_uint64),
                ("spills", ctypes.c_uint64), ("bytes_copied", ctypes.c_uint64),
                ("staged_calls", ctypes.c_uint64), ("staged_bytes", ctypes.c_uint64),
                ("prefetch_installs", ctypes.c_uint64), ("prefetch_hits", ctypes.c_uint64),
                ("prefetch_bytes", ctypes.c_uint64), ("device_status", ctypes.c_uint32)]


_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i32p = ctypes.POINTER(ctypes.c_int32)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_ip = ctypes.POINTER(ctypes.c_int)
_st = ctypes.c_int


def _declare(L):
    L.moe_offload_slots_for_fraction.restype = ctypes.c_int
    L.moe_offload_slots_for_fraction.argtypes = [ctypes.c_double, ctypes.c_int, ctypes.c_int]
    L.moe_offload_slots_auto.restype = ctypes.c_int
    L.moe_offload_slots_auto.argtypes = [ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_size_t]
    L.moe_offload_create.restype = _st
    L.moe_offload_create.argtypes = [ctypes.POINTER(Config), ctypes.c_int, ctypes.POINTER(_vp),
                                     ctypes.POINTER(_vp), _vp, _vp, ctypes.POINTER(_vp),
                                     ctypes.POINTER(_vp)]
    L.moe_offload_route_topk.restype = _st
    L.moe_offload_route_topk.argtypes = [_vp, ctypes.c_int, _vp, ctypes.c_int, _vp, _vp, _vp]
    L.moe_offload_slot_ensure.restype = _st
    L.moe_offload_slot_ensure.argtypes = [_vp, ctypes.c_int, _vp, ctypes.c_int, _vp, _vp]
    L.moe_offload_miss_copy.restype = _st
    L.moe_offload_miss_copy.argtypes = [_vp, ctypes.c_int, _vp]
    L.moe_offload_grouped_ffn.restype = _st
    L.moe_offload_grouped_ffn.argtypes = [_vp, ctypes.c_int, _vp, _vp, _vp, ctypes.c_int, _vp, _vp]
    L.moe_offload_decode_layer.restype = _st
    L.moe_offload_decode_layer.argtypes = [_vp, ctypes.c_int, _vp, ctypes.c_int, _vp, _vp]
    L.moe_offload_audit.restype = _st
    L.moe_offload_audit.argtypes = [_vp, ctypes.c_int, _vp]
    L.moe_offload_get_stats.restype = _st
    L.moe_offload_get_stats.argtypes = [_vp, ctypes.c_int, ctypes.POINTER(Stats)]
    L.moe_offload_read_table.restype = _st
    L.moe_offload_read_table.argtypes = [_vp, ctypes.c_int, _vp, _vp, _vp, _vp]
    L.moe_offload_profile_read.restype = _st
    L.moe_offload_profile_read.argtypes = [_vp, ctypes.c_int, _vp, _vp, _vp, _vp, ctypes.c_int]
    L.moe_offload_debug_write_table.restype = _st
    L.moe_offload_debug_write_table.argtypes = [_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64]
    L.moe_offload_read_misses.restype = _st
    L.moe_offload_read_misses.argtypes = [_vp, ctypes.c_int, _vp, _vp, ctypes.c_int, _ip, _ip]
    L.moe_offload_prefetch.restype = _st
    L.moe_offload_prefetch.argtypes = [_vp, ctypes.c_int, _vp, ctypes.c_int, _vp]
    L.moe_offload_read_route_counts.restype = _st
    L.moe_offload_read_route_counts.argtypes = [_vp, ctypes.c_int, _vp]
    L.moe_offload_plan_static.restype = ctypes.c_int
    L.moe_offload_plan_static.argtypes = [_vp, ctypes.c_int, ctypes.c_int, _vp]
    L.moe_offload_set_placement.restype = _st
    L.moe_offload_set_placement.argtypes = [_vp, ctypes.c_int, _vp, ctypes.c_int, _vp]
    L.moe_offload_read_prefetch.restype = _st
    L.moe_offload_read_prefetch.argtypes = [_vp, ctypes.c_int, _vp, _vp, _vp, _vp, _vp, ctypes.c_int]
    L.moe_offload_read_slot.restype = _st
    L.moe_offload_read_slot.argtypes = [_vp, ctypes.c_int, ctypes.c_int, _vp, _vp]
    L.moe_offload_read_slot_scales.restype = _st
    L.moe_offload_read_slot_scales.argtypes = [_vp, ctypes.c_int, ctypes.c_int, _vp, _vp]
    L.moe_offload_set_shared_expert.restype = _st
    L.moe_offload_set_shared_expert.argtypes = [_vp, ctypes.c_int, _vp, _vp, _vp, _vp]
    L.moe_offload_reset.restype = _st
    L.moe_offload_reset.argtypes = [_vp]
    L.moe_offload_host_alloc.restype = _st
    L.moe_offload_host_alloc.argtypes = [ctypes.c_size_t, ctypes.POINTER(_vp)]
    L.moe_offload_host_free.restype = None
    L.moe_offload_host_free.argtypes = [_vp]
    L.moe_offload_prefill_times.restype = _st
    L.moe_offload_prefill_times.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp]
    L.moe_offload_prefill_gemm_ms.restype = _st
    L.moe_offload_prefill_gemm_ms.argtypes = [_vp, _vp]
    L.moe_offload_device_bytes.restype = ctypes.c_size_t
    L.moe_offload_device_bytes.argtypes = [_vp]
    L.moe_offload_get_config.restype = _st
    L.moe_offload_get_config.argtypes = [_vp, ctypes.POINTER(Config), ctypes.POINTER(ctypes.c_size_t)]
    L.moe_offload_read_routing.restype = _st
    L.moe_offload_read_routing.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int, _ip]
    L.moe_offload_host_read_gbs.restype = _st
    L.moe_offload_host_read_gbs.argtypes = [ctypes.c_int, _vp, ctypes.c_size_t, ctypes.c_int,
                                            ctypes.POINTER(ctypes.c_double)]
    L.moe_offload_debug_wait.restype = _st
    L.moe_offload_debug_wait.argtypes = [_vp, ctypes.c_longlong, ctypes.c_int]
    L.moe_offload_trace_enable.restype = _st
    L.moe_offload_trace_enable.argtypes = [_vp, ctypes.c_int]
    L.moe_offload_trace_read.restype = _st
    L.moe_offload_trace_read.argtypes = [_vp, _vp, ctypes.c_int]
    L.moe_offload_graph_create.restype = _st
    L.moe_offload_graph_create.argtypes = [_vp, ctypes.c_int, _vp, _vp, ctypes.c_int, ctypes.POINTER(_vp)]
    L.moe_offload_graph_launch.restype = _st
    L.moe_offload_graph_launch.argtypes = [_vp, _vp]
    L.moe_offload_graph_launch_host.restype = _st
    L.moe_offload_graph_launch_host.argtypes = [_vp, _vp, _vp, _vp]
    L.moe_offload_graph_times.restype = _st
    L.moe_offload_graph_times.argtypes = [_vp, _vp, _vp, _vp]
    L.moe_offload_graph_kernel_count.restype = ctypes.c_int
    L.moe_offload_graph_kernel_count.argtypes = [_vp]
    L.moe_offload_graph_destroy.restype = None
    L.moe_offload_graph_destroy.argtypes = [_vp]
    L.moe_offload_grouped_ffn_noalloc.restype = _st
    L.moe_offload_grouped_ffn_noalloc.argtypes = [_vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp,
                                                  _vp, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp]
    L.moe_offload_last_error.restype = ctypes.c_char_p
    L.moe_offload_last_error.argtypes = [_vp]
    L.moe_offload_destroy.restype = None
    L.moe_offload_destroy.argtypes = [_vp]
    return L


def load(path: Optional[str] = None):
    """Load the built library (LIB_PATH unless a path is given). Raises if it has not been
    built: there is no fallback."""
    global _lib
    path = path or LIB_PATH
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libmoe_offload.so not found at {path}; build it first with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` "
                    "or `python expert_cache_router_gb300/build.py`")
            _lib = _declare(ctypes.CDLL(path))
        return _lib
