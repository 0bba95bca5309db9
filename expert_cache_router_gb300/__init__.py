"""Offloaded Mixture-of-Experts layer for GB300 (sm_103a).

Routed expert weights live in pinned, device-mapped host RAM; each layer keeps a
fixed number of GPU expert slots managed by an LRU table on the GPU. The
compute path is the CUDA library libmoe_offload.so (C ABI in
include/moe_offload.h); this package holds its build and a ctypes binding.
"""
from .binding import (MoeOffload, MoeOffloadError, DecodeGraph, PinnedHostArray, slots_for_fraction, slots_auto,
                      grouped_ffn_noalloc, plan_static, host_read_gbs)
from . import _lib

__all__ = ["MoeOffload", "MoeOffloadError", "DecodeGraph", "PinnedHostArray", "slots_for_fraction", "slots_auto",
           "grouped_ffn_noalloc", "plan_static", "host_read_gbs", "_lib"]
