"""Python binding of the offloaded MoE layer (argument marshalling only).

Every method maps one-to-one onto a C entry point of libmoe_offload.so with the
same name; tensors are passed as device pointers and streams as CUDA stream
handles. PyTorch only supplies device memory and streams; all arithmetic runs
in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import numpy as np

from . import _lib as C


class MoeOffloadError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{C.STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _ptr(t) -> int:
    """Address of a torch tensor, numpy array or raw int."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def slots_for_fraction(fraction: float, num_experts: int, top_k: int) -> int:
    return C.load().moe_offload_slots_for_fraction(float(fraction), int(num_experts), int(top_k))


def slots_auto(free_bytes: int, num_layers: int, num_experts: int, top_k: int, expert_bytes: int,
               reserve_bytes: int = int(2.5 * 2**30)) -> int:
    """Slots per layer that fit the free device memory minus a reserve (-1: not even top_k)."""
    return C.load().moe_offload_slots_auto(int(free_bytes), int(reserve_bytes), int(num_layers),
                                          int(num_experts), int(top_k), int(expert_bytes))


def grouped_ffn_noalloc(w13, w2, num_experts: int, hidden: int, inter: int, x, ids, w, T: int,
                        top_k: int, out, status=None, stream=None) -> None:
    """moe_offload_grouped_ffn_noalloc: the grouped FFN for callers that cannot
    allocate device memory (their runtime owns every byte); scratch is a fixed
    library-owned device array, so overlapping calls on one GPU race."""
    L = C.load()
    st = L.moe_offload_grouped_ffn_noalloc(_ptr(w13), _ptr(w2), num_experts, hidden, inter, _ptr(x), _ptr(ids),
                                          _ptr(w), T, top_k, _ptr(out), _ptr(status), _stream(stream))
    if st != C.MOE_OK:
        raise MoeOffloadError(st, L.moe_offload_last_error(None).decode())


def host_read_gbs(host_array, device: int = 0, reps: int = 5) -> float:
    """moe_offload_host_read_gbs: best GB/s of SM loads reading a pinned, mapped host
    array (e.g. a PinnedHostArray's array) from the GPU."""
    L = C.load()
    g = ctypes.c_double()
    nbytes = int(host_array.nbytes) & ~15
    st = L.moe_offload_host_read_gbs(int(device), _ptr(host_array), nbytes, int(reps), ctypes.byref(g))
    if st != C.MOE_OK:
        raise MoeOffloadError(st, L.moe_offload_last_error(None).decode())
    return float(g.value)


def plan_static(counts, num_slots: int) -> np.ndarray:
    """moe_offload_plan_static: the num_slots most-routed experts (ties: lower id)."""
    c = np.ascontiguousarray(counts, dtype=np.uint64)
    out = np.empty(min(num_slots, c.size), np.int32)
    n = C.load().moe_offload_plan_static(c.ctypes.data, int(c.size), int(num_slots), out.ctypes.data)
    if n < 0:
        raise ValueError("plan_static: bad arguments")
    return out[:n]


class PinnedHostArray:
    """Host memory from moe_offload_host_alloc (pinned, mapped), viewed as a numpy
    array; freed when the object is closed or collected."""

    def __init__(self, shape, dtype=np.uint16):
        self._L = C.load()
        nbytes = int(np.prod(shape)) * np.dtype(dtype).itemsize
        p = ctypes.c_void_p()
        st = self._L.moe_offload_host_alloc(nbytes, ctypes.byref(p))
        if st != C.MOE_OK:
            raise MoeOffloadError(st, self._L.moe_offload_last_error(None).decode())
        self.ptr = p.value
        buf = (ctypes.c_byte * nbytes).from_address(self.ptr)
        self.array = np.frombuffer(buf, dtype=dtype, count=int(np.prod(shape))).reshape(shape)

    def close(self):
        if getattr(self, "ptr", None):
            self.array = None
            self._L.moe_offload_host_free(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MoeOffload:
    """One handle: host expert store (pinned + mapped), slots, LRU tables.

    host_w13[l]: [E,2I,H] host array of layer l (numpy uint16 for bf16, uint8 e4m3
                 codes for fp8, or a raw address)
    host_w2[l] : [E,H,I] host array, same element type
    host_s13[l], host_s2[l]: fp8 only, fp32 host arrays [E,2I/128,H/128], [E,H/128,I/128]
    router[l]  : [E,H] bf16 device tensor
    dtype      : "bf16" or "fp8" (e4m3 with 128x128 block scales)
    shared_expert: every layer adds an always-resident shared expert (set_shared_expert)
    prefetch_n : router lookahead, experts per layer prefetched from the previous layer's input
    num_slots  : slots per layer, or 0 for `auto` sizing from the device's free memory less
                 auto_reserve_bytes (0: the library's 2.5 GiB default); num_slots then holds
                 the count chosen and auto_free_bytes the free memory the sizing read
    The caller keeps all of them alive until close().
    """

    def __init__(self, *, num_layers: int, num_experts: int, top_k: int, hidden: int, inter: int,
                 num_slots: int, host_w13: Sequence, host_w2: Sequence, router: Sequence,
                 renormalize: bool = True, max_tokens_graph: int = 8, device: int = 0,
                 dtype: str = "bf16", host_s13: Optional[Sequence] = None,
                 host_s2: Optional[Sequence] = None, shared_expert: bool = False, prefetch_n: int = 0,
                 auto_reserve_bytes: int = 0):
        self._L = C.load()
        code = {"bf16": C.MOE_DTYPE_BF16, "fp8": C.MOE_DTYPE_FP8_E4M3_B128}[dtype]
        self.dtype = dtype
        self.cfg = C.Config(num_layers, num_experts, top_k, hidden, inter, num_slots, code,
                            int(bool(renormalize)), max_tokens_graph, int(bool(shared_expert)), int(prefetch_n),
                            int(auto_reserve_bytes))
        self.prefetch_n = int(prefetch_n)
        self.num_layers, self.num_experts, self.top_k = num_layers, num_experts, top_k
        self.hidden, self.inter, self.num_slots = hidden, inter, num_slots
        self.max_tokens_graph = max_tokens_graph
        self._keep = (list(host_w13), list(host_w2), list(router), host_s13, host_s2)
        self._shared_keep = {}
        arr = ctypes.c_void_p * num_layers
        p13 = arr(*[_ptr(a) for a in host_w13])
        p2 = arr(*[_ptr(a) for a in host_w2])
        pr = arr(*[_ptr(a) for a in router])
        ps13 = arr(*[_ptr(a) for a in host_s13]) if host_s13 is not None else None
        ps2 = arr(*[_ptr(a) for a in host_s2]) if host_s2 is not None else None
        h = ctypes.c_void_p()
        st = self._L.moe_offload_create(ctypes.byref(self.cfg), device, p13, p2, ps13, ps2, pr,
                                        ctypes.byref(h))
        if st != C.MOE_OK:
            raise MoeOffloadError(st, self._L.moe_offload_last_error(None).decode())
        self.h = h
        got = C.Config()
        free = ctypes.c_size_t()
        self._check(self._L.moe_offload_get_config(h, ctypes.byref(got), ctypes.byref(free)))
        self.num_slots = int(got.num_slots)
        self.auto_free_bytes = int(free.value)

    # -- helpers
    def _check(self, st: int) -> None:
        if st != C.MOE_OK:
            raise MoeOffloadError(st, self._L.moe_offload_last_error(self.h).decode())

    def close(self) -> None:
        if getattr(self, "h", None):
            self._L.moe_offload_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    # -- entry points
    def route_topk(self, layer, x, T, ids, w, stream=None):
        self._check(self._L.moe_offload_route_topk(self.h, layer, _ptr(x), T, _ptr(ids), _ptr(w),
                                                   _stream(stream)))

    def slot_ensure(self, layer, ids, T, slot_ids, stream=None):
        self._check(self._L.moe_offload_slot_ensure(self.h, layer, _ptr(ids), T, _ptr(slot_ids),
                                                    _stream(stream)))

    def miss_copy(self, layer, stream=None):
        self._check(self._L.moe_offload_miss_copy(self.h, layer, _stream(stream)))

    def grouped_ffn(self, layer, x, slot_ids, w, T, out, stream=None):
        self._check(self._L.moe_offload_grouped_ffn(self.h, layer, _ptr(x), _ptr(slot_ids), _ptr(w), T,
                                                    _ptr(out), _stream(stream)))

    def decode_layer(self, layer, x, T, out, stream=None):
        self._check(self._L.moe_offload_decode_layer(self.h, layer, _ptr(x), T, _ptr(out),
                                                     _stream(stream)))

    def audit(self, layer, stream=None):
        self._check(self._L.moe_offload_audit(self.h, layer, _stream(stream)))

    def get_stats(self, layer: int = -1, check: bool = True) -> dict:
        s = C.Stats()
        st = self._L.moe_offload_get_stats(self.h, layer, ctypes.byref(s))
        d = {f: int(getattr(s, f)) for f, _ in C.Stats._fields_}
        if check or st not in (C.MOE_OK, C.MOE_ERR_DEVICE_STATUS):
            self._check(st)
        return d

    def read_table(self, layer: int):
        S, E = self.num_slots, self.num_experts
        se = np.empty(S, np.int32)
        es = np.empty(E, np.int32)
        stamp = np.empty(S, np.uint32)
        clock = np.zeros(1, np.uint32)
        self._check(self._L.moe_offload_read_table(self.h, layer, se.ctypes.data, es.ctypes.data,
                                                   stamp.ctypes.data, clock.ctypes.data))
        return se, es, stamp, int(clock[0])

    def profile_read(self, layer: int = -1, clear: bool = False) -> dict:
        """Eager decode profile (MOE_OFFLOAD_PROFILE=1): profiled calls and summed phase times (ms)."""
        calls = ctypes.c_longlong()
        ms = [ctypes.c_double() for _ in range(3)]
        self._check(self._L.moe_offload_profile_read(self.h, layer, ctypes.byref(calls), ctypes.byref(ms[0]),
                                                     ctypes.byref(ms[1]), ctypes.byref(ms[2]), int(bool(clear))))
        return {"calls": calls.value, "head_ms": ms[0].value, "gate_up_ms": ms[1].value, "down_ms": ms[2].value}

    TABLES = {"slot_expert": 0, "expert_slot": 1, "stamp": 2, "clock": 3}

    def debug_write_table(self, layer: int, table: str, index: int, value: int) -> None:
        """Overwrite one word of a layer's slot table (fault injection for the audit)."""
        self._check(self._L.moe_offload_debug_write_table(self.h, layer, self.TABLES[table], index, value))

    def read_misses(self, layer: int):
        cap = self.num_experts
        me = np.empty(cap, np.int32)
        ms = np.empty(cap, np.int32)
        mc, sc = ctypes.c_int(), ctypes.c_int()
        self._check(self._L.moe_offload_read_misses(self.h, layer, me.ctypes.data, ms.ctypes.data, cap,
                                                    ctypes.byref(mc), ctypes.byref(sc)))
        n = mc.value
        return [(int(a), int(b)) for a, b in zip(me[:n], ms[:n])], n, sc.value

    def prefetch(self, layer: int, x, T: int, stream=None) -> None:
        """Router lookahead into `layer` from x, the input of layer - 1 (moe_offload_prefetch)."""
        self._check(self._L.moe_offload_prefetch(self.h, layer, _ptr(x), T, _stream(stream)))

    def read_route_counts(self, layer: int) -> np.ndarray:
        """Routed (token, rank) pairs per expert of `layer` since create or reset."""
        c = np.zeros(self.num_experts, np.uint64)
        self._check(self._L.moe_offload_read_route_counts(self.h, layer, c.ctypes.data))
        return c

    def set_placement(self, layer: int, experts, stream=None) -> None:
        """Freeze `layer` to a static placement: slot i holds experts[i]; others spill."""
        ex = np.ascontiguousarray(experts, dtype=np.int32)
        self._check(self._L.moe_offload_set_placement(self.h, layer, ex.ctypes.data, int(ex.size),
                                                      _stream(stream)))

    def read_prefetch(self, layer: int):
        """(candidates, [(expert, slot), ...]) of the last prefetch install into `layer`."""
        cap = self.num_experts
        cand = np.empty(cap, np.int32)
        ex = np.empty(cap, np.int32)
        sl = np.empty(cap, np.int32)
        nc, ni = ctypes.c_int(), ctypes.c_int()
        self._check(self._L.moe_offload_read_prefetch(self.h, layer, cand.ctypes.data, ctypes.byref(nc),
                                                      ex.ctypes.data, sl.ctypes.data, ctypes.byref(ni), cap))
        return cand[:nc.value].tolist(), list(zip(ex[:ni.value].tolist(), sl[:ni.value].tolist()))

    def read_slot(self, layer: int, slot: int):
        dt = np.uint8 if self.dtype == "fp8" else np.uint16
        w13 = np.empty((2 * self.inter, self.hidden), dt)
        w2 = np.empty((self.hidden, self.inter), dt)
        self._check(self._L.moe_offload_read_slot(self.h, layer, slot, w13.ctypes.data, w2.ctypes.data))
        return w13, w2

    def read_slot_scales(self, layer: int, slot: int):
        s13 = np.empty((2 * self.inter // 128, self.hidden // 128), np.float32)
        s2 = np.empty((self.hidden // 128, self.inter // 128), np.float32)
        self._check(self._L.moe_offload_read_slot_scales(self.h, layer, slot, s13.ctypes.data, s2.ctypes.data))
        return s13, s2

    def set_shared_expert(self, layer: int, w13, w2, s13=None, s2=None) -> None:
        """Device tensors of the layer's shared expert (kept alive by this handle)."""
        self._check(self._L.moe_offload_set_shared_expert(self.h, layer, _ptr(w13), _ptr(s13), _ptr(w2),
                                                          _ptr(s2)))
        self._shared_keep[layer] = (w13, w2, s13, s2)

    def reset(self) -> None:
        self._check(self._L.moe_offload_reset(self.h))

    def device_bytes(self) -> int:
        return int(self._L.moe_offload_device_bytes(self.h))

    def read_routing(self):
        """(ids [T,k], weights [T,k], slot ids [T,k]) of the last decode-path call."""
        cap = self.max_tokens_graph * self.top_k
        ids = np.zeros(cap, np.int32)
        w = np.zeros(cap, np.float32)
        sl = np.zeros(cap, np.int32)
        n = ctypes.c_int()
        self._check(self._L.moe_offload_read_routing(self.h, ids.ctypes.data, w.ctypes.data, sl.ctypes.data, cap,
                                                     ctypes.byref(n)))
        m = n.value
        k = self.top_k
        return ids[:m].reshape(-1, k), w[:m].reshape(-1, k), sl[:m].reshape(-1, k)

    def debug_wait(self, limit_ns: int = 0, stall: bool = False) -> None:
        """Bound of the decode step's early-down waits (0: default) and the debug stall
        that makes the first group's wait of every down warp run out."""
        self._check(self._L.moe_offload_debug_wait(self.h, int(limit_ns), int(bool(stall))))

    def trace_enable(self, on: bool = True) -> None:
        """Decode trace on (records allocated and reset) or off, for launches enqueued
        afterwards; decode graphs keep the setting they were created with."""
        self._check(self._L.moe_offload_trace_enable(self.h, int(bool(on))))

    def trace_read(self, reset: bool = True) -> np.ndarray:
        """The decode trace records, [num_layers, MOE_TRACE_FIELDS] uint64 globaltimer
        stamps (field names in _lib.TRACE_FIELD_NAMES); synchronises the device."""
        out = np.zeros((self.num_layers, C.MOE_TRACE_FIELDS), np.uint64)
        self._check(self._L.moe_offload_trace_read(self.h, out.ctypes.data, int(bool(reset))))
        return out

    def prefill_times(self) -> dict:
        """Phase times (ms) of the last prefill call: route, copy, gemm, combine, staged."""
        v = [ctypes.c_float() for _ in range(4)]
        staged = ctypes.c_int()
        self._check(self._L.moe_offload_prefill_times(self.h, *[ctypes.byref(x) for x in v], ctypes.byref(staged)))
        return dict(route=v[0].value, copy=v[1].value, gemm=v[2].value, combine=v[3].value,
                    staged=bool(staged.value))

    def prefill_gemm_ms(self) -> float:
        """Time (ms) of the last prefill call's two tensor-core GEMM launches alone."""
        v = ctypes.c_float()
        self._check(self._L.moe_offload_prefill_gemm_ms(self.h, ctypes.byref(v)))
        return v.value


class DecodeGraph:
    """A whole-stack decode step captured as one CUDA graph (moe_offload_graph_*).

    x, out: device buffers [L, T, H] bf16 owned by the caller."""

    def __init__(self, moe: MoeOffload, T: int, x, out, timing: bool = False):
        self.moe = moe
        self._L = moe._L
        self.T = T
        self._keep = (x, out)
        g = ctypes.c_void_p()
        moe._check(self._L.moe_offload_graph_create(moe.h, T, _ptr(x), _ptr(out), int(bool(timing)),
                                                    ctypes.byref(g)))
        self.g = g
        self.timing = timing
        self.kernel_count = int(self._L.moe_offload_graph_kernel_count(g))

    def launch(self, stream=None):
        self.moe._check(self._L.moe_offload_graph_launch(self.g, _stream(stream)))

    def launch_host(self, x_host, out_host, stream=None):
        self.moe._check(self._L.moe_offload_graph_launch_host(self.g, _ptr(x_host), _ptr(out_host),
                                                              _stream(stream)))

    def times(self):
        """Per-layer kernel times (ms) of the last launch: head (route + top-k +
        ensure), gate_up (with the copy of installed experts), down + combine."""
        L = self.moe.num_layers
        arrs = [np.zeros(L, np.float32) for _ in range(3)]
        self.moe._check(self._L.moe_offload_graph_times(self.g, *[a.ctypes.data for a in arrs]))
        return arrs

    def close(self):
        if getattr(self, "g", None):
            self._L.moe_offload_graph_destroy(self.g)
            self.g = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
