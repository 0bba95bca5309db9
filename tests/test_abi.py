"""The C ABI library builds, loads and exports every symbol include/moe_offload.h
declares; host-side argument checks work without a GPU (no compute call)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from expert_cache_router_gb300 import build as b
    b.build()
    from expert_cache_router_gb300 import _lib
    return _lib.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe_offload.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"\b(moe_offload_\w+)\s*\(", src)


def test_every_declared_symbol_is_exported(lib):
    from expert_cache_router_gb300 import _lib
    names = _declared()
    assert len(names) >= 15
    assert set(names) == set(_lib.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_slots_for_fraction_host_only(lib):
    f = lib.moe_offload_slots_for_fraction
    assert f(0.2, 128, 8) == 25
    assert f(0.1, 256, 8) == 25
    assert f(0.01, 128, 8) == 8
    assert f(1.0, 8, 2) == 8
    assert f(0.0, 8, 2) == -1
    assert f(1.5, 8, 2) == -1


def test_create_rejects_bad_config_without_gpu(lib):
    from expert_cache_router_gb300 import _lib as C
    bufs = [np.zeros(64, np.uint16) for _ in range(3)]
    arr = ctypes.c_void_p * 1
    p = arr(bufs[0].ctypes.data)
    h = ctypes.c_void_p()
    cfg = C.Config(1, 8, 2, 256, 512, 1, 0, 1, 8, 0, 0)        # S=1 < k=2
    st = lib.moe_offload_create(ctypes.byref(cfg), 0, p, p, None, None, p, ctypes.byref(h))
    assert st == C.MOE_ERR_INVALID and not h.value
    assert b"invalid configuration" in lib.moe_offload_last_error(None)
    cfg = C.Config(1, 8, 2, 250, 512, 4, 0, 1, 8, 0, 0)        # H not a multiple of 256
    assert lib.moe_offload_create(ctypes.byref(cfg), 0, p, p, None, None, p, ctypes.byref(h)) == C.MOE_ERR_INVALID
    cfg = C.Config(1, 8, 2, 256, 512, 4, 7, 1, 8, 0, 0)        # unknown dtype
    assert lib.moe_offload_create(ctypes.byref(cfg), 0, p, p, None, None, p, ctypes.byref(h)) == C.MOE_ERR_INVALID
    cfg = C.Config(1, 8, 2, 256, 512, 4, 0, 1, 8, 0, 0)
    odd = arr(bufs[1].ctypes.data + 2)                          # misaligned host array
    assert lib.moe_offload_create(ctypes.byref(cfg), 0, odd, p, None, None, p, ctypes.byref(h)) == C.MOE_ERR_INVALID
    assert b"16-byte" in lib.moe_offload_last_error(None)


def test_create_checks_fp8_and_shared_expert_arguments_without_gpu(lib):
    from expert_cache_router_gb300 import _lib as C
    buf = np.zeros(64, np.uint32)
    arr = ctypes.c_void_p * 1
    p = arr(buf.ctypes.data)
    fp = (ctypes.POINTER(ctypes.c_float) * 1)(ctypes.cast(buf.ctypes.data, ctypes.POINTER(ctypes.c_float)))
    h = ctypes.c_void_p()
    fp8 = C.MOE_DTYPE_FP8_E4M3_B128

    def create(cfg, s13, s2):
        return lib.moe_offload_create(ctypes.byref(cfg), 0, p, p, s13, s2, p, ctypes.byref(h))

    # FP8 needs both scale tables
    assert create(C.Config(1, 8, 2, 256, 256, 4, fp8, 1, 8, 0, 0), None, None) == C.MOE_ERR_INVALID
    assert b"scale" in lib.moe_offload_last_error(None)
    assert create(C.Config(1, 8, 2, 256, 256, 4, fp8, 1, 8, 0, 0), fp, None) == C.MOE_ERR_INVALID
    # 128 x 128 blocks need I a multiple of 128
    assert create(C.Config(1, 8, 2, 256, 192, 4, fp8, 1, 8, 0, 0), fp, fp) == C.MOE_ERR_INVALID
    assert b"128" in lib.moe_offload_last_error(None)
    # bf16 takes no scale tables
    assert create(C.Config(1, 8, 2, 256, 256, 4, C.MOE_DTYPE_BF16, 1, 8, 0, 0), fp, fp) == C.MOE_ERR_INVALID
    # shared_expert is 0 or 1; pairs including the shared expert's tokens fit 1024
    assert create(C.Config(1, 8, 2, 256, 256, 4, fp8, 1, 8, 2, 0), fp, fp) == C.MOE_ERR_INVALID
    assert create(C.Config(1, 64, 16, 256, 256, 16, fp8, 1, 64, 1, 0), fp, fp) == C.MOE_ERR_INVALID
    assert b"shared_expert" in lib.moe_offload_last_error(None)
    assert not h.value
    assert lib.moe_offload_set_shared_expert(None, 0, None, None, None, None) == C.MOE_ERR_INVALID
    assert lib.moe_offload_read_slot_scales(None, 0, 0, None, None) == C.MOE_ERR_INVALID


def test_null_handle_calls_are_rejected(lib):
    from expert_cache_router_gb300 import _lib as C
    assert lib.moe_offload_route_topk(None, 0, None, 1, None, None, None) == C.MOE_ERR_INVALID
    assert lib.moe_offload_decode_layer(None, 0, None, 1, None, None) == C.MOE_ERR_INVALID
    assert lib.moe_offload_reset(None) == C.MOE_ERR_INVALID
    assert lib.moe_offload_profile_read(None, -1, None, None, None, None, 0) == C.MOE_ERR_INVALID
    assert lib.moe_offload_debug_write_table(None, 0, 0, 0, 0) == C.MOE_ERR_INVALID
    assert lib.moe_offload_audit(None, 0, None) == C.MOE_ERR_INVALID
    assert lib.moe_offload_get_config(None, None, None) == C.MOE_ERR_INVALID
    assert lib.moe_offload_prefill_gemm_ms(None, None) == C.MOE_ERR_INVALID
    assert lib.moe_offload_read_routing(None, None, None, None, 0, None) == C.MOE_ERR_INVALID
    assert lib.moe_offload_debug_wait(None, 0, 0) == C.MOE_ERR_INVALID
    assert lib.moe_offload_trace_enable(None, 1) == C.MOE_ERR_INVALID
    assert lib.moe_offload_trace_read(None, None, 0) == C.MOE_ERR_INVALID
    assert C.MOE_TRACE_FIELDS >= len(C.TRACE_FIELD_NAMES) and set(C.TRACE_MIN_FIELDS) <= set(C.TRACE_FIELD_NAMES)
    lib.moe_offload_destroy(None)


def test_auto_slot_config_is_checked_without_gpu(lib):
    """num_slots = 0 asks for auto sizing; the host checks that need no device still apply."""
    from expert_cache_router_gb300 import _lib as C
    buf = np.zeros(64, np.uint16)
    arr = ctypes.c_void_p * 1
    p = arr(buf.ctypes.data)
    h = ctypes.c_void_p()
    cfg = C.Config(1, 8, 2, 256, 512, 0, 0, 1, 8, 0, 9, 0)    # auto, prefetch_n above E
    assert lib.moe_offload_create(ctypes.byref(cfg), 0, p, p, None, None, p, ctypes.byref(h)) == C.MOE_ERR_INVALID
    assert b"prefetch_n" in lib.moe_offload_last_error(None)
    cfg = C.Config(1, 8, 2, 256, 512, -1, 0, 1, 8, 0, 0, 0)   # negative slot count
    assert lib.moe_offload_create(ctypes.byref(cfg), 0, p, p, None, None, p, ctypes.byref(h)) == C.MOE_ERR_INVALID
    assert not h.value


def test_slots_auto_matches_oracle(lib):
    from oracle import slots_auto
    import random
    rng = random.Random(3)
    for _ in range(2000):
        L = rng.randint(1, 96)
        E = rng.randint(1, 512)
        k = rng.randint(1, min(16, E))
        B = rng.randint(1, 400_000_000)
        reserve = rng.randint(0, 8 * 2 ** 30)
        free = rng.randint(0, 300 * 2 ** 30)
        assert lib.moe_offload_slots_auto(free, reserve, L, E, k, B) == slots_auto(free, reserve, L, E, k, B)


def test_plan_static_matches_oracle_without_gpu(lib):
    from expert_cache_router_gb300 import plan_static
    from oracle import plan_top
    rng = np.random.default_rng(4)
    for _ in range(300):
        E = int(rng.integers(1, 300))
        counts = rng.integers(0, 12, size=E).astype(np.uint64)
        S = int(rng.integers(1, 320))
        assert plan_static(counts, S).tolist() == plan_top(counts, S)
    c = np.zeros(4, np.uint64)
    assert lib.moe_offload_plan_static(c.ctypes.data, 4, 0, c.ctypes.data) == -1


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """No fallback: without the built library the binding raises instead of computing anything."""
    import expert_cache_router_gb300._lib as C
    from expert_cache_router_gb300 import MoeOffload
    monkeypatch.setattr(C, "_lib", None)
    monkeypatch.setattr(C, "LIB_PATH", str(tmp_path / "libmoe_offload.so"))
    with pytest.raises(RuntimeError, match="not found"):
        C.load(str(tmp_path / "libmoe_offload.so"))
    with pytest.raises(RuntimeError, match="not found"):
        MoeOffload(num_layers=1, num_experts=8, top_k=2, hidden=256, inter=256, num_slots=4,
                   host_w13=[0], host_w2=[0], router=[0])
