"""Failure detection through the C ABI, with every fault made on the host: a slot
table corrupted word by word and fed to the audit kernel (the GPU reports it in
the status word, nothing traps), and allocations of create failed on purpose
(create reports out-of-memory and releases what it had taken)."""
import numpy as np
import pytest

from stack import Stack
from workload import TINY

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

AUDIT_FAILED = 1 << 2
MOE_ERR_INVALID, MOE_ERR_OOM, MOE_ERR_DEVICE_STATUS = 1, 3, 5


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def tiny():
    return Stack(TINY, tokens=6, batch=4, stream=7)


def _bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))


def _decode(h, st, dev, tokens, T=2):
    c = st.cfg
    xd = _bits(st.x[:tokens, :, :T]).to(dev)
    out = torch.empty((tokens, c.num_layers, T, c.hidden), dtype=torch.int16, device=dev)
    for t in range(tokens):
        for l in range(c.num_layers):
            h.decode_layer(l, xd[t, l], T, out[t, l])
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16)


def _corruptions(se, es, stamp, clock):
    """(name, table, index, value, breaks an invariant) on a populated table."""
    S, E = len(se), len(es)
    s0 = int(np.flatnonzero(se >= 0)[0])
    e0 = int(se[s0])
    e_out = int(np.flatnonzero(es < 0)[0])
    return [
        ("same slot_expert word", "slot_expert", s0, e0, False),
        ("stamp equal to the clock", "stamp", s0, clock, False),
        ("slot names a non-resident expert", "slot_expert", s0, e_out, True),
        ("slot emptied under its expert", "slot_expert", s0, -1, True),
        ("expert points at another's slot", "expert_slot", e_out, s0, True),
        ("resident expert loses its slot", "expert_slot", e0, -1, True),
        ("stamp newer than the clock", "stamp", s0, clock + 1, True),
        ("clock behind the stamps", "clock", 0, 0, True),
    ]


def test_audit_reports_each_corrupted_table_word(dev, tiny):
    from expert_cache_router_gb300 import MoeOffloadError
    h = tiny.handle(torch, dev)
    try:
        ref = _decode(h, tiny, dev, 3)
        layer = 1
        h.audit(layer)
        assert h.get_stats()["device_status"] == 0
        se, es, stamp, clock = h.read_table(layer)
        assert clock == 3 and (se >= 0).sum() > 0 and (es < 0).sum() > 0
        for name, table, index, value, breaks in _corruptions(se, es, stamp, clock):
            h.reset()
            assert np.array_equal(_decode(h, tiny, dev, 3), ref), name
            h.debug_write_table(layer, table, index, value)
            h.audit(layer)
            h.audit(0)  # an untouched layer passes
            if breaks:
                with pytest.raises(MoeOffloadError) as ei:
                    h.get_stats()
                assert ei.value.status == MOE_ERR_DEVICE_STATUS, name
                assert h.get_stats(check=False)["device_status"] == AUDIT_FAILED, name
            else:
                assert h.get_stats()["device_status"] == 0, name
        # reset brings back the empty table and a clean status word
        h.reset()
        assert h.get_stats()["device_status"] == 0
        assert np.array_equal(_decode(h, tiny, dev, 3), ref)
    finally:
        h.close()


def test_debug_write_table_rejects_out_of_range_words(dev, tiny):
    from expert_cache_router_gb300 import MoeOffloadError
    c = tiny.cfg
    S, E = c.num_slots, c.num_experts
    h = tiny.handle(torch, dev)
    try:
        _decode(h, tiny, dev, 2)
        before = h.read_table(0)
        bad = [("slot_expert", 0, E), ("slot_expert", 0, -2), ("slot_expert", S, 0),
               ("expert_slot", 0, S), ("expert_slot", E, 0), ("stamp", S, 0), ("stamp", 0, -1),
               ("stamp", 0, 1 << 32), ("clock", 1, 0), ("clock", 0, -1)]
        for table, index, value in bad:
            with pytest.raises(MoeOffloadError) as ei:
                h.debug_write_table(0, table, index, value)
            assert ei.value.status == MOE_ERR_INVALID, (table, index, value)
        assert h._L.moe_offload_debug_write_table(h.h, 0, 9, 0, 0) == MOE_ERR_INVALID
        assert h._L.moe_offload_debug_write_table(h.h, c.num_layers, 0, 0, 0) == MOE_ERR_INVALID
        after = h.read_table(0)
        assert all(np.array_equal(a, b) for a, b in zip(before[:3], after[:3])) and before[3] == after[3]
        assert h.get_stats()["device_status"] == 0
    finally:
        h.close()


def test_injected_allocation_failures_release_everything(dev, tiny, monkeypatch):
    """Fail create's n-th allocation for n = 0, 1, ... until create succeeds: every
    failure is MOE_ERR_OOM naming the injection, the device memory comes back, and a
    handle made afterwards computes what one made before did."""
    from expert_cache_router_gb300 import MoeOffload, MoeOffloadError
    c = tiny.cfg
    L = c.num_layers
    router = tiny.router_dev(torch, dev)
    # host arrays not yet pinned, so create registers them: registrations are counted too
    w13 = [np.array(tiny.w13[l]) for l in range(L)]
    w2 = [np.array(tiny.w2[l]) for l in range(L)]

    def make():
        return MoeOffload(num_layers=L, num_experts=c.num_experts, top_k=c.top_k, hidden=c.hidden,
                          inter=c.inter, num_slots=c.num_slots, host_w13=w13, host_w2=w2, router=router,
                          renormalize=c.renormalize, max_tokens_graph=8)

    h = make()
    try:
        ref = _decode(h, tiny, dev, 3)
    finally:
        h.close()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    failures = 0
    for n in range(400):
        monkeypatch.setenv("MOE_OFFLOAD_FAIL_ALLOC", str(n))
        try:
            h = make()
        except MoeOffloadError as e:
            assert e.status == MOE_ERR_OOM, (n, str(e))
            assert "injected failure" in str(e), (n, str(e))
            failures += 1
            continue
        h.close()
        break
    else:
        pytest.fail("create still failing after 400 injected allocations")
    # per layer: two slot arrays and four host registrations at least, then the tables and scratch
    assert failures >= 2 * L + 8
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 >= free0 - (4 << 20), (free0, free1)
    monkeypatch.delenv("MOE_OFFLOAD_FAIL_ALLOC")
    h = make()
    try:
        assert np.array_equal(_decode(h, tiny, dev, 3), ref)
        assert h.get_stats()["device_status"] == 0
    finally:
        h.close()


def test_bounded_early_down_wait_runs_out_and_reset_recovers(dev, tiny):
    """A bounded device wait made to run out, with no fault: the down launch of a
    decode step waits per expert group on counters the gate/up CTAs raise. With
    a 1 ms bound and the debug stall (the first group's target is one CTA more
    than its column has) the wait runs out: the call returns at once rather than
    after the 2 s default, the status word carries MOE_DEV_TIMEOUT and nothing
    else (the audit finds the hand-off counters reset, so the last down CTA still
    cleaned up), and after reset, with the stall removed, the handle decodes the
    oracle's outputs again."""
    import time
    from expert_cache_router_gb300 import MoeOffloadError
    from expert_cache_router_gb300._lib import MOE_DEV_TIMEOUT
    from parity import check_layer
    c = tiny.cfg
    T = 2
    h = tiny.handle(torch, dev)
    try:
        xd = _bits(tiny.x[:3, :, :T]).to(dev)
        out = torch.empty((T, c.hidden), dtype=torch.int16, device=dev)
        h.decode_layer(0, xd[0, 0], T, out)          # warm: kernels loaded
        torch.cuda.synchronize()
        h.reset()
        h.debug_wait(limit_ns=1_000_000, stall=True)
        t0 = time.perf_counter()
        h.decode_layer(0, xd[0, 0], T, out)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        assert elapsed < 0.5, elapsed
        with pytest.raises(MoeOffloadError) as ei:
            h.get_stats()
        assert ei.value.status == MOE_ERR_DEVICE_STATUS
        h.audit(0)
        assert h.get_stats(check=False)["device_status"] == MOE_DEV_TIMEOUT
        h.debug_wait(limit_ns=0, stall=False)
        h.reset()
        assert h.get_stats()["device_status"] == 0
        for t in range(3):
            for l in range(c.num_layers):
                h.decode_layer(l, xd[t, l], T, out)
                ids, w, _ = h.read_routing()
                check_layer(out.cpu().numpy().view(np.uint16), tiny.x[t, l, :T], tiny.wr[l], tiny.w13[l],
                            tiny.w2[l], c.top_k, c.renormalize, ids, w, ctx=(t, l))
        assert h.get_stats()["device_status"] == 0
    finally:
        h.close()


def test_bounded_prefill_tile_wait_runs_out_and_reset_recovers(dev):
    """The same, for the tensor-core prefill GEMMs: the down GEMM's CTAs start under
    the gate/up GEMM and wait per row tile for its gate/up CTAs to count themselves
    done. With a 1 ms bound and the debug stall (a target one CTA above what a tile
    has) every such wait runs out: the call returns at once, the status word carries
    MOE_DEV_TIMEOUT and nothing else (each down CTA still loaded and consumed its
    whole ring, so no copy was left in flight), and after reset, with the stall
    removed, a staged prefill computes the oracle's outputs again, row by row."""
    import time
    from expert_cache_router_gb300 import MoeOffloadError
    from expert_cache_router_gb300._lib import MOE_DEV_TIMEOUT
    from parity import check_layer
    T = 48
    st = Stack(TINY, num_layers=2, tokens=1, batch=T, stream=8)
    c = st.cfg
    h = st.handle(torch, dev, num_slots=4)     # 8 experts over 4 slots: every call stages
    try:
        xd = _bits(st.x[0, :, :T]).to(dev)
        out = torch.empty((T, c.hidden), dtype=torch.int16, device=dev)
        h.decode_layer(0, xd[0], T, out)          # warm: kernels loaded, scratch sized
        torch.cuda.synchronize()
        assert h.prefill_times()["staged"]
        h.reset()
        h.debug_wait(limit_ns=1_000_000, stall=True)
        t0 = time.perf_counter()
        h.decode_layer(0, xd[0], T, out)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        assert elapsed < 0.5, elapsed
        with pytest.raises(MoeOffloadError) as ei:
            h.get_stats()
        assert ei.value.status == MOE_ERR_DEVICE_STATUS
        assert h.get_stats(check=False)["device_status"] == MOE_DEV_TIMEOUT
        h.debug_wait(limit_ns=0, stall=False)
        h.reset()
        assert h.get_stats()["device_status"] == 0
        for l in range(c.num_layers):
            h.decode_layer(l, xd[l], T, out)
            ids = torch.empty((T, c.top_k), dtype=torch.int32, device=dev)
            w = torch.empty((T, c.top_k), dtype=torch.float32, device=dev)
            h.route_topk(l, xd[l], T, ids, w)
            torch.cuda.synchronize()
            assert h.prefill_times()["staged"]
            check_layer(out.cpu().numpy().view(np.uint16), st.x[0, l, :T], st.wr[l], st.w13[l], st.w2[l],
                        c.top_k, c.renormalize, ids.cpu().numpy(), w.cpu().numpy(), ctx=l)
        assert h.get_stats()["device_status"] == 0
    finally:
        h.close()


def test_debug_wait_rejects_bad_arguments(dev, tiny):
    from expert_cache_router_gb300 import MoeOffloadError
    h = tiny.handle(torch, dev)
    try:
        for lim, stall in ((-1, False), (0, 2)):
            with pytest.raises(MoeOffloadError) as ei:
                h._check(h._L.moe_offload_debug_wait(h.h, lim, stall))
            assert ei.value.status == MOE_ERR_INVALID
    finally:
        h.close()
