"""Static expert placement (the "PolyStrata" page, workflow steps 1-3: profile,
plan the most-routed experts into the slots, serve) on the GPU, through the C
ABI, against the oracle's frozen-table rule.

Bars: the device profile (routed pairs per expert) equals the count of the GPU's
own ids; the plan equals the oracle's; slot ids, tables and stamps bit-exact
against the frozen simulator fed the GPU's ids; placed slots hold the store's
bytes; outputs bit-identical to LRU (audit on, graph replay, lookahead on);
prefill of a frozen layer stages."""
import numpy as np
import pytest

from workload import TINY, QWEN3_30B_A3B
from stack import Stack
from parity import check_layer

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def tiny():
    return Stack(TINY, tokens=20, batch=8)


def _bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))


def _u16(t):
    return t.cpu().numpy().view(np.uint16)


def _route_ensure(h, l, xd, T, k, dev):
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    h.route_topk(l, xd, T, ids, w)
    slot = torch.empty_like(ids)
    h.slot_ensure(l, ids, T, slot)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), slot.cpu().numpy()


def _profile_and_place(h, st, dev, T, tokens):
    """Profile `tokens` steps with LRU, then freeze every layer to the top plan."""
    import oracle
    from expert_cache_router_gb300 import plan_static
    c = st.cfg
    want = [np.zeros(c.num_experts, np.uint64) for _ in range(c.num_layers)]
    for t in range(tokens):
        for l in range(c.num_layers):
            ids, _ = _route_ensure(h, l, _bits(st.x[t, l, :T]).to(dev), T, c.top_k, dev)
            want[l] += np.bincount(ids.ravel(), minlength=c.num_experts).astype(np.uint64)
    plans = []
    for l in range(c.num_layers):
        counts = h.read_route_counts(l)
        assert np.array_equal(counts, want[l])
        plan = plan_static(counts, c.num_slots)
        assert plan.tolist() == oracle.plan_top(counts, c.num_slots)
        h.set_placement(l, plan)
        plans.append(plan.tolist())
    return plans


@pytest.mark.parametrize("T", [1, 4])
def test_static_placement_matches_frozen_simulator(dev, tiny, T):
    import oracle
    c = tiny.cfg
    h = tiny.handle(torch, dev)
    try:
        plans = _profile_and_place(h, tiny, dev, T, tokens=6)
        sims = []
        for l in range(c.num_layers):
            s = oracle.SlotCacheSim(c.num_experts, c.num_slots)
            s.freeze(plans[l])
            se, es, stamp, clock = h.read_table(l)
            s.clock = clock
            assert se.tolist() == s.slot_expert and np.all(stamp == 0)
            for slot, e in enumerate(plans[l]):
                w13, w2 = h.read_slot(l, slot)
                assert np.array_equal(w13, tiny.w13[l, e]) and np.array_equal(w2, tiny.w2[l, e])
            sims.append(s)
        spills = 0
        for t in range(6, 14):
            for l in range(c.num_layers):
                ids, slot = _route_ensure(h, l, _bits(tiny.x[t, l, :T]).to(dev), T, c.top_k, dev)
                r = sims[l].ensure(ids)
                assert slot.tolist() == r.slot_ids.tolist()
                se, es, stamp, clock = h.read_table(l)
                sse, ses, sst, sclock = sims[l].snapshot()
                assert np.array_equal(se, sse) and np.array_equal(es, ses)
                assert np.array_equal(stamp, sst) and clock == sclock
                spills += r.spill_count
        st = h.get_stats()
        assert st["device_status"] == 0
        assert spills > 0
    finally:
        h.close()


def _decode_all(h, st, dev, T, t0, tokens, audit=True):
    c = st.cfg
    xd = _bits(st.x[t0:t0 + tokens, :, :T]).to(dev)
    out = torch.empty((tokens, c.num_layers, T, c.hidden), dtype=torch.int16, device=dev)
    for t in range(tokens):
        for l in range(c.num_layers):
            h.decode_layer(l, xd[t, l], T, out[t, l])
            if audit:
                h.audit(l)
    torch.cuda.synchronize()
    return _u16(out)


@pytest.mark.parametrize("T", [1, 8])
def test_placement_outputs_equal_lru_and_graph(dev, tiny, T):
    from expert_cache_router_gb300 import DecodeGraph
    c = tiny.cfg
    ref_h = tiny.handle(torch, dev)
    try:
        ref = _decode_all(ref_h, tiny, dev, T, 6, 8)
    finally:
        ref_h.close()
    for N in (0, 2):
        h = tiny.handle(torch, dev, prefetch_n=N)
        try:
            _profile_and_place(h, tiny, dev, T, tokens=6)
            out = _decode_all(h, tiny, dev, T, 6, 8)
            st = h.get_stats()
            assert np.array_equal(out, ref)
            assert st["device_status"] == 0 and st["prefetch_installs"] == 0
            xb = torch.zeros((c.num_layers, T, c.hidden), dtype=torch.int16, device=dev)
            ob = torch.zeros_like(xb)
            g = DecodeGraph(h, T, xb, ob)
            xs = _bits(tiny.x[6:14, :, :T]).to(dev)
            got = []
            for t in range(8):
                xb.copy_(xs[t])
                g.launch()
                got.append(_u16(ob.clone()))
            assert np.array_equal(np.stack(got), ref)
            g.close()
        finally:
            h.close()


def test_prefill_of_a_frozen_layer_stages(dev, tiny):
    c = tiny.cfg
    h = tiny.handle(torch, dev, max_tokens_graph=4)
    try:
        _profile_and_place(h, tiny, dev, 1, tokens=4)
        before = [h.read_table(l)[0].tolist() for l in range(c.num_layers)]
        T = 8
        x = tiny.x[4, 1, :T]
        out = torch.empty((T, c.hidden), dtype=torch.int16, device=dev)
        h.decode_layer(1, _bits(x).to(dev), T, out)
        torch.cuda.synchronize()
        assert h.prefill_times()["staged"] == 1
        assert [h.read_table(l)[0].tolist() for l in range(c.num_layers)] == before
        ids = torch.empty((T, c.top_k), dtype=torch.int32, device=dev)
        w = torch.empty((T, c.top_k), dtype=torch.float32, device=dev)
        h.route_topk(1, _bits(x).to(dev), T, ids, w)   # the routing kernel of the prefill path
        torch.cuda.synchronize()
        check_layer(_u16(out), x, tiny.wr[1], tiny.w13[1], tiny.w2[1], c.top_k, c.renormalize,
                    ids.cpu().numpy(), w.cpu().numpy())
    finally:
        h.close()


def test_set_placement_rejects_bad_plans(dev, tiny):
    from expert_cache_router_gb300 import MoeOffloadError
    c = tiny.cfg
    h = tiny.handle(torch, dev)
    try:
        for bad in ([0, 0], list(range(c.num_slots + 1)), [c.num_experts], []):
            with pytest.raises(MoeOffloadError):
                h.set_placement(0, bad)
        h.set_placement(0, [3, 1])
        h.reset()                                   # back to an empty LRU table
        se, _, _, _ = h.read_table(0)
        assert np.all(se == -1)
    finally:
        h.close()
