"""Edge cases at the limits of the configuration, through the C ABI: the most
experts (1024), the largest top-k (16) and a 64-token call (T*k = 1024 pairs,
the head's non-cluster path and the FFN's largest grouping), slot counts from
k to E, the widest hidden size (8192), empty calls."""
import numpy as np
import pytest

from workload import Workload
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


def _bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))


def _u16(t):
    return t.cpu().numpy().view(np.uint16)


def _decode(h, st, dev, T, tokens, routing=None):
    """decode_layer + audit over tokens x layers; with routing = [] also reads each
    call's routing (ids, weights, slot ids) into routing[t][l]."""
    c = st.cfg
    xd = _bits(st.x[:tokens, :, :T]).to(dev)
    out = torch.empty((tokens, c.num_layers, T, c.hidden), dtype=torch.int16, device=dev)
    for t in range(tokens):
        if routing is not None:
            routing.append([])
        for l in range(c.num_layers):
            h.decode_layer(l, xd[t, l], T, out[t, l])
            h.audit(l)
            if routing is not None:
                routing[t].append(h.read_routing())
    torch.cuda.synchronize()
    return _u16(out)


def _check_outputs(st, out, routing, T):
    c = st.cfg
    for t in range(len(routing)):
        for l in range(c.num_layers):
            ids, w, _ = routing[t][l]
            check_layer(out[t, l], st.x[t, l, :T], st.wr[l], st.w13[l], st.w2[l], c.top_k, c.renormalize, ids, w,
                        ctx=(t, l))


WIDE = Workload(name="edge_E1024_k16_H256_I64", config_id=97, num_layers=2, num_experts=1024, top_k=16,
                hidden=256, inter=64, num_slots=1024, batches=(64,), decode_tokens=2, rho=0.9, skew=False)


@pytest.fixture(scope="module")
def wide():
    return Stack(WIDE, tokens=2, batch=64)


def test_1024_experts_top16_64_tokens_against_oracle(dev, wide):
    h = wide.handle(torch, dev, max_tokens_graph=64)
    routing = []
    try:
        out = _decode(h, wide, dev, 64, 2, routing=routing)
        assert h.get_stats()["device_status"] == 0
    finally:
        h.close()
    _check_outputs(wide, out, routing, 64)


def test_1024_experts_bit_identical_from_k_slots_to_e_slots(dev, wide):
    outs = []
    for S in (16, 100, 1024):
        h = wide.handle(torch, dev, num_slots=S, max_tokens_graph=64)
        try:
            outs.append(_decode(h, wide, dev, 64, 2))
            st = h.get_stats()
            assert st["device_status"] == 0
            if S == 16:
                assert st["spills"] > 0
        finally:
            h.close()
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_1024_pair_graph_matches_eager(dev, wide):
    from expert_cache_router_gb300 import DecodeGraph
    c = wide.cfg
    h = wide.handle(torch, dev, num_slots=64, max_tokens_graph=64)
    try:
        eager = _decode(h, wide, dev, 64, 2)
        h.reset()
        xb = torch.zeros((c.num_layers, 64, c.hidden), dtype=torch.int16, device=dev)
        ob = torch.zeros_like(xb)
        g = DecodeGraph(h, 64, xb, ob)
        xs = _bits(wide.x[:2, :, :64]).to(dev)
        got = []
        for t in range(2):
            xb.copy_(xs[t])
            g.launch()
            got.append(_u16(ob.clone()))
        assert np.array_equal(np.stack(got), eager)
        g.close()
    finally:
        h.close()


def test_widest_hidden_size(dev):
    cfg = Workload(name="edge_E8_k2_H8192_I64_S2", config_id=96, num_layers=2, num_experts=8, top_k=2,
                   hidden=8192, inter=64, num_slots=2, batches=(1,), decode_tokens=4, rho=0.9, skew=False)
    st = Stack(cfg, tokens=3, batch=8)
    for T in (1, 8):
        h = st.handle(torch, dev)
        routing = []
        try:
            out = _decode(h, st, dev, T, 3, routing=routing)
            assert h.get_stats()["device_status"] == 0
        finally:
            h.close()
        _check_outputs(st, out, routing, T)


def test_empty_calls_do_nothing(dev):
    from workload import TINY
    st = Stack(TINY, tokens=1, batch=1)
    h = st.handle(torch, dev)
    try:
        x = _bits(st.x[0, 0, :1]).to(dev)
        ids = torch.full((1, TINY.top_k), -7, dtype=torch.int32, device=dev)
        w = torch.zeros((1, TINY.top_k), dtype=torch.float32, device=dev)
        out = torch.full((1, TINY.hidden), 5, dtype=torch.int16, device=dev)
        h.route_topk(0, x, 0, ids, w)
        h.slot_ensure(0, ids, 0, ids)
        h.grouped_ffn(0, x, ids, w, 0, out)
        h.decode_layer(0, x, 0, out)
        torch.cuda.synchronize()
        assert np.all(ids.cpu().numpy() == -7) and np.all(out.cpu().numpy() == 5)
        s = h.get_stats()
        assert s["calls"] == 0 and s["device_status"] == 0
        se, _, _, clock = h.read_table(0)
        assert np.all(se == -1) and clock == 0
    finally:
        h.close()


@pytest.mark.parametrize("k,T", [(12, 4), (16, 2), (8, 16)])
def test_cluster_head_topk_equals_route_topk(dev, k, T):
    """The fused cluster head's top-k (an 8-entry bitonic list per warp for k <= 8,
    k rounds of a warp maximum above) gives the same ids and weights, bit for bit,
    as the standalone route_topk kernel, and its slot table matches the simulator
    replaying those ids; outputs match the oracle on every row."""
    from oracle import SlotCacheSim
    cfg = Workload(name=f"edge_E64_k{k}_H256_I64", config_id=95, num_layers=2, num_experts=64, top_k=k,
                   hidden=256, inter=64, num_slots=max(k, 20), batches=(T,), decode_tokens=3, rho=0.9, skew=False)
    st = Stack(cfg, tokens=3, batch=T)
    h = st.handle(torch, dev, max_tokens_graph=T)
    sims = [SlotCacheSim(cfg.num_experts, cfg.num_slots) for _ in range(cfg.num_layers)]
    try:
        xd = _bits(st.x[:3, :, :T]).to(dev)
        out = torch.empty((T, cfg.hidden), dtype=torch.int16, device=dev)
        ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        w = torch.empty((T, k), dtype=torch.float32, device=dev)
        for t in range(3):
            for l in range(cfg.num_layers):
                h.decode_layer(l, xd[t, l], T, out)
                gids, gw, gslot = h.read_routing()
                h.route_topk(l, xd[t, l], T, ids, w)
                torch.cuda.synchronize()
                assert np.array_equal(gids, ids.cpu().numpy()), (t, l)
                assert np.array_equal(gw.view(np.uint32), w.cpu().numpy().view(np.uint32)), (t, l)
                assert np.array_equal(gslot, sims[l].ensure(gids).slot_ids), (t, l)
                check_layer(_u16(out), st.x[t, l, :T], st.wr[l], st.w13[l], st.w2[l], k, cfg.renormalize, gids, gw,
                            ctx=(t, l))
        assert h.get_stats()["device_status"] == 0
    finally:
        h.close()
