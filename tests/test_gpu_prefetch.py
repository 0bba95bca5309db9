"""Router-lookahead prefetch (FreeToken issue #677, "Proposal") on the GPU,
through the C ABI, against the oracle's install rule.

Bars: predicted candidates equal the oracle's away from predictor near-ties;
prefetch installs, slot maps and stamps bit-exact against the LRU simulator
fed the GPU's own demand ids and candidates; the fused decode path's tables
equal the separate entry points'; layer outputs bit-identical with the
lookahead on and off (audit on); graph replay equals eager calls; prefetched
slots hold the store's bytes."""
import numpy as np
import pytest

from workload import TINY, TINY_FP8, FP8_LOOKAHEAD, Workload
from stack import Stack, Fp8Stack
from parity import TIE, check_layer

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
    return Stack(TINY, tokens=12, batch=8)


def _bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))


def _u16(t):
    return t.cpu().numpy().view(np.uint16)


def _gap(lg, k):
    s = np.sort(np.asarray(lg, np.float64), axis=1)[:, ::-1]
    return s[:, k - 1] - s[:, k] if lg.shape[1] > k else np.full(lg.shape[0], np.inf)


def _tables(h, L):
    return [tuple(np.asarray(v).tolist() if not isinstance(v, int) else v for v in h.read_table(l))
            for l in range(L)]


@pytest.mark.parametrize("T,N", [(1, 2), (4, 3)])
def test_prefetch_install_matches_simulator(dev, tiny, T, N):
    """route_topk + slot_ensure + miss_copy per layer, then the lookahead into
    the next layer; the simulator replays the GPU's demand ids and candidates."""
    import oracle
    c = tiny.cfg
    L, k, E, S = c.num_layers, c.top_k, c.num_experts, c.num_slots
    sims = [oracle.SlotCacheSim(E, S) for _ in range(L)]
    h = tiny.handle(torch, dev, prefetch_n=N)
    checked = 0
    try:
        for t in range(8):
            for l in range(L):
                x = tiny.x[t, l, :T]
                xd = _bits(x).to(dev)
                ids = torch.empty((T, k), dtype=torch.int32, device=dev)
                w = torch.empty((T, k), dtype=torch.float32, device=dev)
                h.route_topk(l, xd, T, ids, w)
                slot = torch.empty_like(ids)
                h.slot_ensure(l, ids, T, slot)
                h.miss_copy(l)
                torch.cuda.synchronize()
                r = sims[l].ensure(ids.cpu().numpy())
                assert slot.cpu().numpy().tolist() == r.slot_ids.tolist()
                if l + 1 == L:
                    continue
                h.prefetch(l + 1, xd, T)
                cand, inst = h.read_prefetch(l + 1)
                lg = oracle.router_logits(x, tiny.wr[l + 1])
                pid, _ = oracle.topk(lg, k, c.renormalize)
                want = oracle.lookahead_candidates(pid, lg)
                best = sorted((max(float(lg[tt, e]) for tt in range(T) if e in pid[tt]) for e in want),
                              reverse=True)
                order_gap = min((a - b for a, b in zip(best, best[1:])), default=np.inf)
                if np.all(_gap(lg, k) >= TIE) and order_gap >= TIE:
                    # membership and order are both away from rounding-level ties
                    assert cand == want
                    checked += 1
                ri = sims[l + 1].prefetch_install(cand, N)
                assert inst == ri.installs
                for ll in (l, l + 1):
                    se, es, stamp, clock = h.read_table(ll)
                    sse, ses, sst, sclock = sims[ll].snapshot()
                    assert np.array_equal(se, sse) and np.array_equal(es, ses)
                    assert np.array_equal(stamp, sst) and clock == sclock
                for e, s in inst:                     # the copy is joined by the device sync above
                    w13, w2 = h.read_slot(l + 1, s)
                    assert np.array_equal(w13, tiny.w13[l + 1, e]) and np.array_equal(w2, tiny.w2[l + 1, e])
        st = h.get_stats()
        assert st["prefetch_installs"] > 0 and st["prefetch_hits"] <= st["prefetch_installs"]
        assert checked > 0
    finally:
        h.close()


def _decode_all(h, st, dev, T, tokens, audit=False, routing=None):
    c = st.cfg
    xd = _bits(st.x[:tokens, :, :T]).to(dev)
    out = torch.empty((tokens, c.num_layers, T, c.hidden), dtype=torch.int16, device=dev)
    for t in range(tokens):
        if routing is not None:
            routing.append([])
        for l in range(c.num_layers):
            h.decode_layer(l, xd[t, l], T, out[t, l])
            if audit:
                h.audit(l)
            if routing is not None:
                routing[t].append(h.read_routing())
    torch.cuda.synchronize()
    return _u16(out)


def _check_fp8_outputs(st, out, routing, T):
    c = st.cfg
    for t in range(len(routing)):
        for l in range(c.num_layers):
            ids, w, _ = routing[t][l]
            check_layer(out[t, l], st.x[t, l, :T], st.wr[l], st.w13[l], st.w2[l], c.top_k, c.renormalize, ids, w,
                        fp8=(st.s13[l], st.s2[l]), shared=st.shared[l], ctx=(t, l))


@pytest.mark.parametrize("T", [1, 4])
def test_fused_lookahead_equals_separate_entry_points(dev, tiny, T):
    c = tiny.cfg
    L, k = c.num_layers, c.top_k
    N = 2
    ha = tiny.handle(torch, dev, prefetch_n=N)
    hb = tiny.handle(torch, dev, prefetch_n=N)
    try:
        xd = _bits(tiny.x[:6, :, :T]).to(dev)
        oa = torch.empty((T, c.hidden), dtype=torch.int16, device=dev)
        ob = torch.empty_like(oa)
        for t in range(6):
            for l in range(L):
                ha.decode_layer(l, xd[t, l], T, oa)
                ids = torch.empty((T, k), dtype=torch.int32, device=dev)
                w = torch.empty((T, k), dtype=torch.float32, device=dev)
                hb.route_topk(l, xd[t, l], T, ids, w)
                slot = torch.empty_like(ids)
                hb.slot_ensure(l, ids, T, slot)
                if l + 1 < L:
                    hb.prefetch(l + 1, xd[t, l], T)
                hb.miss_copy(l)
                hb.grouped_ffn(l, xd[t, l], slot, w, T, ob)
                torch.cuda.synchronize()
                assert np.array_equal(_u16(oa), _u16(ob)), (t, l)
            assert _tables(ha, L) == _tables(hb, L), t
            for l in range(1, L):
                assert ha.read_prefetch(l) == hb.read_prefetch(l)
        sa, sb = ha.get_stats(), hb.get_stats()
        for key in ("hits", "misses", "prefetch_installs", "prefetch_hits", "prefetch_bytes"):
            assert sa[key] == sb[key], key
    finally:
        ha.close()
        hb.close()


@pytest.mark.parametrize("T", [1, 4, 8])
def test_outputs_bit_identical_with_lookahead_on_and_off(dev, tiny, T):
    ref = None
    for N in (0, 1, 2, tiny.cfg.num_slots):
        h = tiny.handle(torch, dev, prefetch_n=N)
        try:
            out = _decode_all(h, tiny, dev, T, tokens=8, audit=True)
            st = h.get_stats()
        finally:
            h.close()
        assert st["device_status"] == 0
        if N:
            assert st["prefetch_installs"] > 0
        if ref is None:
            ref = out
        else:
            assert np.array_equal(out, ref), N


def test_lookahead_graph_replay_matches_eager(dev, tiny):
    from expert_cache_router_gb300 import DecodeGraph
    c = tiny.cfg
    L = c.num_layers
    for T in (1, 4):
        h = tiny.handle(torch, dev, prefetch_n=2)
        try:
            eager = _decode_all(h, tiny, dev, T, tokens=6)
            tab_eager = _tables(h, L)
            st_eager = h.get_stats()
            h.reset()
            xb = torch.zeros((L, T, c.hidden), dtype=torch.int16, device=dev)
            ob = torch.zeros_like(xb)
            for timing in (False, True):
                h.reset()
                g = DecodeGraph(h, T, xb, ob, timing=timing)
                xs = _bits(tiny.x[:6, :, :T]).to(dev)
                got = []
                for t in range(6):
                    xb.copy_(xs[t])
                    g.launch()
                    got.append(_u16(ob.clone()))
                torch.cuda.synchronize()
                assert np.array_equal(np.stack(got), eager)
                assert _tables(h, L) == tab_eager
                st = h.get_stats()
                assert st["prefetch_installs"] == st_eager["prefetch_installs"]
                g.close()
        finally:
            h.close()


def test_fp8_lookahead_matches_oracle_and_is_bit_identical(dev):
    st = Fp8Stack(TINY_FP8, tokens=6, batch=4)
    outs = {}
    routing = []
    for N in (0, 2):
        h = st.handle(torch, dev, prefetch_n=N)
        try:
            outs[N] = _decode_all(h, st, dev, 4, tokens=6, audit=True, routing=routing if N else None)
            s = h.get_stats()
            assert s["device_status"] == 0
            if N:
                assert s["prefetch_installs"] > 0
        finally:
            h.close()
    assert np.array_equal(outs[0], outs[2])
    _check_fp8_outputs(st, outs[2], routing, 4)


def test_lookahead_two_launch_path_for_wide_routers(dev):
    """E = 512 (above the cluster head's 256): the lookahead runs as the route
    kernels plus the install kernel; fused equals separate, outputs unchanged."""
    cfg = Workload(name="wide_E512_k4_H256_I64_S16", config_id=99, num_layers=3, num_experts=512, top_k=4,
                   hidden=256, inter=64, num_slots=16, batches=(1,), decode_tokens=8, rho=0.9, skew=False)
    st = Stack(cfg, tokens=6, batch=2)
    outs = {}
    tabs = {}
    for N in (0, 4):
        h = st.handle(torch, dev, prefetch_n=N)
        try:
            outs[N] = _decode_all(h, st, dev, 2, tokens=6, audit=True)
            tabs[N] = _tables(h, cfg.num_layers)
            s = h.get_stats()
            assert s["device_status"] == 0
            if N:
                assert s["prefetch_installs"] > 0
                # replay the same steps through the separate entry points
                h2 = st.handle(torch, dev, prefetch_n=N)
                try:
                    xd = _bits(st.x[:6, :, :2]).to(dev)
                    o = torch.empty((2, cfg.hidden), dtype=torch.int16, device=dev)
                    for t in range(6):
                        for l in range(cfg.num_layers):
                            ids = torch.empty((2, cfg.top_k), dtype=torch.int32, device=dev)
                            w = torch.empty((2, cfg.top_k), dtype=torch.float32, device=dev)
                            h2.route_topk(l, xd[t, l], 2, ids, w)
                            slot = torch.empty_like(ids)
                            h2.slot_ensure(l, ids, 2, slot)
                            if l + 1 < cfg.num_layers:
                                h2.prefetch(l + 1, xd[t, l], 2)
                            h2.miss_copy(l)
                            h2.grouped_ffn(l, xd[t, l], slot, w, 2, o)
                    torch.cuda.synchronize()
                    assert _tables(h2, cfg.num_layers) == tabs[N]
                finally:
                    h2.close()
        finally:
            h.close()
    assert np.array_equal(outs[0], outs[4])


@pytest.mark.parametrize("T", [1, 8])
def test_fp8_full_size_lookahead_tables_match_simulator(dev, T):
    """The 256-expert FP8 shape (k=8, H=2048, I=512, 25 slots, shared expert) with
    the lookahead at N=4 on three layers, through the fused cluster head: after
    every decode call the GPU's routed ids replay through the LRU simulator (slot
    ids, miss list, counts, table, stamps, clock bit-exact), its prefetch
    candidates equal the oracle predictor's away from near-ties and replay
    through the simulator's install (installs, both layers' tables bit-exact),
    installed slots hold the store's bytes, and every output row matches the
    oracle on the GPU's routing."""
    import oracle
    st = Fp8Stack(FP8_LOOKAHEAD, num_layers=3, tokens=8, batch=T)
    c = st.cfg
    L, k, E, S, N = c.num_layers, c.top_k, c.num_experts, c.num_slots, c.prefetch_n
    sims = [oracle.SlotCacheSim(E, S) for _ in range(L)]
    h = st.handle(torch, dev, prefetch_n=N)
    xd = _bits(st.x[:8, :, :T]).to(dev)
    out = torch.empty((8, L, T, c.hidden), dtype=torch.int16, device=dev)
    routing = []
    checked = 0
    try:
        for t in range(8):
            routing.append([])
            for l in range(L):
                h.decode_layer(l, xd[t, l], T, out[t, l])
                ids, w, slot = h.read_routing()
                routing[t].append((ids, w, slot))
                r = sims[l].ensure(ids)
                assert np.array_equal(slot, r.slot_ids), (t, l)
                ml, mc, sc = h.read_misses(l)
                assert ml == r.miss_list and mc == r.miss_count and sc == r.spill_count, (t, l)
                if l + 1 < L:
                    cand, inst = h.read_prefetch(l + 1)
                    lg = oracle.router_logits(st.x[t, l, :T], st.wr[l + 1])
                    pid, _ = oracle.topk(lg, k, c.renormalize)
                    want = oracle.lookahead_candidates(pid, lg)
                    best = sorted((max(float(lg[tt, e]) for tt in range(T) if e in pid[tt]) for e in want),
                                  reverse=True)
                    order_gap = min((a - b for a, b in zip(best, best[1:])), default=np.inf)
                    if np.all(_gap(lg, k) >= TIE) and order_gap >= TIE:
                        assert cand == want, (t, l)
                        checked += 1
                    ri = sims[l + 1].prefetch_install(cand, N)
                    assert inst == ri.installs, (t, l)
                    for e, s_ in inst[:2]:
                        w13, w2 = h.read_slot(l + 1, s_)
                        assert np.array_equal(w13, st.w13[l + 1, e]) and np.array_equal(w2, st.w2[l + 1, e])
                for ll in range(l, min(l + 2, L)):
                    se, es, stamp, clock = h.read_table(ll)
                    sse, ses, sst, sclock = sims[ll].snapshot()
                    assert np.array_equal(se, sse) and np.array_equal(es, ses), (t, l, ll)
                    assert np.array_equal(stamp, sst) and clock == sclock, (t, l, ll)
        s = h.get_stats()
        assert s["device_status"] == 0 and s["prefetch_installs"] > 0
    finally:
        h.close()
    assert checked > 0
    _check_fp8_outputs(st, _u16(out), routing, T)


def test_audit_after_every_update_env(dev, tiny, monkeypatch):
    """MOE_OFFLOAD_AUDIT=1: an audit launch follows every table update (eager and in the graph,
    lookahead included); outputs are unchanged and no audit fails."""
    from expert_cache_router_gb300 import DecodeGraph
    c = tiny.cfg
    ref_h = tiny.handle(torch, dev, prefetch_n=2)
    try:
        ref = _decode_all(ref_h, tiny, dev, 4, tokens=6)
    finally:
        ref_h.close()
    monkeypatch.setenv("MOE_OFFLOAD_AUDIT", "1")
    h = tiny.handle(torch, dev, prefetch_n=2)
    try:
        out = _decode_all(h, tiny, dev, 4, tokens=6)
        assert np.array_equal(out, ref)
        h.reset()
        xb = torch.zeros((c.num_layers, 4, c.hidden), dtype=torch.int16, device=dev)
        ob = torch.zeros_like(xb)
        g = DecodeGraph(h, 4, xb, ob)
        assert g.kernel_count == c.num_layers * 4 + (c.num_layers - 1)
        xs = _bits(tiny.x[:6, :, :4]).to(dev)
        got = []
        for t in range(6):
            xb.copy_(xs[t])
            g.launch()
            got.append(_u16(ob.clone()))
        assert np.array_equal(np.stack(got), ref)
        g.close()
        assert h.get_stats()["device_status"] == 0
    finally:
        h.close()
