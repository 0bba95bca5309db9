"""CUDA path vs the CPU oracle, through the C ABI.

Bars: routing ids exact except where the oracle's k-th and (k+1)-th logits are
within 1e-3; slot maps, miss lists, counts and slot bytes bit-exact against the
LRU simulator fed the GPU's own id trace; every row of every layer output within
relative L2 5e-3 of the oracle's fp32 output, the oracle FFN evaluated on the
GPU's own routing (so near-tie rows are checked too); outputs bit-identical
across slot counts, spills, graph replay and audit on/off."""
import numpy as np
import pytest

from workload import TINY, QWEN3_30B_A3B, MIXTRAL_8X7B, gen
from stack import Stack
from parity import TIE, TOL, assert_rows, check_layer, check_routing

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
    return Stack(TINY, tokens=16, batch=8)


def _bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))


def _u16(t):
    return t.cpu().numpy().view(np.uint16)


def _check_route(x, wr, k, ids, w, renorm=True):
    import oracle
    return check_routing(oracle.router_logits(x, wr), k, renorm, ids, w)


def _gpu_route(h, layer, x, dev):
    """The GPU's routing of x [T, H] through route_topk (the kernel the prefill path runs)."""
    T = x.shape[0]
    ids = torch.empty((T, h.top_k), dtype=torch.int32, device=dev)
    w = torch.empty((T, h.top_k), dtype=torch.float32, device=dev)
    h.route_topk(layer, _bits(x).to(dev), T, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


# ------------------------------------------------------------------ routing
@pytest.mark.parametrize("T", [1, 3, 8])
def test_route_topk_decode(dev, tiny, T):
    c = tiny.cfg
    h = tiny.handle(torch, dev)
    try:
        for l in range(c.num_layers):
            x = tiny.x[0, l, :T]
            ids = torch.empty((T, c.top_k), dtype=torch.int32, device=dev)
            w = torch.empty((T, c.top_k), dtype=torch.float32, device=dev)
            h.route_topk(l, _bits(x).to(dev), T, ids, w)
            torch.cuda.synchronize()
            _check_route(x, tiny.wr[l], c.top_k, ids.cpu().numpy(), w.cpu().numpy())
    finally:
        h.close()


def test_route_topk_prefill_sized(dev):
    """T=2048 (separate top-k launch) on the Qwen3-30B-A3B router shape."""
    from dataclasses import replace
    import oracle
    cfg = replace(QWEN3_30B_A3B, num_layers=1)
    wr = gen.router_weights(cfg)
    mu = gen.input_means(cfg, wr)
    x = gen.router_inputs(cfg, mu, 2048, 1)[:, 0, 0, :]
    from expert_cache_router_gb300 import MoeOffload
    w13 = np.zeros((cfg.num_experts, 2 * cfg.inter, cfg.hidden), np.uint16)
    w2 = np.zeros((cfg.num_experts, cfg.hidden, cfg.inter), np.uint16)
    h = MoeOffload(num_layers=1, num_experts=cfg.num_experts, top_k=cfg.top_k, hidden=cfg.hidden,
                   inter=cfg.inter, num_slots=cfg.num_slots, host_w13=[w13], host_w2=[w2],
                   router=[_bits(wr[0]).to(dev)])
    try:
        T = x.shape[0]
        ids = torch.empty((T, cfg.top_k), dtype=torch.int32, device=dev)
        w = torch.empty((T, cfg.top_k), dtype=torch.float32, device=dev)
        h.route_topk(0, _bits(x).to(dev), T, ids, w)
        torch.cuda.synchronize()
        sample = np.arange(0, T, 7)
        same = _check_route(x[sample], wr[0], cfg.top_k, ids.cpu().numpy()[sample], w.cpu().numpy()[sample])
        assert same.mean() > 0.95
    finally:
        h.close()


# -------------------------------------------------------------- slot table
def _run_trace(h, dev, sim, calls, layer=0, check_slots_of=None):
    for ids in calls:
        T = ids.shape[0]
        ids_d = torch.from_numpy(ids.astype(np.int32)).to(dev)
        slot_d = torch.empty_like(ids_d)
        h.slot_ensure(layer, ids_d, T, slot_d)
        h.miss_copy(layer)
        r = sim.ensure(ids)
        got_slots = slot_d.cpu().numpy()
        assert np.array_equal(got_slots, r.slot_ids)
        ml, mc, sc = h.read_misses(layer)
        assert ml == r.miss_list and mc == r.miss_count and sc == r.spill_count
        se, es, st, clock = h.read_table(layer)
        sse, ses, sst, sclock = sim.snapshot()
        assert np.array_equal(se, sse) and np.array_equal(es, ses)
        assert np.array_equal(st, sst) and clock == sclock
        if check_slots_of is not None:
            w13, w2 = check_slots_of
            for e, s in r.miss_list:
                if s < h.num_slots:
                    g13, g2 = h.read_slot(layer, s)
                    assert np.array_equal(g13, w13[e]) and np.array_equal(g2, w2[e])


@pytest.mark.parametrize("S", [2, 4, 8])
def test_slot_ensure_random_traces_tiny(dev, tiny, S):
    from oracle import SlotCacheSim
    c = tiny.cfg
    rng = np.random.default_rng(100 + S)
    calls = []
    for _ in range(40):
        T = int(rng.integers(1, 9))
        calls.append(np.stack([rng.choice(c.num_experts, size=c.top_k, replace=False) for _ in range(T)]))
    h = tiny.handle(torch, dev, num_slots=S)
    try:
        _run_trace(h, dev, SlotCacheSim(c.num_experts, S), calls, layer=1,
                   check_slots_of=(tiny.w13[1], tiny.w2[1]))
        h.audit(1)
        assert h.get_stats()["device_status"] == 0
    finally:
        h.close()


def test_slot_ensure_hand_traces(dev, tiny):
    """The hand-worked golden traces, replayed on the GPU table."""
    from lru_golden import load_traces
    from expert_cache_router_gb300 import MoeOffload
    c = tiny.cfg
    for tr in load_traces():
        if any(cl["kind"] != "call" for cl in tr["calls"]):
            continue
        E, S = tr["E"], tr["S"]
        w13 = np.zeros((E, 2 * c.inter, c.hidden), np.uint16)
        w2 = np.zeros((E, c.hidden, c.inter), np.uint16)
        wr = torch.zeros((E, c.hidden), dtype=torch.int16, device=dev)
        h = MoeOffload(num_layers=1, num_experts=E, top_k=len(tr["calls"][0]["ids"][0]), hidden=c.hidden,
                       inter=c.inter, num_slots=S, host_w13=[w13], host_w2=[w2], router=[wr])
        try:
            for cl in tr["calls"]:
                ids = torch.tensor(cl["ids"], dtype=torch.int32, device=dev)
                slot = torch.empty_like(ids)
                h.slot_ensure(0, ids, ids.shape[0], slot)
                assert slot.cpu().numpy().tolist() == cl["slot_ids"]
                ml, mc, sc = h.read_misses(0)
                assert ml == cl["miss"] and mc == cl["miss_count"] and sc == cl["spill"]
            se, es, st, clock = h.read_table(0)
            assert se.tolist() == tr["final"]["slot_expert"]
            assert st.tolist() == tr["final"]["stamp"] and clock == tr["final"]["clock"]
        finally:
            h.close()


@pytest.mark.parametrize("S", [25, 40, 64, 65])
def test_slot_ensure_qwen_shape_with_spills(dev, S):
    """E=128, k=8 at 1 to 8 tokens (up to 64 distinct experts: spills at S=25).
    Calls of up to 32 pairs on up to 64 slots take the one-warp update, the others
    the block update; S = 40 and 64 put free slots in both halves of the warp's
    key registers, S = 65 is the first size past it."""
    from oracle import SlotCacheSim
    from expert_cache_router_gb300 import MoeOffload
    E, k, H, I = 128, 8, 256, 64
    w13 = np.zeros((E, 2 * I, H), np.uint16)
    w2 = np.zeros((E, H, I), np.uint16)
    wr = torch.zeros((E, H), dtype=torch.int16, device=dev)
    h = MoeOffload(num_layers=1, num_experts=E, top_k=k, hidden=H, inter=I, num_slots=S,
                   host_w13=[w13], host_w2=[w2], router=[wr])
    rng = np.random.default_rng(7)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    calls = [np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(int(rng.integers(1, 9)))])
             for _ in range(60)]
    try:
        _run_trace(h, dev, SlotCacheSim(E, S), calls)
        st = h.get_stats()
        assert st["device_status"] == 0
        if S == 25:
            assert st["spills"] > 0
    finally:
        h.close()


def test_bad_expert_id_sets_device_status(dev, tiny):
    from expert_cache_router_gb300 import MoeOffloadError
    c = tiny.cfg
    h = tiny.handle(torch, dev)
    try:
        ids = torch.tensor([[0, c.num_experts]], dtype=torch.int32, device=dev)
        slot = torch.empty_like(ids)
        h.slot_ensure(0, ids, 1, slot)
        assert slot.cpu().numpy()[0, 1] == -1
        with pytest.raises(MoeOffloadError) as ei:
            h.get_stats()
        assert ei.value.status == 5
        assert h.get_stats(check=False)["device_status"] & 1
        h.reset()
        assert h.get_stats()["device_status"] == 0
    finally:
        h.close()


# -------------------------------------------------------------------- FFN
def _decode_all(h, stack, dev, T, tokens, audit=False, routing=None):
    """decode_layer over tokens x layers; returns outputs [n, L, T, H] (bf16 bits).
    With routing = [] each call is followed by a read of its routing (ids, weights,
    slot ids), appended as routing[t][l]."""
    c = stack.cfg
    xd = _bits(stack.x[:tokens, :, :T]).to(dev)
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


def _check_outputs(stack, out, routing, T, ctx=""):
    """Every row of every (token, layer) output against the oracle on the GPU's routing."""
    c = stack.cfg
    worst = 0.0
    for t in range(len(routing)):
        for l in range(c.num_layers):
            ids, w, _ = routing[t][l]
            worst = max(worst, check_layer(out[t, l], stack.x[t, l, :T], stack.wr[l], stack.w13[l], stack.w2[l],
                                           c.top_k, c.renormalize, ids, w, ctx=(ctx, t, l)))
    return worst


@pytest.mark.parametrize("T", [1, 4, 8])
def test_decode_layer_matches_oracle_tiny(dev, tiny, T):
    h = tiny.handle(torch, dev)
    routing = []
    try:
        out = _decode_all(h, tiny, dev, T, tokens=6, routing=routing)
    finally:
        h.close()
    _check_outputs(tiny, out, routing, T)


def test_grouped_ffn_on_given_ids(dev, tiny):
    """grouped_ffn alone, on ids and weights the test chooses (shared experts across tokens)."""
    import oracle
    c = tiny.cfg
    T = 8
    ids = np.array([[0, 1], [1, 0], [2, 3], [3, 7], [7, 0], [5, 6], [6, 5], [4, 1]], np.int32)
    w = np.random.default_rng(3).random((T, c.top_k)).astype(np.float32)
    h = tiny.handle(torch, dev, num_slots=8)
    try:
        ids_d = torch.from_numpy(ids).to(dev)
        slot = torch.empty_like(ids_d)
        h.slot_ensure(2, ids_d, T, slot)
        h.miss_copy(2)
        out = torch.empty((T, c.hidden), dtype=torch.int16, device=dev)
        x = tiny.x[0, 2, :T]
        h.grouped_ffn(2, _bits(x).to(dev), slot, torch.from_numpy(w).to(dev), T, out)
        torch.cuda.synchronize()
        ref_f, _ = oracle.moe_ffn(x, ids, w, tiny.w13[2], tiny.w2[2])
        assert_rows(oracle.bf16_to_f32(_u16(out)), ref_f)
    finally:
        h.close()


def test_outputs_bit_identical_across_slot_counts(dev, tiny):
    """Placement never changes the result: every S in [k, E], batch 1 and batch 8 (spills)."""
    c = tiny.cfg
    ref = {}
    for S in range(c.top_k, c.num_experts + 1):
        h = tiny.handle(torch, dev, num_slots=S)
        try:
            for T in (1, 8):
                out = _decode_all(h, tiny, dev, T, tokens=8)
                if T not in ref:
                    ref[T] = out
                else:
                    assert np.array_equal(out, ref[T]), f"S={S} T={T} differs"
            st = h.get_stats()
            assert st["device_status"] == 0
            if S == c.top_k:
                assert st["spills"] > 0
        finally:
            h.close()
    # batch rows are independent: row 0 of the batch-8 run equals the batch-1 run
    assert np.array_equal(ref[8][:, :, 0], ref[1][:, :, 0])


def test_audit_on_does_not_change_outputs(dev, tiny):
    h = tiny.handle(torch, dev)
    try:
        a = _decode_all(h, tiny, dev, 4, tokens=6, audit=True)
        assert h.get_stats()["device_status"] == 0
        h.reset()
        b = _decode_all(h, tiny, dev, 4, tokens=6)
        assert np.array_equal(a, b)
    finally:
        h.close()


def test_eager_profile_counts_every_call_and_changes_nothing(dev, tiny, monkeypatch):
    """MOE_OFFLOAD_PROFILE=1: events around the head, gate/up and down of every eager decode
    call; the profile counts each call once per layer, graph replays are not profiled, and
    outputs equal those of an unprofiled handle."""
    from expert_cache_router_gb300 import DecodeGraph
    c = tiny.cfg
    T, tokens = 2, 5
    h = tiny.handle(torch, dev)
    try:
        ref = _decode_all(h, tiny, dev, T, tokens=tokens)
        assert h.profile_read()["calls"] == 0
    finally:
        h.close()
    monkeypatch.setenv("MOE_OFFLOAD_PROFILE", "1")
    h = tiny.handle(torch, dev)
    try:
        out = _decode_all(h, tiny, dev, T, tokens=tokens)
        assert np.array_equal(out, ref)
        for l in range(c.num_layers):
            p = h.profile_read(l)
            assert p["calls"] == tokens, (l, p)
            assert p["head_ms"] > 0 and p["gate_up_ms"] > 0 and p["down_ms"] > 0, (l, p)
        tot = h.profile_read(-1, clear=True)
        assert tot["calls"] == tokens * c.num_layers
        assert h.profile_read()["calls"] == 0
        h.reset()
        xb = torch.zeros((c.num_layers, T, c.hidden), dtype=torch.int16, device=dev)
        ob = torch.zeros_like(xb)
        g = DecodeGraph(h, T, xb, ob)
        for t in range(2):
            xb.copy_(_bits(tiny.x[t, :, :T]).to(dev))
            g.launch()
        torch.cuda.synchronize()
        g.close()
        assert h.profile_read()["calls"] == 0
        assert h.get_stats()["device_status"] == 0
    finally:
        h.close()


def test_cuda_graph_replay_matches_eager(dev, tiny):
    c = tiny.cfg
    T = 2
    h = tiny.handle(torch, dev)
    try:
        eager = _decode_all(h, tiny, dev, T, tokens=8)
        h.reset()
        xbuf = torch.zeros((c.num_layers, T, c.hidden), dtype=torch.int16, device=dev)
        obuf = torch.zeros((c.num_layers, T, c.hidden), dtype=torch.int16, device=dev)
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for l in range(c.num_layers):
                    h.decode_layer(l, xbuf[l], T, obuf[l], stream=s)
        torch.cuda.synchronize()
        h.reset()  # capture enqueued nothing; start from an empty table
        xs = _bits(tiny.x[:8, :, :T]).to(dev)
        outs = []
        for t in range(8):
            xbuf.copy_(xs[t])
            g.replay()
            outs.append(obuf.clone())
        torch.cuda.synchronize()
        got = np.stack([_u16(o) for o in outs])
        assert np.array_equal(got, eager)
    finally:
        h.close()


def test_prefill_path_under_capture_is_rejected(dev, tiny):
    from expert_cache_router_gb300 import MoeOffloadError
    c = tiny.cfg
    h = tiny.handle(torch, dev)
    try:
        x = torch.zeros((32, c.hidden), dtype=torch.int16, device=dev)
        out = torch.empty_like(x)
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        caught = None
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                try:
                    h.decode_layer(0, x, 32, out, stream=s)
                except MoeOffloadError as e:
                    caught = e
                out.zero_()
        assert caught is not None and caught.status == 4
    finally:
        h.close()


# ---------------------------------------------------------------- prefill
@pytest.mark.parametrize("audit_each", [False, True])
def test_prefill_staged_and_slot_paths(dev, audit_each, monkeypatch):
    import oracle
    if audit_each:
        monkeypatch.setenv("MOE_OFFLOAD_AUDIT", "1")
    from oracle import SlotCacheSim
    st_ = Stack(TINY, num_layers=2, tokens=1, batch=48, stream=3)
    c = st_.cfg
    T = 48
    for S, expect_staged in ((4, True), (8, False)):
        h = st_.handle(torch, dev, num_slots=S)
        try:
            before = h.read_table(0)
            x = st_.x[0, 0, :T]
            out = torch.empty((T, c.hidden), dtype=torch.int16, device=dev)
            h.decode_layer(0, _bits(x).to(dev), T, out)
            torch.cuda.synchronize()
            stats = h.get_stats()
            gids, gw = _gpu_route(h, 0, x, dev)
            check_layer(_u16(out), x, st_.wr[0], st_.w13[0], st_.w2[0], c.top_k, True, gids, gw)
            r = oracle.moe_layer(x, st_.wr[0], st_.w13[0], st_.w2[0], c.top_k)
            assert stats["device_status"] == 0
            after = h.read_table(0)
            if expect_staged:
                assert stats["staged_calls"] == 1 and stats["calls"] == 0
                assert all(np.array_equal(a, b) for a, b in zip(before[:3], after[:3]))
            else:
                assert stats["staged_calls"] == 0 and stats["calls"] == 1
                sim = SlotCacheSim(c.num_experts, S)
                sim.ensure(gids)
                assert np.array_equal(after[0], sim.snapshot()[0])
                assert r["ids"].shape == gids.shape
        finally:
            h.close()


# -------------------------------------------------- full-size layer shapes
@pytest.fixture(scope="module")
def qwen2():
    """Two layers at the full Qwen3-30B-A3B layer size (E=128, k=8, H=2048, I=768)."""
    return Stack(QWEN3_30B_A3B, num_layers=2, tokens=10, batch=8)


@pytest.mark.parametrize("T,tokens", [(1, 10), (8, 8)])
def test_qwen3_30b_a3b_decode_full_size(dev, qwen2, T, tokens):
    """The decode path the benchmark times (fused cluster head: router logits into
    CTA 0's shared memory, block-rank or warp top-k, slot update; gate/up with the
    copy folded in; down + combine), at the full Qwen3-30B-A3B layer size and
    S=25: after every call the GPU's own routed ids are replayed through the LRU
    simulator and the slot ids, miss list, counts, table, stamps and clock must
    match bit for bit; every output row is checked against the oracle on the
    GPU's routing. T=8 touches up to 64 distinct experts per call: spills."""
    from oracle import SlotCacheSim
    c = qwen2.cfg
    h = qwen2.handle(torch, dev)
    sims = [SlotCacheSim(c.num_experts, c.num_slots) for _ in range(c.num_layers)]
    xd = _bits(qwen2.x[:tokens, :, :T]).to(dev)
    out = torch.empty((tokens, c.num_layers, T, c.hidden), dtype=torch.int16, device=dev)
    routing = []
    try:
        for t in range(tokens):
            routing.append([])
            for l in range(c.num_layers):
                h.decode_layer(l, xd[t, l], T, out[t, l])
                ids, w, slot = h.read_routing()
                routing[t].append((ids, w, slot))
                r = sims[l].ensure(ids)
                assert np.array_equal(slot, r.slot_ids), (t, l)
                ml, mc, sc = h.read_misses(l)
                assert ml == r.miss_list and mc == r.miss_count and sc == r.spill_count, (t, l)
                se, es, st, clock = h.read_table(l)
                sse, ses, sst, sclock = sims[l].snapshot()
                assert np.array_equal(se, sse) and np.array_equal(es, ses), (t, l)
                assert np.array_equal(st, sst) and clock == sclock, (t, l)
        stats = h.get_stats()
        h.audit(0)
        h.audit(1)
        assert h.get_stats()["device_status"] == 0
    finally:
        h.close()
    assert stats["device_status"] == 0
    if T == 8:
        assert stats["spills"] > 0
    _check_outputs(qwen2, _u16(out), routing, T, ctx="qwen")


@pytest.mark.parametrize("T", [1, 8])
def test_outputs_bit_identical_across_slot_counts_full_size(dev, qwen2, T):
    """Placement never changes the result, at the Qwen3-30B-A3B layer size:
    S in {8, 25, 64, 128}; T=8 at S=8 spills."""
    ref = None
    for S in (8, 25, 64, 128):
        h = qwen2.handle(torch, dev, num_slots=S)
        try:
            out = _decode_all(h, qwen2, dev, T, tokens=6)
            st = h.get_stats()
        finally:
            h.close()
        assert st["device_status"] == 0
        if T == 8 and S == 8:
            assert st["spills"] > 0
        if S == 128:
            assert st["spills"] == 0
        if ref is None:
            ref = out
        else:
            assert np.array_equal(out, ref), f"S={S} T={T} differs"


@pytest.mark.parametrize("S", [2, 4])
def test_mixtral_8x7b_layer_full_size(dev, S):
    """One layer at the full Mixtral-8x7B layer size (E=8, k=2, H=4096, I=14336)."""
    st_ = Stack(MIXTRAL_8X7B, num_layers=1, tokens=3, batch=1)
    h = st_.handle(torch, dev, num_slots=S)
    routing = []
    try:
        out = _decode_all(h, st_, dev, 1, tokens=3, routing=routing)
        stats = h.get_stats()
    finally:
        h.close()
    assert stats["device_status"] == 0 and stats["misses"] >= 2
    _check_outputs(st_, out, routing, 1, ctx=("mixtral", S))


def test_library_decode_graph_matches_eager_and_times(dev, tiny):
    """moe_offload_graph_*: the whole-stack step graph, replayed per token,
    equals eager decode_layer; timing events give positive per-layer kernel
    times; the host-buffer launch gives the same bytes."""
    from expert_cache_router_gb300 import DecodeGraph
    c = tiny.cfg
    for T in (1, 8):
        h = tiny.handle(torch, dev)
        try:
            eager = _decode_all(h, tiny, dev, T, tokens=6)
            h.reset()
            xb = torch.zeros((c.num_layers, T, c.hidden), dtype=torch.int16, device=dev)
            ob = torch.zeros_like(xb)
            g = DecodeGraph(h, T, xb, ob, timing=True)
            xs = _bits(tiny.x[:6, :, :T]).to(dev)
            got = []
            for t in range(6):
                xb.copy_(xs[t])
                g.launch()
                hd, gu, dn = g.times()
                assert np.all(hd > 0) and np.all(gu > 0) and np.all(dn > 0)
                got.append(_u16(ob.clone()))
            assert np.array_equal(np.stack(got), eager)
            assert g.kernel_count == c.num_layers * 3
            h.reset()
            xh = _bits(tiny.x[:6, :, :T]).pin_memory()
            oh = torch.empty((6, c.num_layers, T, c.hidden), dtype=torch.int16).pin_memory()
            for t in range(6):
                g.launch_host(xh[t], oh[t])
            assert np.array_equal(oh.numpy().view(np.uint16), eager)
            g.close()
        finally:
            h.close()


@pytest.mark.parametrize("T", [1, 8])
def test_fused_decode_path_equals_separate_entry_points(dev, tiny, T):
    """decode_layer (router+ensure in one launch, miss copy folded into the
    gate/up launch) leaves the same tables, slot bytes and outputs as the four
    separate entry points route_topk -> slot_ensure -> miss_copy -> grouped_ffn."""
    c = tiny.cfg
    ha = tiny.handle(torch, dev, num_slots=3)
    hb = tiny.handle(torch, dev, num_slots=3)
    try:
        xs = _bits(tiny.x[:6, :, :T]).to(dev)
        ids = torch.empty((T, c.top_k), dtype=torch.int32, device=dev)
        w = torch.empty((T, c.top_k), dtype=torch.float32, device=dev)
        slot = torch.empty_like(ids)
        oa = torch.empty((T, c.hidden), dtype=torch.int16, device=dev)
        ob = torch.empty_like(oa)
        for t in range(6):
            for l in range(c.num_layers):
                ha.decode_layer(l, xs[t, l], T, oa)
                hb.route_topk(l, xs[t, l], T, ids, w)
                hb.slot_ensure(l, ids, T, slot)
                hb.miss_copy(l)
                hb.grouped_ffn(l, xs[t, l], slot, w, T, ob)
                torch.cuda.synchronize()
                assert torch.equal(oa, ob)
                ta, tb = ha.read_table(l), hb.read_table(l)
                assert all(np.array_equal(p, q) for p, q in zip(ta[:3], tb[:3])) and ta[3] == tb[3]
                assert ha.read_misses(l) == hb.read_misses(l)
        for l in range(c.num_layers):
            for s in range(3):
                a13, a2 = ha.read_slot(l, s)
                b13, b2 = hb.read_slot(l, s)
                assert np.array_equal(a13, b13) and np.array_equal(a2, b2)
        assert ha.get_stats() == hb.get_stats()
    finally:
        ha.close()
        hb.close()


def test_prefill_full_size_qwen3_30b_a3b(dev):
    """A 2048-token prompt on one full Qwen3-30B-A3B layer (E=128, k=8, H=2048,
    I=768, S=25): the whole layer is staged and the tensor-core grouped GEMMs
    run; a sample of the tokens (near-tie rows included, on the GPU's routing)
    is checked against the oracle row by row."""
    st_ = Stack(QWEN3_30B_A3B, num_layers=1, tokens=1, batch=2048, stream=2)
    c = st_.cfg
    T = 2048
    h = st_.handle(torch, dev)
    try:
        x = st_.x[0, 0, :T]
        out = torch.empty((T, c.hidden), dtype=torch.int16, device=dev)
        h.decode_layer(0, _bits(x).to(dev), T, out)
        torch.cuda.synchronize()
        times = h.prefill_times()
        gemm_kernels = h.prefill_gemm_ms()
        stats = h.get_stats()
        gids, gw = _gpu_route(h, 0, x, dev)
    finally:
        h.close()
    assert times["staged"] and stats["staged_calls"] == 1 and stats["device_status"] == 0
    assert times["gemm"] > 0 and times["copy"] > 0
    assert 0 < gemm_kernels <= times["gemm"]  # the GEMM launches alone, inside the bucketing + GEMM phase
    sample = np.arange(0, T, 97)
    check_layer(_u16(out)[sample], x[sample], st_.wr[0], st_.w13[0], st_.w2[0], c.top_k, True, gids[sample],
                gw[sample])


def test_prefill_mixtral_8x7b_layer_full_size(dev):
    """Tensor-core prefill on one Mixtral-8x7B-shaped layer (E=8, k=2, H=4096, I=14336,
    S=4, 512 tokens, staged): 112 gate/up and 16 down column blocks per row tile, K up
    to 14336; sampled rows, near-ties included, against the oracle on the GPU's routing."""
    T = 512
    st_ = Stack(MIXTRAL_8X7B, num_layers=1, tokens=1, batch=T, stream=9)
    c = st_.cfg
    h = st_.handle(torch, dev, num_slots=4)
    try:
        x = st_.x[0, 0, :T]
        out = torch.empty((T, c.hidden), dtype=torch.int16, device=dev)
        h.decode_layer(0, _bits(x).to(dev), T, out)
        torch.cuda.synchronize()
        times = h.prefill_times()
        gemm_kernels = h.prefill_gemm_ms()
        stats = h.get_stats()
        gids, gw = _gpu_route(h, 0, x, dev)
    finally:
        h.close()
    assert times["staged"] and stats["device_status"] == 0
    assert 0 < gemm_kernels <= times["gemm"]
    sample = np.arange(0, T, 29)
    check_layer(_u16(out)[sample], x[sample], st_.wr[0], st_.w13[0], st_.w2[0], c.top_k, True, gids[sample],
                gw[sample])


@pytest.mark.parametrize("T, S, staged", [(333, 25, True), (64, 128, False)])
def test_prefill_ragged_and_slot_path_qwen3_30b_a3b(dev, T, S, staged):
    """Tensor-core prefill on one full Qwen3-30B-A3B layer at a token count that leaves
    every bucket's last 128-row tile ragged (T=333, staged), and on the slot path (S=128:
    every distinct expert gets a slot, so the GEMMs read the slot tensors after the
    ensure and miss copy); sampled rows, near-ties included, against the oracle on the
    GPU's routing."""
    st_ = Stack(QWEN3_30B_A3B, num_layers=1, tokens=1, batch=T, stream=6)
    c = st_.cfg
    h = st_.handle(torch, dev, num_slots=S)
    try:
        x = st_.x[0, 0, :T]
        out = torch.empty((T, c.hidden), dtype=torch.int16, device=dev)
        h.decode_layer(0, _bits(x).to(dev), T, out)
        torch.cuda.synchronize()
        times = h.prefill_times()
        gemm_kernels = h.prefill_gemm_ms()
        stats = h.get_stats()
        gids, gw = _gpu_route(h, 0, x, dev)
    finally:
        h.close()
    assert times["staged"] == staged and stats["device_status"] == 0
    assert 0 < gemm_kernels <= times["gemm"]
    sample = np.arange(0, T, 7)
    check_layer(_u16(out)[sample], x[sample], st_.wr[0], st_.w13[0], st_.w2[0], c.top_k, True, gids[sample],
                gw[sample])


def test_prefill_speculative_staging_in_and_out_of_order(dev):
    """Layer l+1 is staged while layer l computes; calls in order, out of order,
    repeated and interleaved with decode calls all give the oracle's outputs,
    and every staged call counts its bytes once."""
    import oracle
    st_ = Stack(TINY, num_layers=4, tokens=2, batch=48, stream=5)
    c = st_.cfg
    T = 48
    h = st_.handle(torch, dev, num_slots=4)
    try:
        out = torch.empty((T, c.hidden), dtype=torch.int16, device=dev)
        o1 = torch.empty((1, c.hidden), dtype=torch.int16, device=dev)
        order = [0, 1, 2, 3, 2, 0, 3, 1, 1]
        for n, l in enumerate(order):
            x = st_.x[0, l, :T]
            h.decode_layer(l, _bits(x).to(dev), T, out)
            if n == 4:
                h.decode_layer(0, _bits(st_.x[1, 0, :1]).to(dev), 1, o1)   # a decode call in between
            torch.cuda.synchronize()
            assert h.prefill_times()["staged"]
            gids, gw = _gpu_route(h, l, x, dev)
            check_layer(_u16(out), x, st_.wr[l], st_.w13[l], st_.w2[l], c.top_k, True, gids, gw, ctx=(n, l))
        stats = h.get_stats()
        B_e = c.expert_bytes
        assert stats["staged_calls"] == len(order)
        assert stats["staged_bytes"] == len(order) * c.num_experts * B_e
    finally:
        h.close()


# ----------------------------------------------------------- auto sizing
def test_auto_slot_count_from_free_device_memory(dev, tiny):
    """num_slots = 0 ("MoE expert offload" page, Options table: `auto` sizes every
    layer's slots from the free VRAM after loading, less a reserve): the count
    the library chose equals the oracle's closed form on the free bytes it read;
    a reserve that leaves room for fewer than top_k slots fails with
    MOE_ERR_OOM; an auto-sized handle decodes the oracle's outputs."""
    import oracle
    from expert_cache_router_gb300 import MoeOffloadError
    c = tiny.cfg
    L, E, k = c.num_layers, c.num_experts, c.top_k
    B = c.expert_bytes
    probe = tiny.handle(torch, dev, num_slots=0, auto_reserve_bytes=1 << 20)
    try:
        assert probe.num_slots == oracle.slots_auto(probe.auto_free_bytes, 1 << 20, L, E, k, B) == E
        free0 = probe.auto_free_bytes
    finally:
        probe.close()
    for want_s in (4, 6):
        # free memory moves by a few MB between creates; the check is against what the library read
        reserve = free0 - int((want_s + 0.5) * L * B)
        h = tiny.handle(torch, dev, num_slots=0, auto_reserve_bytes=reserve)
        try:
            assert h.num_slots == oracle.slots_auto(h.auto_free_bytes, reserve, L, E, k, B)
            assert k <= h.num_slots < E
            if want_s == 4:
                routing = []
                out = _decode_all(h, tiny, dev, 4, tokens=4, routing=routing)
                st = h.get_stats()
                assert st["device_status"] == 0 and st["misses"] > 0
                _check_outputs(tiny, out, routing, 4, ctx="auto")
        finally:
            h.close()
    with pytest.raises(MoeOffloadError) as ei:
        tiny.handle(torch, dev, num_slots=0, auto_reserve_bytes=free0 + (1 << 30))
    assert ei.value.status == 3 and "auto slots" in str(ei.value)
