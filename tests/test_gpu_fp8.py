"""FP8 e4m3 experts with 128 x 128 block scales and the always-resident shared
expert: CUDA path vs the oracle, through the C ABI.

Bars as for bf16: every row of every layer output within relative L2 5e-3 of
the oracle's fp32 output, the oracle evaluated on the GPU's own routing (near-tie
rows included); slot bytes and slot scales bit-exact against the host store;
outputs bit-identical across slot counts (spills included) and between graph
replay and eager calls."""
import numpy as np
import pytest

from workload import TINY, TINY_FP8, FP8_LOOKAHEAD, gen
from stack import Stack, Fp8Stack
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
def tiny8():
    return Fp8Stack(TINY_FP8, tokens=8, batch=8)


def _bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))


def _u16(t):
    return t.cpu().numpy().view(np.uint16)


def _gpu_route(h, layer, x, dev):
    T = x.shape[0]
    ids = torch.empty((T, h.top_k), dtype=torch.int32, device=dev)
    w = torch.empty((T, h.top_k), dtype=torch.float32, device=dev)
    h.route_topk(layer, _bits(x).to(dev), T, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


def _decode_all(h, st, dev, T, tokens, routing=None):
    c = st.cfg
    xd = _bits(st.x[:tokens, :, :T]).to(dev)
    out = torch.empty((tokens, c.num_layers, T, c.hidden), dtype=torch.int16, device=dev)
    for t in range(tokens):
        if routing is not None:
            routing.append([])
        for l in range(c.num_layers):
            h.decode_layer(l, xd[t, l], T, out[t, l])
            if routing is not None:
                routing[t].append(h.read_routing())
    torch.cuda.synchronize()
    return _u16(out)


def _check_fp8(st, got_bits, x, l, ids, w, shared=True, ctx=None):
    c = st.cfg
    check_layer(got_bits, x, st.wr[l], st.w13[l], st.w2[l], c.top_k, c.renormalize, ids, w,
                fp8=(st.s13[l], st.s2[l]), shared=st.shared[l] if shared else None, ctx=ctx)


def _check_vs_oracle(st, out, routing, T, shared=True):
    for t in range(len(routing)):
        for l in range(st.cfg.num_layers):
            ids, w, _ = routing[t][l]
            _check_fp8(st, out[t, l], st.x[t, l, :T], l, ids, w, shared, ctx=(t, l))


@pytest.mark.parametrize("shared", [True, False])
@pytest.mark.parametrize("T", [1, 3, 8])
def test_fp8_decode_matches_oracle_tiny(dev, tiny8, T, shared):
    h = tiny8.handle(torch, dev, shared=shared)
    routing = []
    try:
        out = _decode_all(h, tiny8, dev, T, tokens=6, routing=routing)
        assert h.get_stats()["device_status"] == 0
    finally:
        h.close()
    _check_vs_oracle(tiny8, out, routing, T, shared)


def test_fp8_slots_hold_store_bytes_and_scales(dev, tiny8):
    c = tiny8.cfg
    h = tiny8.handle(torch, dev, num_slots=6)
    try:
        _decode_all(h, tiny8, dev, 8, tokens=4)
        seen = 0
        for l in range(c.num_layers):
            se, _, _, _ = h.read_table(l)
            for s, e in enumerate(se.tolist()):
                if e < 0:
                    continue
                w13, w2 = h.read_slot(l, s)
                s13, s2 = h.read_slot_scales(l, s)
                assert np.array_equal(w13, tiny8.w13[l, e]) and np.array_equal(w2, tiny8.w2[l, e])
                assert np.array_equal(s13.view(np.uint32), tiny8.s13[l, e].view(np.uint32))
                assert np.array_equal(s2.view(np.uint32), tiny8.s2[l, e].view(np.uint32))
                seen += 1
        assert seen == 6 * c.num_layers
    finally:
        h.close()


def test_fp8_outputs_bit_identical_across_slot_counts(dev, tiny8):
    """Placement never changes the result: S from k (spills at batch 8) to E."""
    c = tiny8.cfg
    ref = None
    for S in (c.top_k, 3, 4, 8, c.num_experts):
        h = tiny8.handle(torch, dev, num_slots=S)
        try:
            out = _decode_all(h, tiny8, dev, 8, tokens=4)
            stats = h.get_stats()
        finally:
            h.close()
        if S == c.top_k:
            assert stats["spills"] > 0
        if ref is None:
            ref = out
        else:
            assert np.array_equal(out, ref), S


def test_fp8_library_graph_matches_eager(dev, tiny8):
    from expert_cache_router_gb300 import DecodeGraph
    c = tiny8.cfg
    T = 4
    h = tiny8.handle(torch, dev)
    try:
        eager = _decode_all(h, tiny8, dev, T, tokens=6)
        h.reset()
        xb = torch.zeros((c.num_layers, T, c.hidden), dtype=torch.int16, device=dev)
        ob = torch.zeros_like(xb)
        g = DecodeGraph(h, T, xb, ob)
        xs = _bits(tiny8.x[:6, :, :T]).to(dev)
        got = []
        for t in range(6):
            xb.copy_(xs[t])
            g.launch()
            got.append(_u16(ob.clone()))
        assert np.array_equal(np.stack(got), eager)
        g.close()
    finally:
        h.close()


def test_fp8_rejects_missing_shared_expert(dev, tiny8):
    from expert_cache_router_gb300 import MoeOffloadError
    c = tiny8.cfg
    x = _bits(tiny8.x[0, 0, :1]).to(dev)
    out = torch.empty((1, c.hidden), dtype=torch.int16, device=dev)
    h = tiny8.handle(torch, dev, set_shared=False)
    try:
        with pytest.raises(MoeOffloadError) as ei:
            h.decode_layer(0, x, 1, out)
        assert ei.value.status == 1 and "shared expert" in str(ei.value)
    finally:
        h.close()



def test_bf16_shared_expert_is_added_after_the_routed_ranks(dev):
    """bf16 handle with a shared expert: out = bf16(sum_j w_j y_j + y_shared)."""
    import oracle
    from expert_cache_router_gb300 import MoeOffload
    st = Stack(TINY, tokens=4, batch=8)
    c = st.cfg
    L, H, I = c.num_layers, c.hidden, c.inter
    sh = [(gen.random_bf16((2 * I, H), seed=900 + l, std=c.weight_std),
           gen.random_bf16((H, I), seed=950 + l, std=c.weight_std)) for l in range(L)]
    shd = [(_bits(a).to(dev), _bits(b).to(dev)) for a, b in sh]
    h = MoeOffload(num_layers=L, num_experts=c.num_experts, top_k=c.top_k, hidden=H, inter=I,
                   num_slots=c.num_slots, host_w13=[st.w13[l] for l in range(L)],
                   host_w2=[st.w2[l] for l in range(L)], router=st.router_dev(torch, dev),
                   renormalize=c.renormalize, max_tokens_graph=8, shared_expert=True)
    routing = []
    try:
        for l in range(L):
            h.set_shared_expert(l, shd[l][0], shd[l][1])
        T = 8
        out = _decode_all(h, st, dev, T, tokens=4, routing=routing)
    finally:
        h.close()
    for t in range(4):
        for l in range(L):
            x = st.x[t, l, :T]
            xf = oracle.bf16_to_f32(x)
            ysh = np.stack([oracle.expert_ffn(sh[l][0], sh[l][1], xf[i]) for i in range(T)])
            ids, w, _ = routing[t][l]
            check_layer(out[t, l], x, st.wr[l], st.w13[l], st.w2[l], c.top_k, c.renormalize, ids, w, extra=ysh,
                        ctx=(t, l))


@pytest.mark.parametrize("T", [1, 4])
def test_fp8_full_size_layers(dev, T):
    """The 256-expert FP8 shape (k=8, H=2048, I=512, 25 slots, shared expert) on two layers."""
    st = Fp8Stack(FP8_LOOKAHEAD, num_layers=2, tokens=4, batch=T)
    h = st.handle(torch, dev)
    routing = []
    try:
        out = _decode_all(h, st, dev, T, tokens=4, routing=routing)
        s = h.get_stats()
        assert s["device_status"] == 0 and s["misses"] > 0
    finally:
        h.close()
    _check_vs_oracle(st, out, routing, T)


@pytest.mark.parametrize("shared", [True, False])
def test_fp8_prefill_matches_oracle(dev, shared):
    """Prefill (T above the graph bound) of FP8 experts: staged with dequantisation to bf16
    (one more rounding of each weight than the oracle's fp32 product), shared expert as
    one more group; outputs within the same relative L2 bar."""
    st = Fp8Stack(TINY_FP8, tokens=1, batch=48)
    c = st.cfg
    T = 48
    h = st.handle(torch, dev, max_tokens_graph=4, shared=shared)
    try:
        out = torch.empty((T, c.hidden), dtype=torch.int16, device=dev)
        for l in range(c.num_layers):
            x = st.x[0, l, :T]
            h.decode_layer(l, _bits(x).to(dev), T, out)
            torch.cuda.synchronize()
            assert h.prefill_times()["staged"]
            ids, w = _gpu_route(h, l, x, dev)
            _check_fp8(st, _u16(out), x, l, ids, w, shared, ctx=l)
        assert h.get_stats()["staged_calls"] == c.num_layers
    finally:
        h.close()


def test_fp8_full_size_prefill(dev):
    """The 256-expert FP8 shape with its shared expert, a 128-token prompt on two layers (tensor-core GEMMs)."""
    st = Fp8Stack(FP8_LOOKAHEAD, num_layers=2, tokens=1, batch=128)
    c = st.cfg
    h = st.handle(torch, dev)
    try:
        out = torch.empty((128, c.hidden), dtype=torch.int16, device=dev)
        for l in range(2):
            x = st.x[0, l, :128]
            h.decode_layer(l, _bits(x).to(dev), 128, out)
            torch.cuda.synchronize()
            sample = np.arange(0, 128, 8)
            ids, w = _gpu_route(h, l, x, dev)
            _check_fp8(st, _u16(out)[sample], x[sample], l, ids[sample], w[sample], ctx=l)
    finally:
        h.close()


def test_bf16_shared_expert_prefill(dev):
    import oracle
    from expert_cache_router_gb300 import MoeOffload
    st = Stack(TINY, tokens=1, batch=40)
    c = st.cfg
    L, H, I = c.num_layers, c.hidden, c.inter
    sh = [(gen.random_bf16((2 * I, H), seed=700 + l, std=c.weight_std),
           gen.random_bf16((H, I), seed=750 + l, std=c.weight_std)) for l in range(L)]
    shd = [(_bits(a).to(dev), _bits(b).to(dev)) for a, b in sh]
    h = MoeOffload(num_layers=L, num_experts=c.num_experts, top_k=c.top_k, hidden=H, inter=I,
                   num_slots=c.num_slots, host_w13=[st.w13[l] for l in range(L)],
                   host_w2=[st.w2[l] for l in range(L)], router=st.router_dev(torch, dev),
                   renormalize=c.renormalize, max_tokens_graph=8, shared_expert=True)
    try:
        for l in range(L):
            h.set_shared_expert(l, shd[l][0], shd[l][1])
        T = 40
        out = torch.empty((T, H), dtype=torch.int16, device=dev)
        for l in range(L):
            x = st.x[0, l, :T]
            h.decode_layer(l, _bits(x).to(dev), T, out)
            torch.cuda.synchronize()
            xf = oracle.bf16_to_f32(x)
            ysh = np.stack([oracle.expert_ffn(sh[l][0], sh[l][1], xf[i]) for i in range(T)])
            ids, w = _gpu_route(h, l, x, dev)
            check_layer(_u16(out), x, st.wr[l], st.w13[l], st.w2[l], c.top_k, c.renormalize, ids, w, extra=ysh,
                        ctx=l)
    finally:
        h.close()
