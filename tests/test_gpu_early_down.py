"""The early down hand-off of the decode step (the down launch waits, per expert
group, on counters that the gate/up CTAs raise, instead of on the whole gate/up
launch) computes exactly what the full wait computes: eager and in the decode
graph, with hits, installs and spills in one call, bf16 and FP8 with the shared
expert, with and without the lookahead. With MOE_OFFLOAD_AUDIT=1 every table
update is followed by an audit that also requires the counters to be back at
zero, so a call that failed to reset them is reported."""
import numpy as np
import pytest

from stack import Fp8Stack, Stack
from workload import TINY, TINY_FP8

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


def _run(h, st, dev, T, tokens):
    """Eager decode_layer over tokens x layers, then the same tokens through the library's graph."""
    from expert_cache_router_gb300 import DecodeGraph
    c = st.cfg
    xd = _bits(st.x[:tokens, :, :T]).to(dev)
    out = torch.empty((tokens, c.num_layers, T, c.hidden), dtype=torch.int16, device=dev)
    for t in range(tokens):
        for l in range(c.num_layers):
            h.decode_layer(l, xd[t, l], T, out[t, l])
    torch.cuda.synchronize()
    eager = _u16(out)
    stats = h.get_stats()
    h.reset()
    xb = torch.zeros((c.num_layers, T, c.hidden), dtype=torch.int16, device=dev)
    ob = torch.zeros_like(xb)
    g = DecodeGraph(h, T, xb, ob)
    got = []
    for t in range(tokens):
        xb.copy_(xd[t])
        g.launch()
        got.append(_u16(ob.clone()))
    g.close()
    return eager, np.stack(got), stats


CASES = [
    # (name, stack kind, T, slots, lookahead)
    ("bf16 b1", "bf16", 1, None, 0),
    ("bf16 b4 spills", "bf16", 4, 2, 0),
    ("bf16 b8", "bf16", 8, 4, 0),
    ("bf16 b4 lookahead", "bf16", 4, None, 2),
    ("fp8+shared b1", "fp8", 1, None, 0),
    ("fp8+shared b8 spills", "fp8", 8, 8, 0),
]


@pytest.fixture(scope="module")
def stacks():
    return {"bf16": Stack(TINY, tokens=8, batch=8, stream=11),
            "fp8": Fp8Stack(TINY_FP8, tokens=8, batch=8, stream=11)}


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_early_down_equals_full_wait(dev, stacks, monkeypatch, case):
    name, kind, T, S, N = case
    st = stacks[kind]
    monkeypatch.setenv("MOE_OFFLOAD_AUDIT", "1")
    res = {}
    for early in ("0", "1"):
        monkeypatch.setenv("MOE_OFFLOAD_EARLY_DOWN", early)
        h = st.handle(torch, dev, num_slots=S, prefetch_n=N)
        try:
            eager, graph, stats = _run(h, st, dev, T, tokens=8)
            assert h.get_stats()["device_status"] == 0, name
        finally:
            h.close()
        assert stats["device_status"] == 0, name
        assert np.array_equal(graph, eager), name
        res[early] = (eager, stats)
    assert np.array_equal(res["0"][0], res["1"][0]), name
    for key in ("misses", "spills", "hits", "bytes_copied"):
        assert res["0"][1][key] == res["1"][1][key], (name, key)
    if "spills" in name:
        assert res["1"][1]["spills"] > 0, name


# ------------------------------------------------------------------ prefill
def _prefill(h, st, dev, T, layers):
    """One staged call of T tokens per layer; returns the outputs and the stats."""
    c = st.cfg
    out = torch.empty((layers, T, c.hidden), dtype=torch.int16, device=dev)
    for l in range(layers):
        h.decode_layer(l, _bits(st.x[0, l, :T]).to(dev), T, out[l])
    torch.cuda.synchronize()
    return _u16(out), h.get_stats()


PREFILL_CASES = [
    # (name, stack kind, T, slots): every call touches more distinct experts than slots, so it stages
    ("bf16 T48 S4", "bf16", 48, 4),
    ("fp8+shared T48", "fp8", 48, None),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=[c[0] for c in PREFILL_CASES])
def test_prefill_early_down_equals_full_wait(dev, monkeypatch, case):
    """The tensor-core prefill GEMMs with the down launch started under the gate/up
    launch (per-tile counts) write the same bits as with the down launch after it."""
    name, kind, T, S = case
    st = (Stack(TINY, num_layers=2, tokens=1, batch=T, stream=5) if kind == "bf16"
          else Fp8Stack(TINY_FP8, tokens=1, batch=T, stream=5))
    layers = st.cfg.num_layers
    res = {}
    for early in ("0", "1"):
        monkeypatch.setenv("MOE_OFFLOAD_EARLY_DOWN", early)
        h = st.handle(torch, dev, num_slots=S)
        try:
            res[early] = _prefill(h, st, dev, T, layers)
        finally:
            h.close()
        assert res[early][1]["device_status"] == 0, name
        assert res[early][1]["staged_calls"] == layers, name
    assert np.array_equal(res["0"][0], res["1"][0]), name


def test_prefill_early_down_full_size_qwen3_30b_a3b(dev, monkeypatch):
    """A 2048-token prompt on one full Qwen3-30B-A3B layer (hundreds of 128-row tiles,
    so down CTAs start while gate/up tiles are still running): same bits either way."""
    from workload import QWEN3_30B_A3B
    st = Stack(QWEN3_30B_A3B, num_layers=1, tokens=1, batch=2048, stream=2)
    res = {}
    for early in ("0", "1"):
        monkeypatch.setenv("MOE_OFFLOAD_EARLY_DOWN", early)
        h = st.handle(torch, dev)
        try:
            res[early] = _prefill(h, st, dev, 2048, 1)
        finally:
            h.close()
        assert res[early][1]["device_status"] == 0
        assert res[early][1]["staged_calls"] == 1
    assert np.array_equal(res["0"][0], res["1"][0])
