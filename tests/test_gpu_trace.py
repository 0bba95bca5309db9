"""Decode trace (moe_offload_trace_enable / moe_offload_trace_read): the stamps of a
traced decode graph are in step order within a layer and across layers, layers
with installed experts stamp the host fields, and tracing changes no output bit."""
import numpy as np
import pytest

from workload import TINY
from stack import Stack

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _run(h, st, dev, tokens, trace):
    from expert_cache_router_gb300 import DecodeGraph
    c = st.cfg
    h.reset()
    if trace:
        h.trace_enable(True)
    xb = torch.zeros((c.num_layers, 1, c.hidden), dtype=torch.int16, device=dev)
    ob = torch.zeros_like(xb)
    g = DecodeGraph(h, 1, xb, ob)
    xs = torch.from_numpy(np.ascontiguousarray(st.x[:tokens, :, :1]).view(np.int16)).to(dev)
    outs, recs, installs = [], [], []
    try:
        for t in range(tokens):
            xb.copy_(xs[t])
            g.launch()
            torch.cuda.synchronize()
            outs.append(ob.cpu().numpy().copy())
            if trace:
                recs.append(h.trace_read(reset=True))
                installs.append([h.read_misses(l)[1] - h.read_misses(l)[2] for l in range(c.num_layers)])
    finally:
        g.close()
        if trace:
            h.trace_enable(False)
    return np.stack(outs), recs, installs


def test_decode_trace_is_ordered_and_changes_no_output(dev):
    from expert_cache_router_gb300 import _lib as C
    st = Stack(TINY, num_layers=4, tokens=12)
    h = st.handle(torch, dev, num_slots=2)  # few slots: most layers install experts
    try:
        plain, _, _ = _run(h, st, dev, 12, trace=False)
        traced, recs, installs = _run(h, st, dev, 12, trace=True)
        assert np.array_equal(plain, traced)
        f = {n: i for i, n in enumerate(C.TRACE_FIELD_NAMES)}
        unset_min = np.uint64(0xFFFFFFFFFFFFFFFF)
        seen_install = False
        for t, (rec, inst) in enumerate(zip(recs, installs)):
            for l in range(st.cfg.num_layers):
                r = rec[l]
                order = [r[f["head_wait"]], r[f["head_logits"]], r[f["head_topk"]], r[f["head_done"]],
                         r[f["gate_first"]], r[f["gate_done"]], r[f["down_done"]]]
                assert all(v > 0 for v in order), (t, l, r)
                assert r[f["gate_first"]] != unset_min and r[f["down_first"]] != unset_min
                assert all(a <= b for a, b in zip(order, order[1:])), (t, l, order)
                assert r[f["down_first"]] <= r[f["down_done"]] and r[f["down_waits"]] <= r[f["down_done"]]
                assert r[f["down_waits"]] <= r[f["down_out"]] <= r[f["down_done"]]
                if l + 1 < st.cfg.num_layers:  # the next head passes its wait after this down completes
                    assert rec[l + 1][f["head_wait"]] >= r[f["down_done"]]
                if inst[l] > 0:
                    seen_install = True
                    assert r[f["host_first"]] != unset_min and r[f["gate_first"]] <= r[f["host_first"]]
                    # the W2 copy may finish before the installed expert's first W13 chunk is used
                    assert r[f["host_first"]] <= r[f["host_done"]] <= r[f["gate_done"]]
                    assert r[f["copy_done"]] <= r[f["gate_done"]]
                else:
                    assert r[f["host_first"]] == unset_min
        assert seen_install
        # off again: a plain graph stamps nothing
        h.trace_enable(True)
        h.trace_read(reset=True)
        h.trace_enable(False)
        _run(h, st, dev, 2, trace=False)
        rec = h.trace_read(reset=False)
        assert np.all(rec[:, f["head_done"]] == 0) and np.all(rec[:, f["gate_first"]] == unset_min)
    finally:
        h.close()
