"""The grouped FFN entry point that allocates nothing.

It is meant for callers that cannot call cudaMalloc (their serving runtime owns
every byte of device memory through its own allocator, or they may not allocate
after start-up). Through the C ABI it must give what the handle-based
moe_offload_grouped_ffn gives, within the tests' relative-L2 bound of 5e-3, on
two calls in a row (the shared scratch array keeps the first call's contents),
and it must refuse sizes beyond its fixed scratch with MOE_ERR_INVALID.

This file is collected last on purpose; it also runs alone in a fresh process.
"""
import numpy as np
import pytest

from workload import TINY
from stack import Stack, rel_l2

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
TOL = 5e-3


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))


def test_noalloc_ffn_matches_handle_ffn_on_two_calls(dev):
    import oracle
    from expert_cache_router_gb300 import grouped_ffn_noalloc
    st = Stack(TINY, num_layers=1, tokens=2, batch=8)
    c = st.cfg
    E, k, H, I = c.num_experts, c.top_k, c.hidden, c.inter
    w13_d = _bits(st.w13[0]).to(dev)
    w2_d = _bits(st.w2[0]).to(dev)
    h = st.handle(torch, dev, num_slots=E)
    rng = np.random.default_rng(21)
    try:
        for call, T in enumerate((8, 3)):
            x = st.x[call, 0, :T]
            ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
            w = rng.random((T, k)).astype(np.float32)
            x_d, ids_d, w_d = _bits(x).to(dev), torch.from_numpy(ids).to(dev), torch.from_numpy(w).to(dev)
            # the existing entry point, through a handle (slots hold the experts)
            slot_d = torch.empty_like(ids_d)
            h.slot_ensure(0, ids_d, T, slot_d)
            h.miss_copy(0)
            out_ref = torch.empty((T, H), dtype=torch.int16, device=dev)
            h.grouped_ffn(0, x_d, slot_d, w_d, T, out_ref)
            # the allocation-free entry point on the same inputs
            status = torch.zeros(1, dtype=torch.int32, device=dev)
            out_new = torch.full((T, H), -1, dtype=torch.int16, device=dev)
            grouped_ffn_noalloc(w13_d, w2_d, E, H, I, x_d, ids_d, w_d, T, k, out_new, status=status)
            torch.cuda.synchronize()
            # the same kernels over the resident [E, N, K] arrays and over the slot tensors:
            # identical arithmetic, so identical bits (the "bit-exact GEMM test of the
            # generic path" of the MoE expert offload page, "Supported" section)
            assert np.array_equal(out_new.cpu().numpy(), out_ref.cpu().numpy()), f"call {call}"
            got = oracle.bf16_to_f32(out_new.cpu().numpy().view(np.uint16))
            assert int(status.item()) == 0
            want, _ = oracle.moe_ffn(x, ids, w, st.w13[0], st.w2[0])
            assert rel_l2(got, want) <= TOL
    finally:
        h.close()


def test_noalloc_ffn_rejects_sizes_beyond_its_scratch(dev):
    from expert_cache_router_gb300 import grouped_ffn_noalloc, MoeOffloadError
    E, k, H, I, T = 8, 2, 256, 512, 33           # T*k = 66 > 64
    w13 = torch.zeros((E, 2 * I, H), dtype=torch.int16, device=dev)
    w2 = torch.zeros((E, H, I), dtype=torch.int16, device=dev)
    x = torch.zeros((T, H), dtype=torch.int16, device=dev)
    ids = torch.zeros((T, k), dtype=torch.int32, device=dev)
    w = torch.zeros((T, k), dtype=torch.float32, device=dev)
    out = torch.zeros((T, H), dtype=torch.int16, device=dev)
    with pytest.raises(MoeOffloadError) as ei:
        grouped_ffn_noalloc(w13, w2, E, H, I, x, ids, w, T, k, out)
    assert ei.value.status == 1 and "exceeds" in str(ei.value)


def _noalloc_case(dev, E, k, H, I, T, seed):
    """Seeded weights, inputs, ids and weights for one no-alloc call (device tensors + host copies)."""
    from workload import gen
    w13 = gen.random_bf16((E, 2 * I, H), seed=seed, std=0.02)
    w2 = gen.random_bf16((E, H, I), seed=seed + 1, std=0.02)
    x = gen.random_bf16((T, H), seed=seed + 2, std=1.0)
    ids = gen.random_ids((T, k), E, seed=seed + 3)
    w = np.random.default_rng(seed + 4).random((T, k)).astype(np.float32)
    d = dict(w13=_bits(w13).to(dev), w2=_bits(w2).to(dev), x=_bits(x).to(dev),
             ids=torch.from_numpy(ids.astype(np.int32)).to(dev), w=torch.from_numpy(w).to(dev))
    return dict(w13=w13, w2=w2, x=x, ids=ids.astype(np.int32), w=w), d


@pytest.mark.parametrize("E,k,I,T", [(8, 2, 512, 32), (2, 2, 16384, 32)])
def test_noalloc_accepts_its_exact_limits(dev, E, k, I, T):
    """T*k = 64 pairs (the pair limit) and T*k*I = 2^20 fp32 values (the scratch
    limit, 4 MiB) are accepted; every row matches the oracle."""
    import oracle
    from expert_cache_router_gb300 import grouped_ffn_noalloc
    from parity import assert_rows
    H = 256
    assert T * k == 64 and T * k * I <= 1 << 20
    hst, d = _noalloc_case(dev, E, k, H, I, T, seed=31 + I)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.full((T, H), -1, dtype=torch.int16, device=dev)
    grouped_ffn_noalloc(d["w13"], d["w2"], E, H, I, d["x"], d["ids"], d["w"], T, k, out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want, _ = oracle.moe_ffn(hst["x"], hst["ids"], hst["w"], hst["w13"], hst["w2"])
    assert_rows(oracle.bf16_to_f32(out.cpu().numpy().view(np.uint16)), want)


def test_noalloc_rejects_one_step_past_the_scratch_limit(dev):
    """T*k = 64 and I = 16448: T*k*I is 64 x 64 floats past 2^20, refused before any launch."""
    from expert_cache_router_gb300 import grouped_ffn_noalloc, MoeOffloadError
    E, k, H, I, T = 2, 2, 256, 16448, 32
    out = torch.full((T, H), 7, dtype=torch.int16, device=dev)
    z = torch.zeros(16, dtype=torch.int32, device=dev)  # never read: the call is refused first
    with pytest.raises(MoeOffloadError) as ei:
        grouped_ffn_noalloc(z, z, E, H, I, z, z, z, T, k, out)
    assert ei.value.status == 1 and "fixed scratch" in str(ei.value)
    torch.cuda.synchronize()
    assert bool((out == 7).all())


def test_noalloc_flags_an_expert_id_outside_the_arrays(dev):
    """An id equal to E sets MOE_DEV_BAD_SLOT_ID in the caller's status word; the
    other tokens' rows are still computed."""
    import oracle
    from expert_cache_router_gb300 import grouped_ffn_noalloc
    from expert_cache_router_gb300._lib import MOE_DEV_BAD_SLOT_ID
    from parity import assert_rows
    E, k, H, I, T = 8, 2, 256, 512, 4
    hst, d = _noalloc_case(dev, E, k, H, I, T, seed=77)
    bad = hst["ids"].copy()
    bad[1, 0] = E
    d["ids"] = torch.from_numpy(bad).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.zeros((T, H), dtype=torch.int16, device=dev)
    grouped_ffn_noalloc(d["w13"], d["w2"], E, H, I, d["x"], d["ids"], d["w"], T, k, out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & MOE_DEV_BAD_SLOT_ID
    rows = [0, 2, 3]
    want, _ = oracle.moe_ffn(hst["x"][rows], hst["ids"][rows], hst["w"][rows], hst["w13"], hst["w2"])
    assert_rows(oracle.bf16_to_f32(out.cpu().numpy().view(np.uint16))[rows], want)


def test_noalloc_in_a_second_context_of_the_same_device(dev):
    """A plug-in runtime may call the entry point under a driver context of its
    own. In a second context on the same device (buffers allocated there, made
    current on this thread), two calls give the bits of the call in the first
    context: the scratch array's address is looked up in the current context on
    every call, so a cached address from the other context is never used."""
    import ctypes
    from expert_cache_router_gb300 import grouped_ffn_noalloc, _lib as C
    E, k, H, I, T = 8, 2, 256, 512, 5
    hst, d = _noalloc_case(dev, E, k, H, I, T, seed=91)
    ref = torch.zeros((T, H), dtype=torch.int16, device=dev)
    grouped_ffn_noalloc(d["w13"], d["w2"], E, H, I, d["x"], d["ids"], d["w"], T, k, ref)
    torch.cuda.synchronize()
    ref = ref.cpu().numpy()

    cu = ctypes.CDLL("libcuda.so.1")
    u64, vp, sz = ctypes.c_uint64, ctypes.c_void_p, ctypes.c_size_t
    for name, args in (("cuCtxGetCurrent", [ctypes.POINTER(vp)]),
                       ("cuCtxSetCurrent", [vp]),
                       ("cuCtxCreate_v2", [ctypes.POINTER(vp), ctypes.c_uint, ctypes.c_int]),
                       ("cuCtxDestroy_v2", [vp]),
                       ("cuCtxSynchronize", []),
                       ("cuDeviceGet", [ctypes.POINTER(ctypes.c_int), ctypes.c_int]),
                       ("cuMemAlloc_v2", [ctypes.POINTER(u64), sz]),
                       ("cuMemFree_v2", [u64]),
                       ("cuMemsetD32_v2", [u64, ctypes.c_uint, sz]),
                       ("cuMemcpyHtoD_v2", [u64, vp, sz]),
                       ("cuMemcpyDtoH_v2", [vp, u64, sz])):
        if not hasattr(cu, name):
            pytest.skip(f"driver without {name}")
        getattr(cu, name).argtypes = args
        getattr(cu, name).restype = ctypes.c_int

    def ck(r, what):
        assert r == 0, f"{what}: CUresult {r}"

    first = vp()
    ck(cu.cuCtxGetCurrent(ctypes.byref(first)), "cuCtxGetCurrent")
    cudev = ctypes.c_int()
    ck(cu.cuDeviceGet(ctypes.byref(cudev), dev.index or 0), "cuDeviceGet")
    ctx = vp()
    ck(cu.cuCtxCreate_v2(ctypes.byref(ctx), 0, cudev), "cuCtxCreate")  # current on this thread now
    bufs = []
    try:
        def put(a):
            a = np.ascontiguousarray(a)
            p = u64()
            ck(cu.cuMemAlloc_v2(ctypes.byref(p), max(a.nbytes, 16)), "cuMemAlloc")
            bufs.append(p.value)
            ck(cu.cuMemcpyHtoD_v2(p.value, a.ctypes.data, a.nbytes), "cuMemcpyHtoD")
            return p.value
        w13, w2, x = put(hst["w13"].view(np.int16)), put(hst["w2"].view(np.int16)), put(hst["x"].view(np.int16))
        ids, w = put(hst["ids"]), put(hst["w"])
        out, status = put(np.zeros((T, H), np.int16)), put(np.zeros(4, np.uint32))
        L = C.load()
        for call in range(2):
            ck(cu.cuMemsetD32_v2(out, 0x7FFF7FFF, T * H // 2), "cuMemsetD32")
            st = L.moe_offload_grouped_ffn_noalloc(w13, w2, E, H, I, x, ids, w, T, k, out, status, None)
            assert st == C.MOE_OK, L.moe_offload_last_error(None).decode()
            ck(cu.cuCtxSynchronize(), "cuCtxSynchronize")
            got = np.zeros((T, H), np.int16)
            ck(cu.cuMemcpyDtoH_v2(got.ctypes.data, out, got.nbytes), "cuMemcpyDtoH")
            sw = np.zeros(4, np.uint32)
            ck(cu.cuMemcpyDtoH_v2(sw.ctypes.data, status, sw.nbytes), "cuMemcpyDtoH")
            assert np.array_equal(got, ref), f"call {call} in the second context"
            assert int(sw[0]) == 0
    finally:
        for p in bufs:
            cu.cuMemFree_v2(p)
        cu.cuCtxDestroy_v2(ctx)
        cu.cuCtxSetCurrent(first)
    torch.cuda.synchronize()  # the first context still works
