"""Parity bars shared by the GPU tests.

Routing: the GPU's routed ids equal the oracle's, except on rows where the
oracle's k-th and (k+1)-th logits lie within TIE of each other. On such a row
the GPU may pick the other side of the near-tie; its picks must still be a valid
top-k of the oracle's logits up to TIE, and its weights must be the softmax of
the oracle's logits taken at its own ids.

Layer outputs: the oracle FFN is evaluated on the GPU's own routed ids and
weights, so that every row is checked, near-tie rows included, and each row's
relative L2 error against the oracle's fp32 output (before its bf16 rounding)
must be at most TOL. A norm pooled over a whole call would let one bad row
through when the others are good.
"""
from __future__ import annotations

import numpy as np

TIE = 1e-3
TOL = 5e-3


def rel_l2_rows(got, want) -> np.ndarray:
    """Relative L2 error of every row of got against want ([T, H] each)."""
    got = np.asarray(got, np.float64).reshape(np.shape(want)[0], -1)
    want = np.asarray(want, np.float64).reshape(got.shape[0], -1)
    num = np.linalg.norm(got - want, axis=1)
    den = np.maximum(np.linalg.norm(want, axis=1), 1e-30)
    return num / den


def assert_rows(got, want, tol: float = TOL, ctx=None) -> float:
    """Every row within tol; returns the worst row's error."""
    r = rel_l2_rows(got, want)
    worst = float(r.max()) if r.size else 0.0
    assert worst <= tol, f"row {int(np.argmax(r))} rel-L2 {worst:.3e} > {tol} {ctx if ctx is not None else ''}"
    return worst


def logit_gap(lg, k: int) -> np.ndarray:
    """Per row: k-th minus (k+1)-th largest logit (inf when E == k)."""
    lg = np.asarray(lg, np.float64)
    if lg.shape[1] <= k:
        return np.full(lg.shape[0], np.inf)
    s = -np.sort(-lg, axis=1)
    return s[:, k - 1] - s[:, k]


def check_routing(lg, k: int, renorm: bool, gpu_ids, gpu_w, w_rtol: float = 1e-4) -> np.ndarray:
    """Checks the GPU's routing against the oracle's logits lg [T, E] (fp32 from
    the oracle). Returns the mask of rows whose ids equal the oracle's top-k."""
    import oracle
    lg = np.asarray(lg, np.float32)
    gpu_ids = np.asarray(gpu_ids).reshape(lg.shape[0], k)
    gpu_w = np.asarray(gpu_w, np.float64).reshape(lg.shape[0], k)
    rid, rw = oracle.topk(lg, k, renorm)
    same = np.all(gpu_ids == rid, axis=1)
    gap = logit_gap(lg, k)
    assert np.all(same | (gap < TIE)), "routing differs away from a near-tie"
    if same.any():
        assert np.allclose(gpu_w[same], rw[same], rtol=1e-5, atol=1e-7)
    lg64 = lg.astype(np.float64)
    for t in np.flatnonzero(~same):
        ids = gpu_ids[t]
        assert len(set(ids.tolist())) == k and ids.min() >= 0 and ids.max() < lg.shape[1]
        kth = -np.sort(-lg64[t])[k - 1]
        # every GPU pick lies within TIE of the oracle's k-th logit or above it,
        # in descending order up to TIE
        picked = lg64[t, ids]
        assert np.all(picked >= kth - TIE), (t, ids, picked, kth)
        assert np.all(np.diff(picked) <= TIE), (t, ids, picked)
        e = np.exp(picked - picked.max())
        want = e / e.sum() if renorm else np.exp(picked - lg64[t].max()) / np.exp(lg64[t] - lg64[t].max()).sum()
        assert np.allclose(gpu_w[t], want, rtol=w_rtol, atol=1e-6), (t, gpu_w[t], want)
    return same


def check_layer(got_bits, x, wr, w13, w2, k: int, renorm: bool, gpu_ids, gpu_w, tol: float = TOL,
                fp8=None, shared=None, extra=None, ctx=None) -> float:
    """One layer call: routing against the oracle's logits, then every output row
    against the oracle FFN on the GPU's ids and weights. got_bits [T, H] bf16 bits;
    fp8 = (s13, s2) for FP8 experts (w13/w2 hold e4m3 codes); shared = the FP8
    shared expert (w13, s13, w2, s2) or None; extra = an fp32 [T, H] term the
    oracle adds to its output (a bf16 shared expert). Returns the worst row error."""
    import oracle
    lg = oracle.router_logits(x, wr)
    check_routing(lg, k, renorm, gpu_ids, gpu_w)
    ids = np.asarray(gpu_ids, np.int32).reshape(-1, k)
    w = np.asarray(gpu_w, np.float32).reshape(-1, k)
    if fp8 is None:
        want, _ = oracle.moe_ffn(x, ids, w, w13, w2)
    else:
        want, _ = oracle.moe_ffn_fp8(x, ids, w, w13, fp8[0], w2, fp8[1], shared=shared)
    if extra is not None:
        want = want + np.asarray(extra, np.float32)
    got = oracle.bf16_to_f32(np.asarray(got_bits).view(np.uint16))
    return assert_rows(got, want, tol, ctx)
