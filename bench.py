#!/usr/bin/env python
"""Offloaded MoE decode benchmark on one GB300 (replicas for --gpus N).

Workload (default): the Qwen3-30B-A3B-shaped stack, 48 layers x 128 experts,
top-8, H=2048, I=768, 25 GPU slots per layer, bf16 experts (54 GiB) in pinned,
mapped host RAM, Zipf(1.1)-like skewed AR(1) router inputs, synthetic and
seeded. One step = one decode token through all 48 MoE layers (route, LRU slot
ensure, miss copy, grouped FFN), replayed as one CUDA graph. Every timed pass
starts from an empty slot table.

Prints ONE JSON line (rank 0). Timed passes over the same K-token stream:
  A  graph replays, inputs resident in HBM                   -> value, ms_per_step
  B  the same steps with CUDA events around each layer's kernels -> roofline
  E  end to end through moe_offload_graph_launch_host        -> e2e
plus pass A at batch 8 and the CPU oracle on a bounded sample -> cpu_baseline.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from dataclasses import replace

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "offloaded MoE decode tok/s at batch 1/8; misses/token; H2D & HBM GB/s vs peak"
DTYPE_NAME = {False: "bf16", True: "fp8_e4m3_b128 weights x bf16 activations, fp32 accumulate"}
# DRAM bytes (read + write) per launch of the two decode FFN kernels, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum, one pass) of four steady-state launches of each
# current kernel on a two-layer stack of this layer shape at batch 1 (LRU, no lookahead; gate/up:
# the mean of two launches with one expert installed and two with none); the profiles directory
# holds the command and the figures. Installed experts arrive over NVLink-C2C, which is not DRAM traffic, and their
# slot writes stay in L2 within a launch. Workloads without a capture report null.
NCU_DRAM_BYTES_PER_LAUNCH = {
    "qwen3_30b_a3b_L48_E128_k8_H2048_I768_S25": {"gate_up": 47.31e6, "down": 25.26e6},
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=256)
    p.add_argument("--warmup", type=int, default=16)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="qwen3", choices=["qwen3", "mixtral", "tiny", "fp8", "tiny_fp8"])
    p.add_argument("--slots", type=int, default=0, help="override slots per layer")
    p.add_argument("--layers", type=int, default=0, help="override the layer count (quick checks only)")
    p.add_argument("--no-b8", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-prefill", action="store_true")
    p.add_argument("--no-trace", action="store_true", help="skip the untimed traced passes")
    p.add_argument("--no-sub", action="store_true",
                   help="skip the Mixtral-8x7B-shape and FP8-lookahead sub-runs of the default workload")
    p.add_argument("--prefill-tokens", type=int, default=2048)
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--policy", choices=["lru", "static"], default="lru",
                   help="slot policy: LRU eviction, or a static top-S placement profiled on a separate stream")
    p.add_argument("--profile-tokens", type=int, default=64)
    p.add_argument("--prefetch", type=int, default=-1,
                   help="router-lookahead experts per layer (default: the workload's own setting)")
    return p.parse_args()


def workload(args):
    from workload import QWEN3_30B_A3B, MIXTRAL_8X7B, TINY, FP8_LOOKAHEAD, TINY_FP8
    cfg = {"qwen3": QWEN3_30B_A3B, "mixtral": MIXTRAL_8X7B, "tiny": TINY, "fp8": FP8_LOOKAHEAD,
           "tiny_fp8": TINY_FP8}[args.workload]
    if args.slots:
        cfg = replace(cfg, num_slots=args.slots)
    if args.layers:
        cfg = replace(cfg, num_layers=args.layers)
    if args.prefetch >= 0:
        cfg = replace(cfg, prefetch_n=args.prefetch)
    return cfg


class Dist:
    """Rank bookkeeping; replicas only (no data-path collective)."""

    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons, sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "power_w_max": max(r["power"] for r in rows)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except Exception:
        return {}


def h2d_ceiling(torch, dev) -> float:
    """Pinned cudaMemcpyAsync host->device ceiling in GB/s (1 GiB copies, best of 5)."""
    n = 1 << 30
    src = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    src.fill_(1)
    dst = torch.empty(n, dtype=torch.uint8, device=dev)
    best = float("inf")
    for i in range(7):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        b.synchronize()
        if i >= 2:
            best = min(best, a.elapsed_time(b))
    del src, dst
    return n / (best * 1e-3) / 1e9


_PINNED = []


def pinned_allocator(shape, dtype=None):
    """Host store in pinned, mapped memory from the CUDA library (moe_offload_host_alloc).
    On GB300, GPU reads of registered pageable memory ran at 18-160 GB/s in some
    address ranges, pinned memory at the full 211 GB/s everywhere."""
    import numpy as np
    from expert_cache_router_gb300 import PinnedHostArray
    a = PinnedHostArray(shape, np.uint16 if dtype is None else dtype)
    _PINNED.append(a)
    return a.array


class Store:
    """Synthetic host expert store of a workload: bf16 experts, or FP8 e4m3
    experts with 128 x 128 block scales (and a shared expert per layer)."""

    def __init__(self, cfg, prefix="", allocator=None, layers=None):
        """layers: generate only these layers' experts (row i holds layer layers[i])."""
        from workload import gen
        t0 = time.time()
        self.cfg = cfg
        self.layers = list(range(cfg.num_layers)) if layers is None else list(layers)
        self.row = {l: i for i, l in enumerate(self.layers)}
        part = replace(cfg, num_layers=len(self.layers))
        self.s13 = self.s2 = self.shared = None
        if cfg.fp8:
            self.w13, self.s13, self.w2, self.s2 = gen.alloc_fp8_store(part, allocator)
            gen.fill_fp8_store(cfg, self.w13, self.s13, self.w2, self.s2, layers=self.layers)
            if cfg.shared_expert:
                self.shared = gen.shared_experts_fp8(cfg)
        else:
            self.w13, self.w2 = gen.alloc_expert_store(part, allocator)
            gen.fill_expert_store(cfg, self.w13, self.w2, layers=self.layers)
        self.wr = gen.router_weights(cfg)
        self.mu = gen.input_means(cfg, self.wr)
        log(f"{prefix}host store {part.host_bytes / 2**30:.1f} GiB ({len(self.layers)} layers) generated in "
            f"{time.time() - t0:.1f} s")

    def inputs(self, n_tokens, batch, stream=0):
        from workload import gen
        f = gen.router_inputs_2d if self.cfg.ar_layers else gen.router_inputs
        return f(self.cfg, self.mu, n_tokens, batch, stream=stream)

    def handle(self, torch, dev, router, device=0):
        from expert_cache_router_gb300 import MoeOffload
        c = self.cfg
        L = c.num_layers
        moe = MoeOffload(num_layers=L, num_experts=c.num_experts, top_k=c.top_k, hidden=c.hidden,
                         inter=c.inter, num_slots=c.num_slots, host_w13=[self.w13[l] for l in range(L)],
                         host_w2=[self.w2[l] for l in range(L)], router=router, renormalize=c.renormalize,
                         max_tokens_graph=8, device=device, dtype="fp8" if c.fp8 else "bf16",
                         host_s13=[self.s13[l] for l in range(L)] if c.fp8 else None,
                         host_s2=[self.s2[l] for l in range(L)] if c.fp8 else None,
                         shared_expert=bool(self.shared), prefetch_n=c.prefetch_n)
        if self.shared:
            import numpy as np
            for l, sh in enumerate(self.shared):
                q13, s13, q2, s2 = (torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in sh)
                moe.set_shared_expert(l, q13, q2, s13, s2)
        return moe

    def oracle_token(self, x, l):
        """The oracle on one layer of one token batch x [B, H]: route, top-k, FFN, combine."""
        import oracle
        c = self.cfg
        i = self.row[l]
        if not c.fp8:
            return oracle.moe_layer(x, self.wr[l], self.w13[i], self.w2[i], c.top_k, c.renormalize)
        ids, w = oracle.topk(oracle.router_logits(x, self.wr[l]), c.top_k, c.renormalize)
        return oracle.moe_ffn_fp8(x, ids, w, self.w13[i], self.s13[i], self.w2[i], self.s2[i],
                                  shared=self.shared[l] if self.shared else None)

    def shared_bytes(self):
        """(W13, W2) bytes of one layer's shared expert, 0 without one."""
        if not self.shared:
            return 0, 0
        q13, s13, q2, s2 = self.shared[0]
        return q13.nbytes + s13.nbytes, q2.nbytes + s2.nbytes

    def expert_split(self):
        """(W13, W2) bytes of one routed expert, block scales included."""
        c = self.cfg
        if c.fp8:
            return (self.w13[0, 0].nbytes + self.s13[0, 0].nbytes, self.w2[0, 0].nbytes + self.s2[0, 0].nbytes)
        return self.w13[0, 0].nbytes, self.w2[0, 0].nbytes


def cpu_oracle_rate(store, x, seconds):
    """The oracle (plain C, OpenMP over output rows) on the first tokens of the
    timed stream at batch 1: route + top-k + k-expert FFN, every layer, until
    `seconds` have passed. Returns (tok/s, tokens, threads, seconds)."""
    import oracle
    oracle.build()
    t0 = time.time()
    tokens = 0
    while tokens < x.shape[0]:
        for l in range(store.cfg.num_layers):
            store.oracle_token(x[tokens, l, :1], l)
        tokens += 1
        if time.time() - t0 >= seconds:
            break
    dt = time.time() - t0
    return tokens / dt, tokens, oracle.num_threads(), dt


def trace_pass(P, cfg, xdev, tokens, skip=16):
    """Untimed: the decode graph with the trace on (moe_offload_trace_enable), one
    token at a time from an empty table, records read after each token. Returns, for
    layer calls with and without installed experts after the first `skip` tokens, the
    median of each segment of a layer in microseconds."""
    import numpy as np
    import torch
    from expert_cache_router_gb300 import DecodeGraph, _lib as C
    moe, L, H = P.moe, cfg.num_layers, cfg.hidden
    f = {n: i for i, n in enumerate(C.TRACE_FIELD_NAMES)}
    gx = torch.zeros((L, 1, H), dtype=torch.int16, device=xdev.device)
    go = torch.zeros_like(gx)
    P.restart()
    moe.trace_enable(True)
    g = DecodeGraph(moe, 1, gx, go)
    rows = {True: [], False: []}
    try:
        for t in range(tokens):
            gx.copy_(xdev[t])
            g.launch(P.stream)
            rec = moe.trace_read(reset=True).astype(np.float64) / 1e3   # us
            if t < skip:
                continue
            for l in range(1, L):
                r, prev = rec[l], rec[l - 1]
                _, n_miss, n_spill = moe.read_misses(l)
                seg = {"release_after_previous_down": r[f["head_wait"]] - prev[f["down_done"]],
                       "head": r[f["head_done"]] - r[f["head_wait"]],
                       "head_logits": r[f["head_logits"]] - r[f["head_wait"]],
                       "head_topk": r[f["head_topk"]] - r[f["head_logits"]],
                       "head_table": r[f["head_done"]] - r[f["head_topk"]],
                       "head_to_gate_up": r[f["gate_first"]] - r[f["head_done"]],
                       "gate_up": r[f["gate_done"]] - r[f["gate_first"]],
                       "down_tail_after_gate_up": r[f["down_out"]] - r[f["gate_done"]],
                       "down_waits_after_gate_up": r[f["down_waits"]] - r[f["gate_done"]],
                       "layer": r[f["down_done"]] - prev[f["down_done"]]}
                if n_miss - n_spill > 0:
                    seg["first_host_bytes_after_gate_up_start"] = r[f["host_first"]] - r[f["gate_first"]]
                    seg["host_stream_end_to_gate_up_end"] = r[f["gate_done"]] - max(r[f["copy_done"]],
                                                                                    r[f["host_done"]])
                rows[n_miss - n_spill > 0].append(seg)
    finally:
        g.close()
        moe.trace_enable(False)
        torch.cuda.synchronize()

    def med(rs):
        keys = sorted({k for r in rs for k in r})
        return {k: round(float(np.median([r[k] for r in rs if k in r])), 2) for k in keys}
    return {"tokens": tokens, "skipped": skip, "layer_calls_with_installs": len(rows[True]),
            "layer_calls_without": len(rows[False]), "with_installs_us": med(rows[True]),
            "without_installs_us": med(rows[False]),
            "how": "globaltimer stamps of the traced one-token kernels (moe_offload_trace_read), medians over "
                   "layers 1..L-1 of every token after the first `skipped`; untimed: a traced step runs "
                   "slightly slower than the timed one"}


def prefill_pass(args, cfg, moe, store, dev, stream):
    """Prefill of one prompt through every layer (the staging path when a layer's
    distinct experts outnumber its slots), then 64 decode tokens on the slots.
    Returns a dict for the JSON line."""
    import numpy as np
    import torch
    L, H, T = cfg.num_layers, cfg.hidden, args.prefill_tokens
    xp = store.inputs(T, 1, stream=2)                                     # [T, L, 1, H]
    xl = torch.from_numpy(np.ascontiguousarray(xp[:, :, 0, :].transpose(1, 0, 2)).view(np.int16)).to(dev)
    out = torch.empty((T, H), dtype=torch.int16, device=dev)
    moe.reset()
    moe.decode_layer(0, xl[0], T, out, stream)                            # sizes the prefill scratch
    torch.cuda.synchronize()
    moe.reset()
    phases = np.zeros(4)
    staged = 0
    last = None
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    last_kernels = None
    for l in range(L):
        moe.decode_layer(l, xl[l], T, out, stream)
        t = moe.prefill_times()
        phases += [t["route"], t["copy"], t["gemm"], t["combine"]]
        staged += int(t["staged"])
        last = t
        if l == L - 1:
            try:
                last_kernels = moe.prefill_gemm_ms()  # the two tensor-core GEMM launches alone
            except Exception:
                last_kernels = None  # CUDA-core GEMMs (shapes the tensor-core tiles do not cover)
    b.record(stream)
    torch.cuda.synchronize()
    secs = a.elapsed_time(b) * 1e-3
    st = moe.get_stats()
    # 64 decode tokens after the prompt, on the slot path (the table was left untouched by staged layers)
    xd = torch.from_numpy(store.inputs(64, 1, stream=3).view(np.int16)).to(dev)
    o1 = torch.empty((1, H), dtype=torch.int16, device=dev)
    c, d = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c.record(stream)
    for t in range(64):
        for l in range(L):
            moe.decode_layer(l, xd[t, l], 1, o1, stream)
    d.record(stream)
    torch.cuda.synchronize()
    gemm_flop = 2.0 * T * (cfg.top_k + (1 if cfg.shared_expert else 0)) * (2 * cfg.inter * H + H * cfg.inter)
    peaks = measured_peaks()
    route_ms, copy_ms, gemm_ms, comb_ms = (phases / L).tolist()
    tflops = gemm_flop / (gemm_ms * 1e-3) / 1e12 if gemm_ms else None
    # The last layer stages no next layer, so its GEMM phase runs with the SMs and HBM to
    # itself: the grouped GEMMs' roofline is taken there. At ~128 rows per expert the GEMMs
    # are bound by the staged weight bytes (every expert's W13 and W2 read once from HBM).
    # Staged weights are bf16 (FP8 experts are dequantised by the staging copy), the shared
    # expert staged as one more group.
    weight_bytes = (cfg.num_experts + (1 if cfg.shared_expert else 0)) * 3 * cfg.hidden * cfg.inter * 2
    lg = last_kernels * 1e-3 if last and last["staged"] and last_kernels else None
    gemm_roof = None
    if lg:
        ach = weight_bytes / lg / 1e9
        gemm_roof = {"kernel": "tc_grouped_gemm (gate/up + SiLU, then down): the two launches, CUDA events around them",
                     "bound": "hbm", "achieved": ach, "peak": peaks.get("hbm_gbs"), "unit": "GB/s",
                     "frac": ach / peaks["hbm_gbs"] if peaks.get("hbm_gbs") else None,
                     "hbm_bytes_per_layer": weight_bytes, "ms": last_kernels,
                     "tflops": gemm_flop / lg / 1e12,
                     "frac_of_bf16_peak": (gemm_flop / lg / 1e12) / peaks["bf16_tflops"] if peaks.get("bf16_tflops") else None,
                     "phase_ms_with_bucketing_and_gather": last["gemm"],
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs and bf16_tflops (burst, of measured)",
                     "layer": L - 1}
    return {"workload": f"prefill {T} tokens then 64 decode tokens, {cfg.name}",
            "prompt_tokens": T, "ms": secs * 1e3, "tok_s": T / secs, "layers_staged": staged,
            "per_layer_ms": {"route_topk_distinct": route_ms, "staging_copy_or_wait": copy_ms,
                             "bucket_gather_grouped_gemms": gemm_ms, "combine": comb_ms},
            "staged_gbs_over_prefill": st["staged_bytes"] / secs / 1e9,
            "staging_note": "layer l+1 is staged into a second buffer while layer l computes; the copy phase "
                            "of a layer is the wait for its staging",
            "gemm_tflops_with_staging_alongside": tflops,
            "gemm_roofline_last_layer": gemm_roof,
            "decode_after_prefill_tok_s": 64 / (c.elapsed_time(d) * 1e-3),
            "note": "prefill is host-synchronised per layer (distinct-expert count); GEMM time includes bucketing and the row gather"}


def run_reference(args, dist):
    """Reference arm: the CPU oracle, as it stands, on this machine's host cores."""
    cfg = workload(args)
    if dist.rank != 0:
        return
    from workload import gen
    import oracle
    K, W = args.steps, args.warmup
    L = cfg.num_layers
    # Each step is one token through a sample of at most 12 evenly spaced layers (time scaled to
    # all layers): the oracle's cost per layer does not depend on which layer it is, and the
    # host store it needs stays small (12 of 48 layers: 14 GiB instead of 54 GiB).
    n = min(L, 12)
    cand = sorted(set(int(i * L / n) for i in range(n)))
    store = Store(cfg, layers=cand)
    oracle.build()
    x = store.inputs(K + max(W, 1), 1)
    t0 = time.time()
    for t in range(max(W, 1)):
        for l in cand:
            store.oracle_token(x[t, l, :1], l)
    per_layer = (time.time() - t0) / (max(W, 1) * len(cand))
    # fewer sampled layers when K tokens over all candidates would pass about 150 s
    layers = max(1, min(len(cand), int(150.0 / max(K * per_layer, 1e-9))))
    sample_layers = sorted(set(cand[int(i * len(cand) / layers)] for i in range(layers)))
    t0 = time.time()
    for t in range(K):
        for l in sample_layers:
            store.oracle_token(x[max(W, 1) + t, l, :1], l)
    dt = time.time() - t0
    step = dt / K * (L / len(sample_layers))
    value = 1.0 / step
    if len(sample_layers) < L:
        sample = (f"{K} decode tokens at batch 1, {len(sample_layers)} of {L} layers per token "
                  f"(layers {','.join(map(str, sample_layers))}), time scaled to {L} layers")
    else:
        sample = f"{K} decode tokens at batch 1, all {L} layers"
    line = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus, "steps": K, "warmup": W,
            "ms_per_step": step * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE_NAME[cfg.fp8], "data": "synthetic", "impl": "reference",
            "config": {"workload": cfg.name, "batch": 1, "parallelism": "replicas"},
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


REPEATS = 5       # timed passes of the headline workload (median reported, min and max beside it)
SUB_REPEATS = 3   # timed passes of each sub-workload variant


def release_pinned():
    """Free every host store allocated through pinned_allocator."""
    for a in _PINNED:
        a.close()
    _PINNED.clear()


class Passes:
    """Timed decode passes of one handle: graph replays over a K-token stream,
    each pass from an empty slot table (LRU) or from the placement (static)."""

    def __init__(self, moe, dist, stream, static=False):
        self.moe, self.dist, self.stream, self.static = moe, dist, stream, static

    def restart(self):
        if not self.static:
            self.moe.reset()
        return self.moe.get_stats() if self.static else None

    @staticmethod
    def delta(st, before):
        return st if before is None else {k: st[k] - before[k] if k != "device_status" else st[k] for k in st}

    def timed(self, graph, gx, xdev, K, instrument=False):
        """K replays: (seconds max over ranks, per-phase ms sums, stats delta)."""
        import numpy as np
        import torch
        before = self.restart()
        sums = np.zeros(3)
        self.dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for t in range(K):
            gx.copy_(xdev[t])
            graph.launch(self.stream)
            if instrument:
                sums += np.array([a.sum() for a in graph.times()], dtype=np.float64)
        e1.record(self.stream)
        torch.cuda.synchronize()
        self.dist.barrier()
        return self.dist.max(e0.elapsed_time(e1) * 1e-3), sums, self.delta(self.moe.get_stats(), before)


def decode_batch(P, cfg, B, xw, xt, xt_host, K, W, repeats, stream, full=True, sampler=None, e2e=False):
    """One batch size: warm-up, `repeats` plain passes (pass A), and with full=True the
    instrumented pass (B) and the misses of the first 16 tokens; e2e adds the host-buffer pass."""
    import numpy as np
    import torch
    from expert_cache_router_gb300 import DecodeGraph
    L, H = cfg.num_layers, cfg.hidden
    moe = P.moe
    gx = torch.zeros((L, B, H), dtype=torch.int16, device=xt.device)
    go = torch.zeros((L, B, H), dtype=torch.int16, device=xt.device)
    g_plain = DecodeGraph(moe, B, gx, go, timing=False)
    for t in range(W):                          # warm-up on its own token stream
        gx.copy_(xw[t])
        g_plain.launch(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    runs = [P.timed(g_plain, gx, xt, K) for _ in range(repeats)]
    clocks = sampler.stop() if sampler else None
    secs = [r[0] for r in runs]
    med = sorted(range(repeats), key=lambda i: secs[i])[repeats // 2]
    r = dict(secs=secs[med], secs_all=secs, stats=runs[med][2], launches=g_plain.kernel_count * K, clocks=clocks)
    if full:
        g_timed = DecodeGraph(moe, B, gx, go, timing=True)
        _, r["phase_ms"], r["stats_b"] = P.timed(g_timed, gx, xt, K, instrument=True)
        g_timed.close()
        before16 = P.restart()                 # misses of the first 16 tokens, for the steady state
        n0 = min(16, K)
        for t in range(n0):
            gx.copy_(xt[t])
            g_plain.launch(stream)
        early = P.delta(moe.get_stats(), before16)["misses"]
        r["steady_misses"] = (r["stats"]["misses"] - early) / max(K - n0, 1)
    if e2e:
        # as many passes as the device-timed value, median taken the same way
        xh = torch.from_numpy(xt_host.view(np.int16)).pin_memory()
        oh = torch.empty((K, L, B, H), dtype=torch.int16).pin_memory()
        e2e_all = []
        for _ in range(repeats):
            P.restart()
            P.dist.barrier()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for t in range(K):
                g_plain.launch_host(xh[t], oh[t], stream)
            b.record(stream)
            torch.cuda.synchronize()
            e2e_all.append(P.dist.max(a.elapsed_time(b) * 1e-3))
        r["e2e_secs"] = sorted(e2e_all)[repeats // 2]
        r["e2e_secs_all"] = e2e_all
    g_plain.close()
    return r


def summarize(cfg, store, r1, K, world, link, hbm_peak, traffic=None):
    """Throughput, misses, link bound, per-layer time split and the two FFN kernels'
    rooflines of a batch-1 result of decode_batch(full=True)."""
    L = cfg.num_layers
    B_e = cfg.expert_bytes
    h2d_gbs = link["copy_engine_gbs"]
    stats = r1["stats"]
    head_ms, gu_ms, dn_ms = r1["phase_ms"]
    total_ms = head_ms + gu_ms + dn_ms
    sb = r1["stats_b"]
    launches = K * L                           # launches of each of the three kernels in pass B
    installs = sb["misses"] - sb["spills"]
    w13_b, w2_b = store.expert_split()
    sh13_b, sh2_b = store.shared_bytes()
    traffic = traffic or {}
    # gate/up launch: installed experts cross the host link whole (W13 computed through, W2
    # copied by its copy CTAs), spilled experts' W13 too; resident experts' W13 come from HBM
    gu_host = installs * B_e + sb["spills"] * w13_b
    # reads of resident W13 + writes into slots (+ the shared expert's W13, every layer)
    gu_hbm = sb["hits"] * w13_b + installs * B_e + launches * sh13_b
    dn_hbm = (sb["hits"] + installs) * w2_b + launches * sh2_b
    dn_host = sb["spills"] * w2_b
    gu_s, dn_s = gu_ms * 1e-3, dn_ms * 1e-3
    gu_bound_s = max(gu_host / (h2d_gbs * 1e9), gu_hbm / (hbm_peak * 1e9) if hbm_peak else 0.0)
    dn_bound_s = max(dn_host / (h2d_gbs * 1e9), dn_hbm / (hbm_peak * 1e9) if hbm_peak else 0.0)
    phases = {"route_topk_ensure": head_ms, "gate_up_with_miss_copy": gu_ms, "down_combine": dn_ms}
    gu_ach = gu_host / gu_s / 1e9 if gu_s else 0.0
    gu_roof = {"kernel": "ffn_gate_up_kernel (moe_grouped_ffn gate/up with the miss copy folded in)",
               "bound": "h2d", "achieved": gu_ach, "peak": h2d_gbs,
               "unit": "GB/s", "frac": gu_ach / h2d_gbs if gu_s else None,
               "traffic": traffic.get("gate_up"),
               "peak_source": "pinned cudaMemcpyAsync host->device ceiling measured in this run (1 GiB copies)",
               "frac_of_sm_read_ceiling": gu_ach / link["sm_read_gbs"] if link.get("sm_read_gbs") else None,
               "host_bytes_per_launch": gu_host / launches, "hbm_bytes_per_launch": gu_hbm / launches,
               "ms_per_launch": gu_ms / launches,
               "frac_of_bound": gu_bound_s / gu_s if gu_s else None}
    dn_roof = {"kernel": "ffn_down_combine_kernel", "bound": "hbm",
               "achieved": dn_hbm / dn_s / 1e9 if dn_s else 0.0, "peak": hbm_peak, "unit": "GB/s",
               "frac": (dn_hbm / dn_s / 1e9) / hbm_peak if (dn_s and hbm_peak) else None,
               "traffic": traffic.get("down"),
               "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)",
               "hbm_bytes_per_launch": dn_hbm / launches, "ms_per_launch": dn_ms / launches,
               "frac_of_bound": dn_bound_s / dn_s if dn_s else None}
    link_bytes = stats["bytes_copied"] + stats["prefetch_bytes"]
    secs = r1["secs"]
    tok = [world * K / x for x in r1["secs_all"]]
    us = 1e3 / launches
    out = {
        "value": world * K / secs, "unit": "tok/s", "ms_per_step": secs / K * 1e3, "tokens": K,
        "repeats": {"n": len(tok), "median": statistics.median(tok), "min": min(tok), "max": max(tok)},
        "misses_per_token": stats["misses"] / K,
        "misses_per_token_steady": r1.get("steady_misses"),
        "hit_rate": stats["hits"] / max(stats["hits"] + stats["misses"], 1),
        "miss_bytes_per_token": stats["bytes_copied"] / K,
        "link_bytes_per_token": link_bytes / K,
        "copy_bound_tok_s": (h2d_gbs * 1e9) / (link_bytes / K) if link_bytes else None,
        "frac_of_copy_bound": (world * K / secs) / ((h2d_gbs * 1e9) / (link_bytes / K)) if link_bytes else None,
        "lookahead": {"prefetch_n": cfg.prefetch_n,
                      "installs_per_token": stats["prefetch_installs"] / K,
                      "hits_per_token": stats["prefetch_hits"] / K,
                      "bytes_per_token": stats["prefetch_bytes"] / K} if cfg.prefetch_n else None,
        "phase_share": {p: round(v / total_ms, 4) for p, v in phases.items()},
        # per layer, from the instrumented pass (events between the launches, so no overlap):
        # gate/up's link time is its host bytes at the copy-engine ceiling; the rest of
        # gate/up is its start (slot ids, grouping, first host bytes) and its HBM-side work
        "per_layer_us": {"head": head_ms * us, "gate_up": gu_ms * us,
                         "gate_up_link_at_ceiling": gu_host / launches / (h2d_gbs * 1e9) * 1e6,
                         "gate_up_beyond_link": gu_ms * us - gu_host / launches / (h2d_gbs * 1e9) * 1e6,
                         "down_tail": dn_ms * us},
        "roofline": gu_roof if gu_ms >= dn_ms else dn_roof,
        "roofline_other": dn_roof if gu_ms >= dn_ms else gu_roof,
        "dominant_kernel": max(phases, key=phases.get),
        "gpu_launches": r1["launches"],
    }
    return out


def sub_workload(args, base, variants, K, W, dev, stream, dist, link, hbm_peak, cpu_seconds=0.0):
    """Another workload on the driver's clock: its own host store (freed afterwards), one
    handle per variant (slot count or lookahead depth), SUB_REPEATS timed passes each; with
    cpu_seconds > 0 (rank 0) also the oracle on the first tokens of the same stream, which
    does not depend on the variant."""
    import numpy as np
    import torch
    store = Store(base, f"[rank {dist.rank}] ", allocator=pinned_allocator)
    try:
        router = [torch.from_numpy(store.wr[l].view(np.int16)).to(dev) for l in range(base.num_layers)]
        xw = torch.from_numpy(store.inputs(W, 1, stream=1).view(np.int16)).to(dev)
        xt_host = store.inputs(K, 1, stream=0)
        xt = torch.from_numpy(xt_host.view(np.int16)).to(dev)
        res = {}
        for label, cfg in variants:
            store.cfg = cfg
            moe = store.handle(torch, dev, router, device=dist.local)
            try:
                P = Passes(moe, dist, stream)
                r = decode_batch(P, cfg, 1, xw, xt, xt_host, K, W, SUB_REPEATS, stream)
                res[label] = dict(workload=cfg.name, slots=cfg.num_slots, prefetch_n=cfg.prefetch_n,
                                  warmup=W, **summarize(cfg, store, r, K, dist.world, link, hbm_peak))
                if dist.rank == 0 and not args.no_trace:
                    res[label]["trace"] = trace_pass(P, cfg, xt, min(K, 64))
            finally:
                moe.close()
        if cpu_seconds > 0 and dist.rank == 0:
            rate, ntok, cores, dt = cpu_oracle_rate(store, xt_host, cpu_seconds)
            res["cpu_baseline"] = {"value": rate, "unit": "tok/s", "cores": cores, "kind": "oracle",
                                   "sample": f"first {ntok} tokens of the timed stream at batch 1, all "
                                             f"{base.num_layers} layers ({dt:.1f} s)"}
        return res
    finally:
        del store
        release_pinned()


def run_ours(args, dist):
    import numpy as np
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from expert_cache_router_gb300 import DecodeGraph, PinnedHostArray, host_read_gbs

    cfg = workload(args)
    K, W = args.steps, args.warmup
    if W < 3:
        raise SystemExit("at least 3 warm-up steps")
    dev = torch.device(f"cuda:{dist.local}")
    torch.cuda.set_device(dev)
    L, H, k = cfg.num_layers, cfg.hidden, cfg.top_k
    B_e = cfg.expert_bytes

    store = Store(cfg, f"[rank {dist.rank}] ", allocator=pinned_allocator)
    router = [torch.from_numpy(store.wr[l].view(np.int16)).to(dev) for l in range(L)]
    batches = [1] if (args.no_b8 or 8 not in cfg.batches) else [1, 8]
    xs = {}
    for B in batches:
        xw = store.inputs(W, B, stream=1)
        xt = store.inputs(K, B, stream=0)
        xs[B] = (torch.from_numpy(xw.view(np.int16)).to(dev), torch.from_numpy(xt.view(np.int16)).to(dev), xt)

    t0 = time.time()
    moe = store.handle(torch, dev, router, device=dist.local)
    log(f"[rank {dist.rank}] handle created in {time.time() - t0:.1f} s, "
        f"{moe.device_bytes() / 2**30:.1f} GiB on the device")
    probe = PinnedHostArray((1 << 29,), np.uint16)      # 1 GiB, pinned and mapped
    probe.array.fill(1)
    link = {"copy_engine_gbs": h2d_ceiling(torch, dev),
            "sm_read_gbs": host_read_gbs(probe.array, dist.local),
            "nominal_pcie_gen5_x16_gbs": 64.0,
            "how": "copy engine: pinned cudaMemcpyAsync host->device, 1 GiB, best of 5; SM reads: "
                   "moe_offload_host_read_gbs (16-byte loads of pinned mapped memory, two CTAs per SM), "
                   "1 GiB, best of 5"}
    probe.close()
    hbm_peak = measured_peaks().get("hbm_gbs")
    stream = torch.cuda.current_stream()

    static = args.policy == "static"
    P = Passes(moe, dist, stream, static)
    placement = None
    if static:
        # Profile on its own token stream with LRU, plan the top-S experts of every layer, freeze.
        from expert_cache_router_gb300 import plan_static
        Pt = args.profile_tokens
        xp = torch.from_numpy(store.inputs(Pt, 1, stream=5).view(np.int16)).to(dev)
        gx = torch.zeros((L, 1, H), dtype=torch.int16, device=dev)
        go = torch.zeros_like(gx)
        g = DecodeGraph(moe, 1, gx, go)
        moe.reset()
        for t in range(Pt):
            gx.copy_(xp[t])
            g.launch(stream)
        torch.cuda.synchronize()
        g.close()
        placed = routed = 0
        for l in range(L):
            counts = moe.read_route_counts(l)
            plan = plan_static(counts, cfg.num_slots)
            moe.set_placement(l, plan)
            placed += int(counts[plan].sum())
            routed += int(counts.sum())
        placement = {"name": "static top-S placement", "profile_tokens": Pt,
                     "profile_stream": "its own seeded stream (not the timed one)",
                     "profile_pairs_served_by_slots": placed / max(routed, 1)}
        log(f"[rank {dist.rank}] static placement from {Pt} profiled tokens: "
            f"{placed / max(routed, 1):.3f} of profiled pairs on slots")

    results = {}
    for B in batches:
        xw, xt, xt_host = xs[B]
        results[B] = decode_batch(P, cfg, B, xw, xt, xt_host, K, W, REPEATS if B == 1 else 1, stream,
                                  full=(B == 1), sampler=ClockSampler(dist.local) if B == 1 else None,
                                  e2e=(B == 1 and not args.no_e2e))

    trace = None
    if not static and dist.rank == 0 and not args.no_trace:
        trace = trace_pass(P, cfg, xs[1][1], min(K, 64))
    r1 = results[1]
    world = dist.world
    stats = r1["stats"]
    traffic = NCU_DRAM_BYTES_PER_LAUNCH.get(cfg.name, {}) if (args.policy == "lru" and not cfg.prefetch_n) else {}
    m = summarize(cfg, store, r1, K, world, link, hbm_peak, traffic)
    line = {
        "metric": METRIC, "value": m["value"], "unit": "tok/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": m["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE_NAME[cfg.fp8], "data": "synthetic",
        "config": {"workload": cfg.name, "batch": 1, "layers": L, "experts": cfg.num_experts, "top_k": k,
                   "host_store": "pinned mapped host memory (moe_offload_host_alloc)",
                   "hidden": H, "inter": cfg.inter, "slots": cfg.num_slots, "expert_bytes": B_e,
                   "shared_expert": bool(store.shared), "prefetch_n": cfg.prefetch_n,
                   "host_store_gib": round(cfg.host_bytes / 2**30, 2),
                   "l2": "inputs larger than L2: each step reads %.2f GB of expert weights"
                         % ((stats["hits"] + stats["misses"]) * B_e / K / 1e9),
                   "timing": f"value = median of {REPEATS} timed passes of K steps, each from an empty "
                             f"slot table; min and max under repeats",
                   "parallelism": f"replicas x{world}"},
        "slot_policy": placement if static else "lru",
        "link": link,
        "h2d_gbs_per_step": stats["bytes_copied"] / r1["secs"] / 1e9,
        "head_us_per_layer": m["per_layer_us"]["head"],
        "clocks": r1["clocks"],
    }
    for key in ("repeats", "misses_per_token", "misses_per_token_steady", "hit_rate", "miss_bytes_per_token",
                "link_bytes_per_token", "copy_bound_tok_s", "frac_of_copy_bound", "lookahead", "phase_share",
                "per_layer_us", "roofline", "roofline_other", "dominant_kernel", "gpu_launches"):
        line[key] = m[key]
    if 8 in results:
        r8 = results[8]
        s8 = r8["stats"]
        line["batch8"] = {"value": world * K * 8 / r8["secs"], "unit": "tok/s", "ms_per_step": r8["secs"] / K * 1e3,
                          "misses_per_step": s8["misses"] / K, "spills_per_step": s8["spills"] / K,
                          "misses_per_token": s8["misses"] / (K * 8), "gpu_launches": r8["launches"]}
    if "e2e_secs" in r1:
        nbytes = L * H * 2
        line["e2e"] = {"value": world * K / r1["e2e_secs"], "unit": "tok/s", "h2d_bytes_per_step": nbytes,
                       "d2h_bytes_per_step": nbytes,
                       "repeats": {"n": len(r1["e2e_secs_all"]),
                                   "min": world * K / max(r1["e2e_secs_all"]),
                                   "max": world * K / min(r1["e2e_secs_all"])},
                       "path": "moe_offload_graph_launch_host: pinned host in, graph replay, pinned host out, per step; "
                               "median of the passes, each from an empty slot table like the device-timed value"}
    if trace is not None:
        line["trace"] = trace
    if not args.no_prefill and cfg.num_experts > cfg.num_slots and not static:
        line["prefill"] = prefill_pass(args, cfg, moe, store, dev, stream)
    moe.close()
    if dist.rank == 0:
        rate, ntok, cores, dt = cpu_oracle_rate(store, xs[1][2], args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": "tok/s", "cores": cores, "kind": "oracle",
                                "sample": f"first {ntok} tokens of the timed stream at batch 1, all {L} layers "
                                          f"({dt:.1f} s)"}
    del store
    release_pinned()
    if not args.no_sub and args.workload == "qwen3" and not static and not args.layers:
        from workload import MIXTRAL_8X7B, FP8_LOOKAHEAD
        # Mixtral-8x7B shape (S = 2 and 4) and the FP8 + lookahead workload (N = 0 and 4), each
        # over its own configured token count and seeded streams
        mx = MIXTRAL_8X7B
        line["mixtral"] = sub_workload(args, mx, [(f"S{S}", replace(mx, num_slots=S)) for S in (2, 4)],
                                       mx.decode_tokens, max(W, 3), dev, stream, dist, link, hbm_peak,
                                       cpu_seconds=min(args.cpu_seconds, 10.0))
        f8 = FP8_LOOKAHEAD
        line["fp8_lookahead"] = sub_workload(args, f8, [(f"N{N}", replace(f8, prefetch_n=N)) for N in (0, 1, 2, 4)],
                                             f8.decode_tokens, max(W, 3), dev, stream, dist, link, hbm_peak,
                                             cpu_seconds=min(args.cpu_seconds, 10.0))
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    dist = Dist()
    if args.impl == "reference":
        run_reference(args, dist)
    else:
        run_ours(args, dist)


if __name__ == "__main__":
    main()
