"""Test helper: a synthetic offloaded MoE stack (host store, routers, inputs) and
the CUDA handle over it. Inputs come from the seeded generator only."""
from __future__ import annotations

from dataclasses import replace

import numpy as np

from workload import gen


class Stack:
    def __init__(self, cfg, num_layers=None, tokens=16, batch=1, stream=0):
        if num_layers is not None:
            cfg = replace(cfg, num_layers=num_layers)
        self.cfg = cfg
        self.w13, self.w2 = gen.alloc_expert_store(cfg)
        gen.fill_expert_store(cfg, self.w13, self.w2)
        self.wr = gen.router_weights(cfg)
        self.mu = gen.input_means(cfg, self.wr)
        self.x = gen.router_inputs(cfg, self.mu, tokens, batch, stream=stream)  # [n, L, B, H]
        self._router_dev = None

    def router_dev(self, torch, dev):
        if self._router_dev is None:
            self._router_dev = [torch.from_numpy(self.wr[l].view(np.int16)).to(dev)
                                for l in range(self.cfg.num_layers)]
        return self._router_dev

    def handle(self, torch, dev, num_slots=None, max_tokens_graph=8, prefetch_n=0, auto_reserve_bytes=0):
        from expert_cache_router_gb300 import MoeOffload
        c = self.cfg
        return MoeOffload(num_layers=c.num_layers, num_experts=c.num_experts, top_k=c.top_k,
                          hidden=c.hidden, inter=c.inter,
                          num_slots=c.num_slots if num_slots is None else num_slots,
                          host_w13=[self.w13[l] for l in range(c.num_layers)],
                          host_w2=[self.w2[l] for l in range(c.num_layers)],
                          router=self.router_dev(torch, dev), renormalize=c.renormalize,
                          max_tokens_graph=max_tokens_graph, prefetch_n=prefetch_n,
                          auto_reserve_bytes=auto_reserve_bytes)


def rel_l2(got, want) -> float:
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))


class Fp8Stack:
    """FP8 e4m3 experts with 128 x 128 block scales and one shared expert per
    layer; inputs from the 2-D (token x layer) AR(1) generator."""

    def __init__(self, cfg, num_layers=None, tokens=8, batch=1, stream=0):
        if num_layers is not None:
            cfg = replace(cfg, num_layers=num_layers)
        self.cfg = cfg
        self.w13, self.s13, self.w2, self.s2 = gen.alloc_fp8_store(cfg)
        gen.fill_fp8_store(cfg, self.w13, self.s13, self.w2, self.s2)
        self.shared = gen.shared_experts_fp8(cfg)
        self.wr = gen.router_weights(cfg)
        self.mu = gen.input_means(cfg, self.wr)
        self.x = gen.router_inputs_2d(cfg, self.mu, tokens, batch, stream=stream)  # [n, L, B, H]
        self._router_dev = None
        self._shared_dev = None

    def router_dev(self, torch, dev):
        if self._router_dev is None:
            self._router_dev = [torch.from_numpy(self.wr[l].view(np.int16)).to(dev)
                                for l in range(self.cfg.num_layers)]
        return self._router_dev

    def shared_dev(self, torch, dev):
        if self._shared_dev is None:
            self._shared_dev = [tuple(torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in sh)
                                for sh in self.shared]
        return self._shared_dev

    def handle(self, torch, dev, num_slots=None, max_tokens_graph=8, shared=True, set_shared=True, prefetch_n=0):
        from expert_cache_router_gb300 import MoeOffload
        c = self.cfg
        L = c.num_layers
        h = MoeOffload(num_layers=L, num_experts=c.num_experts, top_k=c.top_k, hidden=c.hidden,
                       inter=c.inter, num_slots=c.num_slots if num_slots is None else num_slots,
                       host_w13=[self.w13[l] for l in range(L)], host_w2=[self.w2[l] for l in range(L)],
                       host_s13=[self.s13[l] for l in range(L)], host_s2=[self.s2[l] for l in range(L)],
                       router=self.router_dev(torch, dev), renormalize=c.renormalize,
                       max_tokens_graph=max_tokens_graph, dtype="fp8", shared_expert=shared,
                       prefetch_n=prefetch_n)
        if shared and set_shared:
            for l, (q13, s13, q2, s2) in enumerate(self.shared_dev(torch, dev)):
                h.set_shared_expert(l, q13, q2, s13, s2)
        return h

    def oracle_out(self, t, l, T, shared=True):
        """Oracle routing + FP8 FFN (+ shared expert) of token step t, layer l, batch rows :T."""
        import oracle
        x = self.x[t, l, :T]
        lg = oracle.router_logits(x, self.wr[l])
        ids, w = oracle.topk(lg, self.cfg.top_k, self.cfg.renormalize)
        out_f, out_b = oracle.moe_ffn_fp8(x, ids, w, self.w13[l], self.s13[l], self.w2[l], self.s2[l],
                                          shared=self.shared[l] if shared else None)
        return dict(ids=ids, w=w, out_f32=out_f, out_bf16=out_b)
