// Per-layer LRU slot table on the GPU ("MoE expert offload" page, "How it works").
// The standalone ensure kernel is one CTA of 1024 threads per call (the routine
// itself is in ensure_block.cuh), plus the table audit kernel.
#include <stdint.h>

#include "ensure_block.cuh"
#include "kernels.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(kEnsureThreads)
slot_ensure_kernel(LayerTables tab, const int32_t* __restrict__ ids, int Tk, int E, int S,
                   int32_t* __restrict__ slot_ids, uint32_t* status, unsigned long long expert_bytes) {
  __shared__ EnsureSmem sm;
  ensure_load_table(sm, tab, E, S);
  __syncthreads();
  ensure_call(sm, tab, ids, Tk, E, S, slot_ids, status, expert_bytes);
}

// Consistency audit of one layer's table (and, when given, of the FFN's early-down
// counters, which are zero between calls); sets kDevAuditFailed, never traps.
__global__ void __launch_bounds__(kEnsureThreads)
audit_kernel(LayerTables tab, int E, int S, uint32_t* status, const uint32_t* ffn_sync) {
  __shared__ int bad;
  const int tid = threadIdx.x;
  if (tid == 0) bad = 0;
  __syncthreads();
  const uint32_t clock = *tab.clock;
  int b = 0;
  for (int s = tid; s < S; s += kEnsureThreads) {
    const int e = tab.slot_expert[s];
    if (e >= E || e < -1) b = 1;
    else if (e >= 0 && tab.expert_slot[e] != s) b = 1;
    if (tab.stamp[s] > clock) b = 1;
  }
  for (int e = tid; e < E; e += kEnsureThreads) {
    const int s = tab.expert_slot[e];
    if (s >= S || s < -1) b = 1;
    else if (s >= 0 && tab.slot_expert[s] != e) b = 1;
  }
  const int miss = tab.counts[kCntMiss], inst = tab.counts[kCntInstall];
  const int spill = tab.counts[kCntSpill], distinct = tab.counts[kCntDistinct];
  if (tid == 0) {
    if (miss < 0 || inst < 0 || spill < 0 || inst + spill != miss || miss > distinct ||
        distinct > E || inst > S)
      b = 1;
  }
  // The last prefetch install into this layer: sizes and ids in range.
  const int npf = tab.counts[kCntPrefetch], ncand = tab.counts[kCntCandidates];
  if (tid == 0 && (npf < 0 || npf > S || ncand < 0 || ncand > E || npf > ncand)) b = 1;
  const bool pf_ok = npf >= 0 && npf <= S;
  if (pf_ok) {
    for (int i = tid; i < npf; i += kEnsureThreads) {
      const int e = tab.pf_expert[i], s = tab.pf_slot[i];
      if (s < 0 || s >= S || e < 0 || e >= E) b = 1;
    }
  }
  // Each expert of the last miss list still holds its slot, unless a prefetch
  // install that came after that call took the slot.
  if (inst >= 0 && inst <= S) {
    for (int i = tid; i < inst; i += kEnsureThreads) {
      const int e = tab.miss_expert[i], s = tab.miss_slot[i];
      if (s < 0 || s >= S || e < 0 || e >= E) {
        b = 1;
      } else if (tab.slot_expert[s] != e && clock > 0u) {
        bool taken = false;
        for (int j = 0; pf_ok && j < npf; ++j) taken |= tab.pf_slot[j] == s;
        if (!taken) b = 1;
      }
    }
  }
  if (ffn_sync)
    for (int i = tid; i < kFfnSyncWords; i += kEnsureThreads) b |= ffn_sync[i] != 0u;
  if (b) atomicOr(&bad, 1);
  __syncthreads();
  if (tid == 0 && bad) atomicOr(status, kDevAuditFailed);
}

// Prefetch install of one call as its own launch (router lookahead without the
// in-kernel predictor): predicted ids and logits come from the route kernels.
__global__ void __launch_bounds__(kEnsureThreads, 1)
prefetch_install_kernel(const int32_t* __restrict__ pred_ids, const float* pred_logits, int T, int k, int E,
                        LayerTables tab, int S, int N, unsigned long long bytes) {
  __shared__ EnsureSmem sm;
  __shared__ int pid[kEnsureMax];
  for (int p = threadIdx.x; p < T * k; p += kEnsureThreads) pid[p] = pred_ids[p];
  __syncthreads();
  const int nc = lookahead_candidates_block(sm, pid, pred_logits, T, k, E, sm.es);
  install_block(sm, tab, sm.es, nc, N, E, S, bytes, false);
}

}  // namespace

cudaError_t launch_prefetch_install(const int32_t* pred_ids, const float* pred_logits, int T, int k, int E,
                                    LayerTables tab, int S, int N, unsigned long long bytes, cudaStream_t st) {
  if (T <= 0 || N <= 0) return cudaSuccess;
  if (T * k > kEnsureThreads || E > kEnsureMax || S > kEnsureMax) return cudaErrorInvalidValue;
  prefetch_install_kernel<<<1, kEnsureThreads, 0, st>>>(pred_ids, pred_logits, T, k, E, tab, S, N, bytes);
  return cudaGetLastError();
}

cudaError_t launch_slot_ensure(const EnsureArgs& a, cudaStream_t st) {
  if (a.E > kEnsureMax || a.S > kEnsureMax || a.S < 1) return cudaErrorInvalidValue;
  slot_ensure_kernel<<<1, kEnsureThreads, 0, st>>>(a.tab, a.ids, a.Tk, a.E, a.S, a.slot_ids, a.status,
                                             a.expert_bytes);
  return cudaGetLastError();
}

cudaError_t launch_audit(const LayerTables& tab, int E, int S, uint32_t* status, const uint32_t* ffn_sync,
                         cudaStream_t st) {
  if (E > kEnsureMax || S > kEnsureMax) return cudaErrorInvalidValue;
  audit_kernel<<<1, kEnsureThreads, 0, st>>>(tab, E, S, status, ffn_sync);
  return cudaGetLastError();
}

}  // namespace moe
