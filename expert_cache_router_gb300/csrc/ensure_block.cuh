// Slot-table update of one call as a block-wide device routine, shared by the
// standalone ensure kernel and the fused route+ensure kernel ("MoE expert
// offload" page, "How it works": LRU lookup, least-recently-used slots for
// misses, ids rewritten to slot ids, miss count left in device memory).
//
// Thread e owns expert e and thread s owns slot s. The misses of a call, taken
// in ascending expert id, receive the free slots in ascending key order
// (occupied, stamp, slot index); giving them one at a time to the smallest
// free key, as the sequential rule reads, lands on the same slots because each
// installed slot leaves the free set. Misses beyond the free slots are
// spilled: slot id S + spill index, read from host memory by the FFN.
//
// The table is worked on in shared memory: ensure_load_table copies it in (it
// may run early, while the CTA does other work), ensure_block updates the copy
// and writes the whole table back at the end.
//
// Router-lookahead prefetch install (FreeToken issue #677, "Proposal"): the
// next layer's router run on this layer's input predicts that layer's experts;
// right after this layer's ensure, up to N predicted experts that are not
// resident there are installed into the next layer's table as low-priority
// slots (stamp 0: held, unused, first to be evicted). lookahead_candidates_block
// orders the predicted experts (descending predicted logit) and install_block
// writes the install; both run in the CTA that ran ensure_block, so every
// slot-table write stays in one kernel on the compute stream.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace moe {

constexpr int kEnsureThreads = 1024;
constexpr int kEnsureMax = 1024;  // largest E and S

// Exclusive block-wide prefix sum of one int per thread; returns the total via *total.
static __device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    if (lane < nw) warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int before = warp > 0 ? warp_sums[warp - 1] : 0;
  *total = warp_sums[(blockDim.x >> 5) - 1];
  return before + incl - v;
}

struct EnsureSmem {
  int se[kEnsureMax];        // slot -> expert (-1 empty)
  int es[kEnsureMax];        // expert -> slot (-1 not resident)
  uint32_t st[kEnsureMax];   // slot stamps
  unsigned char present[kEnsureMax];
  unsigned char used[kEnsureMax];
  unsigned char missed[kEnsureMax];  // per expert: missed in this call
  unsigned long long key[kEnsureMax];
  int slot_by_rank[kEnsureMax];
  int spill_marker[kEnsureMax];
  int warp_sums[32];
  int s_hits;
  int s_pf_hits;
  int frozen;                // the table holds a static placement: no installs
  uint32_t clock0;
  unsigned s_bad;
};

// Rank of every free slot's key among sm.key[0..S) (distinct keys; used slots,
// sm.used[s] set, are not ranked), recorded as sm.slot_by_rank[rank] = s for
// ranks below limit. One warp per slot: each lane counts the smaller keys among
// every 32nd slot, the warp adds the counts. Every thread calls it (no barrier).
static __device__ __forceinline__ void rank_free_slots(EnsureSmem& sm, int S, int limit) {
  const int lane = threadIdx.x & 31;
  for (int s = threadIdx.x >> 5; s < S; s += blockDim.x >> 5) {
    if (sm.used[s]) continue;  // the same for the whole warp
    const unsigned long long k0 = sm.key[s];
    int r = 0;
    for (int s2 = lane; s2 < S; s2 += 32) r += (sm.key[s2] < k0);
    r = __reduce_add_sync(0xffffffffu, r);
    if (lane == 0 && r < limit) sm.slot_by_rank[r] = s;
  }
}


// Copy the layer's table into shared memory (no barrier; call before ensure_block
// with a __syncthreads in between).
static __device__ __forceinline__ void ensure_load_table(EnsureSmem& sm, const LayerTables& tab, int E, int S) {
  for (int i = threadIdx.x; i < S; i += blockDim.x) {
    sm.se[i] = tab.slot_expert[i];
    sm.st[i] = tab.stamp[i];
  }
  for (int i = threadIdx.x; i < E; i += blockDim.x) sm.es[i] = tab.expert_slot[i];
  if (threadIdx.x == 0) {
    sm.clock0 = *tab.clock;
    sm.frozen = tab.counts[kCntFrozen];
  }
}

// The whole slot-table update of one call, run by one CTA (every thread must
// call it; at least max(E, S) threads) after ensure_load_table and a barrier.
// ids (global or shared memory) may have been written by this CTA before that
// barrier.
static __device__ void ensure_block(EnsureSmem& sm, LayerTables tab, const int32_t* ids, int Tk, int E, int S,
                                    int32_t* slot_ids, uint32_t* status, unsigned long long expert_bytes) {
  const int tid = threadIdx.x;
  if (tid < E) { sm.present[tid] = 0; sm.missed[tid] = 0; sm.spill_marker[tid] = -1; }
  if (tid < S) sm.used[tid] = 0;
  if (tid == 0) { sm.s_hits = 0; sm.s_pf_hits = 0; sm.s_bad = 0u; }
  __syncthreads();
  for (int p = tid; p < Tk; p += blockDim.x) {
    const int e = ids[p];
    if (e >= 0 && e < E) {
      sm.present[e] = 1;
      atomicAdd(&tab.route_counts[e], 1ull);
    } else {
      sm.s_bad = 1u;
    }
  }
  __syncthreads();
  const uint32_t clock = sm.clock0 + 1u;

  // Hits refresh their stamp and take their slot out of the free set.
  int is_miss = 0;
  if (tid < E && sm.present[tid]) {
    const int s = sm.es[tid];
    if (s >= 0) {
      if (sm.st[s] == 0u) atomicAdd(&sm.s_pf_hits, 1);  // first use of a prefetched slot
      sm.st[s] = clock;
      sm.used[s] = 1;
      atomicAdd(&sm.s_hits, 1);
    } else {
      is_miss = 1;
    }
  }
  int misses = 0;
  const int miss_rank = block_exclusive_scan(is_miss, sm.warp_sums, &misses);  // syncs
  const int hits = sm.s_hits;
  const int free_slots = sm.frozen ? 0 : S - hits;  // a static placement spills every miss

  // Key of every free slot: empty before occupied, then stamp, then index.
  if (tid < S) {
    sm.key[tid] = sm.used[tid] ? ~0ull
                               : ((unsigned long long)(sm.se[tid] >= 0) << 42) |
                                     ((unsigned long long)sm.st[tid] << 10) | (unsigned long long)tid;
  }
  __syncthreads();
  rank_free_slots(sm, S, S);  // ranks of the free slots are 0..free_slots-1
  __syncthreads();

  // Install the first free_slots misses; spill the rest.
  if (is_miss) {
    const int e = tid;
    sm.missed[e] = 1;
    if (miss_rank < free_slots) {
      const int v = sm.slot_by_rank[miss_rank];
      const int old = sm.se[v];
      if (old >= 0) sm.es[old] = -1;
      sm.se[v] = e;
      sm.es[e] = v;
      sm.st[v] = clock;
      tab.miss_expert[miss_rank] = e;
      tab.miss_slot[miss_rank] = v;
    } else {
      const int marker = S + (miss_rank - free_slots);
      tab.miss_expert[miss_rank] = e;
      tab.miss_slot[miss_rank] = marker;
      sm.spill_marker[e] = marker;
    }
  }
  __syncthreads();

  // Rewrite expert ids to slot ids (or spill markers); record which pairs' experts come
  // from host memory in this call (installed or spilled).
  for (int p = tid; p < Tk; p += blockDim.x) {
    const int e = ids[p];
    int s = -1, src = -1;
    if (e >= 0 && e < E) {
      s = sm.es[e];
      if (s < 0) s = sm.spill_marker[e];
      if (sm.missed[e]) src = e;
    }
    slot_ids[p] = s;
    if (p < kMaxCallPairs) tab.pair_src[p] = src;
  }
  // Write the table back.
  if (tid < S) {
    tab.slot_expert[tid] = sm.se[tid];
    tab.stamp[tid] = sm.st[tid];
  }
  if (tid < E) tab.expert_slot[tid] = sm.es[tid];
  if (tid == 0) {
    const int installs = misses < free_slots ? misses : free_slots;
    const int spills = misses - installs;
    *tab.clock = clock;
    tab.counts[kCntMiss] = misses;
    tab.counts[kCntSpill] = spills;
    tab.counts[kCntInstall] = installs;
    tab.counts[kCntDistinct] = hits + misses;
    // counters by atomic adds whose results are not used: no read round trip
    atomicAdd(&tab.stats[kStatCalls], 1ull);
    atomicAdd(&tab.stats[kStatHits], (unsigned long long)hits);
    atomicAdd(&tab.stats[kStatMisses], (unsigned long long)misses);
    atomicAdd(&tab.stats[kStatSpills], (unsigned long long)spills);
    atomicAdd(&tab.stats[kStatBytesCopied], (unsigned long long)installs * expert_bytes);
    atomicAdd(&tab.stats[kStatPrefetchHits], (unsigned long long)sm.s_pf_hits);
    if (sm.s_bad) atomicOr(status, kDevBadExpertId);
  }
}

// The same update by one warp, for calls of at most kEnsureWarpPairs pairs on
// at most kEnsureWarpSlots slots: lane p holds pair p, the lowest lane of each
// expert stands for it, and the block's barriers become warp votes. Hits,
// misses (ranked by expert id), installs (the i-th smallest free key for the
// i-th miss, taken one at a time by a warp-wide minimum) and spills follow the
// rule above, so tables, slot ids, miss lists and counts are those of
// ensure_block. Every lane of one warp calls it, after ensure_load_table and a
// barrier; the rest of the CTA may leave.
constexpr int kEnsureWarpPairs = 32;
constexpr int kEnsureWarpSlots = 64;

static __device__ __forceinline__ bool ensure_fits_warp(int Tk, int S) {
  return Tk <= kEnsureWarpPairs && S <= kEnsureWarpSlots;
}

static __device__ __forceinline__ unsigned long long free_slot_key(const EnsureSmem& sm, int s) {
  return ((unsigned long long)(sm.se[s] >= 0) << 42) | ((unsigned long long)sm.st[s] << 10) |
         (unsigned long long)s;
}

static __device__ void ensure_warp(EnsureSmem& sm, LayerTables tab, const int32_t* ids, int Tk, int E, int S,
                                   int32_t* slot_ids, uint32_t* status, unsigned long long expert_bytes) {
  constexpr unsigned kAll = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const uint32_t clock = sm.clock0 + 1u;
  if (lane < S) sm.used[lane] = 0;
  if (lane + 32 < S) sm.used[lane + 32] = 0;
  const int e = lane < Tk ? ids[lane] : -1;
  const bool valid = lane < Tk && e >= 0 && e < E;
  const bool bad = __any_sync(kAll, lane < Tk && !valid);
  if (valid) atomicAdd(&tab.route_counts[e], 1ull);
  // lanes of the same expert (invalid lanes each on their own)
  const unsigned same = __match_any_sync(kAll, valid ? e : -1 - lane);
  const int lead = __ffs(same) - 1;
  const bool first = valid && lead == lane;
  const int s0 = first ? sm.es[e] : -1;
  const bool hit = first && s0 >= 0;
  const bool miss = first && s0 < 0;
  const bool pf_hit = hit && sm.st[s0] == 0u;  // first use of a prefetched slot
  __syncwarp();
  if (hit) {
    sm.st[s0] = clock;
    sm.used[s0] = 1;
  }
  const unsigned miss_mask = __ballot_sync(kAll, miss);
  const int hits = __popc(__ballot_sync(kAll, hit));
  const int pf_hits = __popc(__ballot_sync(kAll, pf_hit));
  const int misses = __popc(miss_mask);
  int miss_rank = 0;  // missed experts with a smaller id
  for (unsigned m = miss_mask; m; m &= m - 1) {
    const int eq = __shfl_sync(kAll, e, __ffs(m) - 1);
    miss_rank += eq < e;
  }
  const int free_slots = sm.frozen ? 0 : S - hits;  // a static placement spills every miss
  const int installs = misses < free_slots ? misses : free_slots;
  __syncwarp();
  if (installs > 0) {
    unsigned long long k0 = (lane < S && !sm.used[lane]) ? free_slot_key(sm, lane) : ~0ull;
    unsigned long long k1 = (lane + 32 < S && !sm.used[lane + 32]) ? free_slot_key(sm, lane + 32) : ~0ull;
    for (int r = 0; r < installs; ++r) {
      const unsigned long long mk = k0 < k1 ? k0 : k1;
      const uint32_t hi = __reduce_min_sync(kAll, (uint32_t)(mk >> 32));
      const uint32_t lo = __reduce_min_sync(kAll, (uint32_t)(mk >> 32) == hi ? (uint32_t)mk : ~0u);
      const unsigned long long win = ((unsigned long long)hi << 32) | lo;
      if (k0 == win) k0 = ~0ull;
      if (k1 == win) k1 = ~0ull;
      if (miss && miss_rank == r) {
        const int v = (int)(lo & 1023u);
        const int old = sm.se[v];
        if (old >= 0) sm.es[old] = -1;
        sm.se[v] = e;
        sm.es[e] = v;
        sm.st[v] = clock;
        tab.miss_expert[r] = e;
        tab.miss_slot[r] = v;
      }
      __syncwarp();
    }
  }
  int marker = -1;
  if (miss && miss_rank >= free_slots) {
    marker = S + (miss_rank - free_slots);
    tab.miss_expert[miss_rank] = e;
    tab.miss_slot[miss_rank] = marker;
  }
  // Expert ids to slot ids (or spill markers), and the pairs read from host memory.
  const int g_marker = __shfl_sync(kAll, marker, lead);
  const int g_missed = __shfl_sync(kAll, (int)miss, lead);
  __syncwarp();
  if (lane < Tk) {
    int s = -1, src = -1;
    if (valid) {
      s = sm.es[e];
      if (s < 0) s = g_marker;
      if (g_missed) src = e;
    }
    slot_ids[lane] = s;
    tab.pair_src[lane] = src;
  }
  // Write the table back.
  for (int i = lane; i < S; i += 32) {
    tab.slot_expert[i] = sm.se[i];
    tab.stamp[i] = sm.st[i];
  }
  for (int i = lane; i < E; i += 32) tab.expert_slot[i] = sm.es[i];
  if (lane == 0) {
    const int spills = misses - installs;
    *tab.clock = clock;
    tab.counts[kCntMiss] = misses;
    tab.counts[kCntSpill] = spills;
    tab.counts[kCntInstall] = installs;
    tab.counts[kCntDistinct] = hits + misses;
    atomicAdd(&tab.stats[kStatCalls], 1ull);
    atomicAdd(&tab.stats[kStatHits], (unsigned long long)hits);
    atomicAdd(&tab.stats[kStatMisses], (unsigned long long)misses);
    atomicAdd(&tab.stats[kStatSpills], (unsigned long long)spills);
    atomicAdd(&tab.stats[kStatBytesCopied], (unsigned long long)installs * expert_bytes);
    atomicAdd(&tab.stats[kStatPrefetchHits], (unsigned long long)pf_hits);
    if (bad) atomicOr(status, kDevBadExpertId);
  }
}

// The update of one call by the whole CTA (every thread calls it): one warp when
// the call fits ensure_warp, else ensure_block.
static __device__ void ensure_call(EnsureSmem& sm, LayerTables tab, const int32_t* ids, int Tk, int E, int S,
                                   int32_t* slot_ids, uint32_t* status, unsigned long long expert_bytes) {
  if (ensure_fits_warp(Tk, S)) {
    if (threadIdx.x < 32) ensure_warp(sm, tab, ids, Tk, E, S, slot_ids, status, expert_bytes);
  } else {
    ensure_block(sm, tab, ids, Tk, E, S, slot_ids, status, expert_bytes);
  }
}

// Prefetch candidates of a call from the predictor's per-token top-k: the
// distinct predicted experts in descending order of their largest predicted
// logit over the tokens that chose them, equal logits by ascending expert id.
// pid [T*k] predicted ids (T*k <= blockDim.x), plog [T][E] predicted logits
// (shared or global memory, written before the caller's last barrier). Writes
// cand[0..n) and returns n. Uses sm.used and sm.key as scratch. Every thread
// calls it.
static __device__ int lookahead_candidates_block(EnsureSmem& sm, const int* pid, const float* plog, int T, int k,
                                                 int E, int* cand) {
  const int n = T * k;
  const int p = threadIdx.x;
  float* val = reinterpret_cast<float*>(sm.key);
  int e = -1;
  float v = -INFINITY;
  if (p < n) {
    e = pid[p];
    if (e >= 0 && e < E) {
      v = plog[(p / k) * E + e];
      if (v != v) v = -INFINITY;
    }
    val[p] = v;
  }
  __syncthreads();
  // pair p stands for its expert when no other pair of that expert has a larger
  // logit (or an equal one at a lower pair index)
  bool rep = p < n && e >= 0 && e < E;
  for (int q = 0; q < n && rep; ++q)
    if (q != p && pid[q] == e && (val[q] > v || (val[q] == v && q < p))) rep = false;
  if (p < n) sm.used[p] = rep ? 1 : 0;
  const int count = __syncthreads_count(rep);
  if (rep) {
    int r = 0;
    for (int q = 0; q < n; ++q)
      if (sm.used[q] && (val[q] > v || (val[q] == v && pid[q] < e))) ++r;
    cand[r] = e;
  }
  __syncthreads();
  return count;
}

// Install of the first N non-resident candidates cand[0..ncand) (ncand <= E,
// ncand <= blockDim.x) into layer table tab at stamp 0, without advancing its
// clock: residency is judged before the install; slots holding a candidate and
// slots this install fills are never victims; each install takes the free slot
// with the smallest key (occupied?, stamp, index), which is the i-th smallest
// key for the i-th install. Records the install list, the candidates and the
// counts. With loaded, sm.se, sm.st and sm.es already hold tab (ensure_load_table
// before a barrier) and cand must not alias sm.es; otherwise the slot entries
// are read here and cand may be sm.es. cand must not alias sm.se, sm.st, sm.used,
// sm.key, sm.slot_by_rank or sm.spill_marker. Every thread calls it.
static __device__ void install_block(EnsureSmem& sm, LayerTables tab, const int* cand, int ncand, int N, int E,
                                     int S, unsigned long long expert_bytes, bool loaded) {
  const int tid = threadIdx.x;
  if (!loaded && tid == 0) sm.frozen = tab.counts[kCntFrozen];
  __syncthreads();
  if (sm.frozen) N = 0;  // a static placement takes no prefetch installs
  if (tid < S) {
    if (!loaded) {
      sm.se[tid] = tab.slot_expert[tid];
      sm.st[tid] = tab.stamp[tid];
    }
    sm.used[tid] = 0;
  }
  __syncthreads();
  int nonres = 0;
  if (tid < ncand) {
    const int e = cand[tid];
    const int s = (e >= 0 && e < E) ? (loaded ? sm.es[e] : tab.expert_slot[e]) : -2;
    if (s >= 0 && s < S) sm.used[s] = 1;  // resident candidates keep their slots
    nonres = s == -1;
  }
  int total = 0;
  const int pos = block_exclusive_scan(nonres, sm.warp_sums, &total);  // syncs
  if (nonres && pos < N) sm.spill_marker[pos] = cand[tid];
  const int ntodo = total < N ? total : N;
  if (tid < S)
    sm.key[tid] = sm.used[tid] ? ~0ull
                               : ((unsigned long long)(sm.se[tid] >= 0) << 42) |
                                     ((unsigned long long)sm.st[tid] << 10) | (unsigned long long)tid;
  const int taken = __syncthreads_count(tid < S && sm.used[tid]);
  const int nopen = S - taken;
  const int ninst = ntodo < nopen ? ntodo : nopen;
  rank_free_slots(sm, S, ninst);
  __syncthreads();
  if (tid < ninst) {
    const int e = sm.spill_marker[tid];
    const int v = sm.slot_by_rank[tid];
    const int old = sm.se[v];
    if (old >= 0) tab.expert_slot[old] = -1;
    tab.slot_expert[v] = e;
    tab.expert_slot[e] = v;
    tab.stamp[v] = 0u;
    tab.pf_expert[tid] = e;
    tab.pf_slot[tid] = v;
  }
  if (tid < ncand) tab.pf_cand[tid] = cand[tid];
  if (tid == 0) {
    tab.counts[kCntPrefetch] = ninst;
    tab.counts[kCntCandidates] = ncand;
    atomicAdd(&tab.stats[kStatPrefetchInstalls], (unsigned long long)ninst);
    atomicAdd(&tab.stats[kStatPrefetchBytes], (unsigned long long)ninst * expert_bytes);
  }
  __syncthreads();
}

}  // namespace moe
