// Router: logits = x . W_r^T (fp32 accumulation), top-k (descending, equal
// logits -> lower expert id), softmax weights over the k chosen (renormalised)
// or over all E. Decode-sized calls are one launch: every CTA computes the
// logits of 8 experts for a chunk of tokens, and the CTA that finishes last
// runs the top-k ("MoE expert offload" page, "How it works": the routed experts
// of each MoE call).
#include <cooperative_groups.h>

#include <climits>
#include <float.h>
#include <math.h>

#include "ensure_block.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kTokChunk = 8;  // most tokens per CTA (grid.y chunks)
constexpr int kSmemMax = 200 * 1024;  // leaves room for static shared memory under the 227 KB opt-in
constexpr int kMaxK = 16;

// x chunk [kTokChunk][H] is staged in shared memory as fp32.
__global__ void __launch_bounds__(kWarps * 32)
route_logits_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr, int T, int E,
                    int H, int tok_chunk, float* __restrict__ logits, int fuse_topk, int k,
                    int renorm, int32_t* __restrict__ ids, float* __restrict__ w, unsigned* done);

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

template <bool kShared>
__device__ __forceinline__ float load_logit(const float* lg, int e) {
  if constexpr (kShared) return lg[e];
  else return __ldcg(lg + e);
}

// One warp: top-k of one row of logits (in shared memory, or in global memory
// read through L2), weights, write out.
template <bool kShared = false>
__device__ void topk_row_warp(const float* lg, int E, int k, int renorm, int32_t* ids_out,
                              float* w_out) {
  const int lane = threadIdx.x & 31;
  int chosen[kMaxK];
  float chosen_v[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    chosen[j] = -1;
    chosen_v[j] = -INFINITY;
  }
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    if (j < k) {
      float bv = -INFINITY;
      int bi = INT_MAX;
      for (int e = lane; e < E; e += 32) {
        float v = load_logit<kShared>(lg, e);
        if (v != v) v = -INFINITY;  // NaN ranks last
        bool taken = false;
#pragma unroll
        for (int q = 0; q < kMaxK; ++q) taken |= (q < j) && (chosen[q] == e);
        if (!taken && better(v, e, bv, bi)) {
          bv = v;
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      chosen[j] = bi;
      chosen_v[j] = bv;
    }
  }
  const float lmax = chosen_v[0];
  float denom = 0.0f;
  if (renorm) {
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < k) denom += expf(chosen_v[j] - lmax);
  } else {
    float part = 0.0f;
    for (int e = lane; e < E; e += 32) {
      float v = load_logit<kShared>(lg, e);
      if (v != v) v = -INFINITY;
      part += expf(v - lmax);
    }
    denom = warp_sum(part);
  }
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k) {
        ids_out[j] = chosen[j];
        w_out[j] = expf(chosen_v[j] - lmax) / denom;
      }
    }
  }
}

__global__ void __launch_bounds__(kWarps * 32)
route_logits_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr, int T, int E,
                    int H, int tok_chunk, float* __restrict__ logits, int fuse_topk, int k,
                    int renorm, int32_t* __restrict__ ids, float* __restrict__ w, unsigned* done) {
  extern __shared__ float xs[];  // [tok_chunk][H], tok_chunk <= kTokChunk
  const int t0 = blockIdx.y * tok_chunk;
  const int nt = min(tok_chunk, T - t0);
  const int h8 = H >> 3;
  for (int i = threadIdx.x; i < nt * h8; i += blockDim.x) {
    const int t = i / h8, c = i - t * h8;
    const uint4 v = *reinterpret_cast<const uint4*>(x + (size_t)(t0 + t) * H + c * 8);
    float* d = xs + t * H + c * 8;
    d[0] = bf16lo(v.x); d[1] = bf16hi(v.x); d[2] = bf16lo(v.y); d[3] = bf16hi(v.y);
    d[4] = bf16lo(v.z); d[5] = bf16hi(v.z); d[6] = bf16lo(v.w); d[7] = bf16hi(v.w);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kWarps + warp;
  if (e < E) {
    float acc[kTokChunk];
#pragma unroll
    for (int t = 0; t < kTokChunk; ++t) acc[t] = 0.0f;
    const uint16_t* row = wr + (size_t)e * H;
    for (int c = lane * 8; c < H; c += 256) {
      const uint4 wv = ld_stream(row + c);
#pragma unroll
      for (int t = 0; t < kTokChunk; ++t)
        if (t < nt) acc[t] = dot8(wv, xs + t * H + c, acc[t]);
    }
#pragma unroll
    for (int t = 0; t < kTokChunk; ++t) {
      const float s = warp_sum(acc[t]);
      if (lane == 0 && t < nt) logits[(size_t)(t0 + t) * E + e] = s;
    }
  }
  if (!fuse_topk) return;
  // The CTA that finishes last ranks every token (logits are read through L2).
  __shared__ unsigned s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned total = gridDim.x * gridDim.y;
    s_last = (atomicAdd(done, 1u) == total - 1u);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int t = warp; t < T; t += kWarps)
    topk_row_warp(logits + (size_t)t * E, E, k, renorm, ids + (size_t)t * k, w + (size_t)t * k);
  if (threadIdx.x == 0) *done = 0u;
}

__global__ void __launch_bounds__(kWarps * 32)
topk_kernel(const float* __restrict__ logits, int T, int E, int k, int renorm,
            int32_t* __restrict__ ids, float* __restrict__ w) {
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (t < T) topk_row_warp(logits + (size_t)t * E, E, k, renorm, ids + (size_t)t * k, w + (size_t)t * k);
}

// Fused decode head: logits with one warp per expert (32 experts per CTA),
// then the last CTA to finish ranks every token and updates the slot table.
// Every CTA copies the layer's slot table into shared memory first (a few KB),
// so the last one starts its update without another round trip. x rows are
// read through L1; each warp streams its weight row with kRowUnroll
// independent 16-byte loads in flight per lane. Each logit is accumulated in
// the same order as route_logits_kernel.
constexpr int kRowUnroll = 8;
constexpr int kHeadSmemLogits = 4096;  // logits staged in shared memory when T*E fits (static smem < 48 KB)

template <int TC>
__global__ void __launch_bounds__(kEnsureThreads, 1)
route_ensure_kernel(RouteEnsureArgs a) {
  __shared__ EnsureSmem sm;
  __shared__ float lsm[kHeadSmemLogits];
  __shared__ unsigned s_last;
  const RouteArgs& r = a.r;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * (kEnsureThreads / 32) + warp;
  const int H = r.H, E = r.E, T = r.T;
  // Nothing here depends on the preceding kernel yet: copy the slot table and
  // pull this warp's router row into L2, then wait for that kernel.
  ensure_load_table(sm, a.tab, E, a.S);
  const uint16_t* row = r.wr + (size_t)(e < E ? e : 0) * H;
  if (e < E)
    for (int c = lane * 64; c < H; c += 32 * 64)  // one prefetch per 128-byte line
      asm volatile("prefetch.global.L2 [%0];" ::"l"(row + c));
  pdl_wait();
  pdl_trigger();
  if (e < E) {
    for (int t0 = 0; t0 < T; t0 += TC) {
      const int nt = min(TC, T - t0);
      float acc[TC];
#pragma unroll
      for (int t = 0; t < TC; ++t) acc[t] = 0.0f;
      for (int c0 = lane * 8; c0 < H; c0 += 256 * kRowUnroll) {
        uint4 wv[kRowUnroll];
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
          const int c = c0 + 256 * u;
          wv[u] = c < H ? ld_stream(row + c) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
          const int c = c0 + 256 * u;
          if (c < H) {
#pragma unroll
            for (int t = 0; t < TC; ++t) {
              if (t < nt) {
                const uint4 xv = __ldg(reinterpret_cast<const uint4*>(r.x + (size_t)(t0 + t) * H + c));
                const float xf[8] = {bf16lo(xv.x), bf16hi(xv.x), bf16lo(xv.y), bf16hi(xv.y),
                                     bf16lo(xv.z), bf16hi(xv.z), bf16lo(xv.w), bf16hi(xv.w)};
                acc[t] = dot8(wv[u], xf, acc[t]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < TC; ++t) {
        const float sv = warp_sum(acc[t]);
        if (lane == 0 && t < nt) r.logits[(size_t)(t0 + t) * E + e] = sv;
      }
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(r.done, 1u) == gridDim.x - 1u);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // Top-k of every token as a block-wide rank: each candidate counts the logits
  // that beat it (larger, or equal with a lower expert id, NaN ranking last).
  // This is the rule topk_row_warp applies one pick at a time, so the same
  // experts come out in the same order; the weights are computed with the same
  // operations in the same order.
  const bool staged = T * E <= kHeadSmemLogits;
  if (staged) {
    for (int i = threadIdx.x; i < T * E; i += kEnsureThreads) lsm[i] = __ldcg(r.logits + i);
    __syncthreads();
  }
  int* sel_id = sm.slot_by_rank;                        // free until ensure_block runs
  float* sel_v = reinterpret_cast<float*>(sm.key);
  const int k = r.k;
  for (int idx = threadIdx.x; idx < T * E; idx += kEnsureThreads) {
    const int t = idx / E, e = idx - t * E;
    const float* row = staged ? lsm + (size_t)t * E : r.logits + (size_t)t * E;
    float v = staged ? row[e] : __ldcg(row + e);
    if (v != v) v = -INFINITY;
    int rank = 0;
    for (int e2 = 0; e2 < E; ++e2) {
      float v2 = staged ? row[e2] : __ldcg(row + e2);
      if (v2 != v2) v2 = -INFINITY;
      rank += (v2 > v) || (v2 == v && e2 < e);
    }
    if (rank < k) {
      sel_id[t * k + rank] = e;
      sel_v[t * k + rank] = v;
    }
  }
  __syncthreads();
  for (int t = warp; t < T; t += kEnsureThreads / 32) {
    const float* row = staged ? lsm + (size_t)t * E : r.logits + (size_t)t * E;
    const float lmax = sel_v[t * k];
    float denom = 0.0f;
    if (r.renorm) {
      for (int j = 0; j < k; ++j) denom += expf(sel_v[t * k + j] - lmax);
    } else {
      float part = 0.0f;
      for (int e = lane; e < E; e += 32) {
        float v = staged ? row[e] : __ldcg(row + e);
        if (v != v) v = -INFINITY;
        part += expf(v - lmax);
      }
      denom = warp_sum(part);
    }
    if (lane == 0) {
      for (int j = 0; j < k; ++j) {
        r.ids[(size_t)t * k + j] = sel_id[t * k + j];
        r.w[(size_t)t * k + j] = expf(sel_v[t * k + j] - lmax) / denom;
      }
    }
  }
  __syncthreads();
  ensure_block(sm, a.tab, r.ids, T * r.k, E, a.S, a.slot_ids, a.status, a.expert_bytes);
  if (threadIdx.x == 0) *r.done = 0u;
}

// Cluster variant of the fused head (E <= 32 * kClusterMaxCtas, T*E <=
// kClusterMaxLogits): one thread-block cluster, one CTA per 32 experts. Each
// warp stores its logits straight into CTA 0's shared memory (distributed
// shared memory: no global round trip, fence or counter); after one cluster
// barrier CTA 0 takes each token's top-k (topk_rows_block) and updates the slot
// table while the other CTAs exit. Same picks, weights and table as the other
// head kernels.
//
// With the router lookahead on (a.pf_n > 0, at least two CTAs), each warp also
// dots the next layer's router row of its expert with the same x (the
// predictor) and stores it into CTA 1's shared memory, and CTA 1 does the rest
// of the lookahead while CTA 0 does the demand side: it copies the next layer's
// table into its shared memory before the dependency wait, takes the predicted
// top-k (the same rule as the demand top-k), orders the candidates and installs
// them (lookahead_candidates_block, install_block). The two CTAs write
// different layers' tables. Dynamic shared memory: x of one token chunk [TC][H]
// (read once per CTA, not once per warp), predicted ids [T][k], candidates [T][k].
constexpr int kClusterMaxCtas = 8;
constexpr int kClusterMaxLogits = 2048;

// Top-k of rows [T][E] of logits in shared memory with the rule of
// topk_row_warp and route_ensure_kernel (larger logit first, equal logits by
// lower expert id, NaN ranking as -inf), one warp per token. Each (logit,
// expert) pair becomes one 64-bit key whose unsigned order is that rule: the
// logit's bits mapped to an order-preserving unsigned integer (NaN read as
// -inf, -0 as +0) in the high word, the complement of the expert id in the low
// word. Lane i holds the keys of experts i*M .. i*M+M-1 (0 beyond E, below
// every real key) and sorts them in registers; then a butterfly over the lanes
// keeps, at every step, the M largest keys of the two lists it joins
// (elementwise max of one list and the other reversed is a bitonic sequence
// holding exactly those, which a bitonic merge sorts). After log2 of the lanes
// in use every lane holds the row's M largest keys in descending order, so pick
// j is the j-th list entry.
__device__ __forceinline__ unsigned long long rank_key(float v, int e) {
  if (v != v) v = -INFINITY;
  if (v == 0.0f) v = 0.0f;  // -0 ranks with +0
  uint32_t b = __float_as_uint(v);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)b << 32) | (unsigned long long)(~(uint32_t)e);
}
__device__ __forceinline__ float key_value(unsigned long long key) {
  const uint32_t b = (uint32_t)(key >> 32);
  return __uint_as_float((b & 0x80000000u) ? (b & 0x7fffffffu) : ~b);
}
__device__ __forceinline__ int key_expert(unsigned long long key) { return (int)(~(uint32_t)key); }

template <int M>
__device__ __forceinline__ void sort_desc(unsigned long long (&a)[M]) {
#pragma unroll
  for (int size = 2; size <= M; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int i = 0; i < M; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          const unsigned long long x = a[i], y = a[j];
          const bool sw = (i & size) == 0 ? (x < y) : (x > y);
          a[i] = sw ? y : x;
          a[j] = sw ? x : y;
        }
      }
    }
  }
}

// Both lanes of a butterfly pair end with the M largest keys of their two lists, descending.
template <int M>
__device__ __forceinline__ void keep_top_of_pair(unsigned long long (&a)[M], int s) {
  unsigned long long b[M];
#pragma unroll
  for (int i = 0; i < M; ++i) {
    const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)a[i], s);
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(a[i] >> 32), s);
    b[i] = ((unsigned long long)hi << 32) | lo;
  }
#pragma unroll
  for (int i = 0; i < M; ++i) a[i] = a[i] > b[M - 1 - i] ? a[i] : b[M - 1 - i];
#pragma unroll
  for (int stride = M >> 1; stride > 0; stride >>= 1) {
#pragma unroll
    for (int i = 0; i < M; ++i) {
      const int j = i ^ stride;
      if (j > i && a[i] < a[j]) {
        const unsigned long long x = a[i];
        a[i] = a[j];
        a[j] = x;
      }
    }
  }
}

// The warp's top-k (k <= M) of one row lg[0..E) (shared memory), E <= 32 * M.
// Lane j < k returns the key of pick j. The butterfly runs over at least k
// lanes, so that lanes 0..k-1 all hold the final list.
template <int M>
__device__ __forceinline__ unsigned long long warp_topk_row(const float* lg, int E, int k) {
  const int lane = threadIdx.x & 31;
  unsigned long long a[M];
#pragma unroll
  for (int q = 0; q < M; ++q) {
    const int e = lane * M + q;
    a[q] = e < E ? rank_key(lg[e], e) : 0ull;
  }
  sort_desc<M>(a);
  const int lanes = (E + M - 1) / M;
  for (int s = 1; s < lanes || s < k; s <<= 1) keep_top_of_pair<M>(a, s);
  unsigned long long mine = 0ull;
#pragma unroll
  for (int q = 0; q < M; ++q)
    if (q == lane) mine = a[q];
  return mine;
}

// The same picks for k > 8 (E <= 256): k rounds of a warp-wide maximum of the
// keys not yet taken (lane i holds experts i, i+32, ...), which needs fewer
// registers than a 16-entry list. Lane j < k returns the key of pick j.
__device__ __forceinline__ unsigned long long warp_topk_rounds(const float* lg, int E, int k) {
  const int lane = threadIdx.x & 31;
  unsigned long long v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < E ? rank_key(lg[e], e) : 0ull;
  }
  unsigned taken = 0u;
  unsigned long long mine = 0ull;
  for (int r = 0; r < k; ++r) {
    unsigned long long best = 0ull;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (!(taken >> j & 1u) && v[j] > best) best = v[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)best, o);
      const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(best >> 32), o);
      const unsigned long long b = ((unsigned long long)hi << 32) | lo;
      best = b > best ? b : best;
    }
    const int e = key_expert(best);
    if ((e & 31) == lane) taken |= 1u << (e >> 5);
    if (r == lane) mine = best;
  }
  return mine;
}

// Top-k of every token of lg [T][E] (shared memory), one warp per token:
// ids[t*k + j] (and vals, when given) receive pick j. Every thread calls it;
// E <= 256, k <= 16.
__device__ __forceinline__ void topk_rows_warps(const float* lg, int T, int E, int k, int* ids, float* vals) {
  const int lane = threadIdx.x & 31;
  const bool small = k <= 8;
  for (int t = threadIdx.x >> 5; t < T; t += blockDim.x >> 5) {
    const unsigned long long key = small ? warp_topk_row<8>(lg + t * E, E, k) : warp_topk_rounds(lg + t * E, E, k);
    if (lane < k) {
      ids[t * k + lane] = key_expert(key);
      if (vals) vals[t * k + lane] = key_value(key);
    }
  }
}

template <int TC>
__global__ void __launch_bounds__(kEnsureThreads, 1)
route_ensure_cluster_kernel(RouteEnsureArgs a) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ EnsureSmem sm;
  __shared__ float lall[kClusterMaxLogits];  // CTA 0: every logit [T][E]; CTA 1: every predicted logit
  extern __shared__ uint4 dyn[];
  const RouteArgs& r = a.r;
  const unsigned crank = cluster.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = (int)crank * 32 + warp;
  const int H = r.H, E = r.E, T = r.T, k = r.k;
  const bool pf = a.pf_n > 0;
  const int tc = T < TC ? T : TC;
  uint16_t* xs = reinterpret_cast<uint16_t*>(dyn);                  // [tc][H] bf16: this chunk's x
  int* ids_s = reinterpret_cast<int*>(xs + (size_t)tc * H);         // [T][k] routed ids (CTA 0)
  int* pid = ids_s + T * k;                                         // [T][k] predicted ids (CTA 1)
  int* cand = pid + T * k;                                          // [T][k] candidates (CTA 1)
  // Every CTA must have started before another writes into its shared memory:
  // arrive now, wait just before the first remote store.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  if (crank == 0) ensure_load_table(sm, a.tab, E, a.S);
  if (pf && crank == 1) ensure_load_table(sm, a.tab_next, E, a.S);
  const uint16_t* row = r.wr + (size_t)(e < E ? e : 0) * H;
  const uint16_t* prow = pf ? a.wr_next + (size_t)(e < E ? e : 0) * H : row;
  if (e < E) {
    for (int c = lane * 64; c < H; c += 32 * 64) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + c));
    if (pf)
      for (int c = lane * 64; c < H; c += 32 * 64) asm volatile("prefetch.global.L2 [%0];" ::"l"(prow + c));
  }
  pdl_wait();
  pdl_trigger();
  float* to0 = cluster.map_shared_rank(lall, 0);
  float* to1 = cluster.map_shared_rank(lall, pf ? 1 : 0);
  bool waited = false;
  const int h8 = H >> 3;
  for (int t0 = 0; t0 < T; t0 += TC) {
    const int nt = min(TC, T - t0);
    // x rows of this chunk, read once per CTA into shared memory
    __syncthreads();
    for (int i = threadIdx.x; i < nt * h8; i += kEnsureThreads)
      dyn[i] = __ldg(reinterpret_cast<const uint4*>(r.x + (size_t)t0 * H) + i);
    __syncthreads();
    for (int pass = 0; pass < (pf ? 2 : 1) && e < E; ++pass) {
      const uint16_t* wrow = pass ? prow : row;
      float* dst = pass ? to1 : to0;
      float acc[TC];
#pragma unroll
      for (int t = 0; t < TC; ++t) acc[t] = 0.0f;
      for (int c0 = lane * 8; c0 < H; c0 += 256 * kRowUnroll) {
        uint4 wv[kRowUnroll];
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
          const int c = c0 + 256 * u;
          wv[u] = c < H ? ld_stream(wrow + c) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
          const int c = c0 + 256 * u;
          if (c < H) {
#pragma unroll
            for (int t = 0; t < TC; ++t) {
              if (t < nt) {
                const uint4 xv = *reinterpret_cast<const uint4*>(xs + (size_t)t * H + c);
                const float xf[8] = {bf16lo(xv.x), bf16hi(xv.x), bf16lo(xv.y), bf16hi(xv.y),
                                     bf16lo(xv.z), bf16hi(xv.z), bf16lo(xv.w), bf16hi(xv.w)};
                acc[t] = dot8(wv[u], xf, acc[t]);
              }
            }
          }
        }
      }
      float sums[TC];
#pragma unroll
      for (int t = 0; t < TC; ++t) sums[t] = warp_sum(acc[t]);
      if (!waited) {
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        waited = true;
      }
      if (lane == 0) {
#pragma unroll
        for (int t = 0; t < TC; ++t)
          if (t < nt) dst[(t0 + t) * E + e] = sums[t];
      }
    }
  }
  if (!waited) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  cluster.sync();  // every logit is in CTA 0's (and predicted ones in CTA 1's) shared memory
  if (pf && crank == 1) {
    // Lookahead into the next layer: predicted top-k, candidates, install.
    topk_rows_warps(lall, T, E, k, pid, nullptr);
    __syncthreads();
    const int nc = lookahead_candidates_block(sm, pid, lall, T, k, E, cand);
    install_block(sm, a.tab_next, cand, nc, a.pf_n, E, a.S, a.pf_bytes, true);
    return;
  }
  if (crank != 0) return;

  // Each token's top-k and weights in one warp; the picks go to the caller's ids
  // and weights and, for the slot update, to shared memory.
  const bool small = k <= 8;
  for (int t = warp; t < T; t += kEnsureThreads / 32) {
    const float* row = lall + t * E;
    const unsigned long long key = small ? warp_topk_row<8>(row, E, k) : warp_topk_rounds(row, E, k);
    const float v = key_value(key);
    const float lmax = __shfl_sync(0xffffffffu, v, 0);
    const float ej = lane < k ? expf(v - lmax) : 0.0f;
    float denom = 0.0f;
    if (r.renorm) {
      for (int j = 0; j < k; ++j) denom += __shfl_sync(0xffffffffu, ej, j);
    } else {
      float part = 0.0f;
      for (int q = lane; q < E; q += 32) {
        float lv = row[q];
        if (lv != lv) lv = -INFINITY;
        part += expf(lv - lmax);
      }
      denom = warp_sum(part);
    }
    if (lane < k) {
      const int e = key_expert(key);
      r.ids[(size_t)t * k + lane] = e;
      r.w[(size_t)t * k + lane] = ej / denom;
      ids_s[t * k + lane] = e;
    }
  }
  __syncthreads();
  ensure_block(sm, a.tab, ids_s, T * k, E, a.S, a.slot_ids, a.status, a.expert_bytes);
}

}  // namespace

// Dynamic shared memory of the cluster head: x of one token chunk [TC][H] bf16,
// then with the lookahead on predicted ids and candidates [T][k] each.
constexpr int kHeadPredSmemMax = kTokChunk * 8192 * 2 + 3 * 1024 * 4;

cudaError_t route_init_attributes() {
  cudaError_t e = cudaFuncSetAttribute(route_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemMax);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(route_ensure_cluster_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kHeadPredSmemMax);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(route_ensure_cluster_kernel<kTokChunk>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kHeadPredSmemMax);
  return e;
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  const int tok_chunk = min(kTokChunk, kSmemMax / (a.H * (int)sizeof(float)));
  if (tok_chunk < 1) return cudaErrorInvalidValue;
  const size_t smem = (size_t)tok_chunk * a.H * sizeof(float);
  const int fuse = a.T <= kRouteFuseT;
  dim3 grid((a.E + kWarps - 1) / kWarps, (a.T + tok_chunk - 1) / tok_chunk);
  route_logits_kernel<<<grid, kWarps * 32, smem, st>>>(a.x, a.wr, a.T, a.E, a.H, tok_chunk, a.logits,
                                                       fuse, a.k, a.renorm, a.ids, a.w, a.done);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || fuse) return e;
  topk_kernel<<<(a.T + kWarps - 1) / kWarps, kWarps * 32, 0, st>>>(a.logits, a.T, a.E, a.k, a.renorm,
                                                                     a.ids, a.w);
  return cudaGetLastError();
}

cudaError_t launch_route_ensure(const RouteEnsureArgs& a, cudaStream_t st) {
  if (a.r.T <= 0) return cudaSuccess;
  if (a.r.T > kRouteEnsureMaxT || a.r.E > kEnsureMax || a.S > kEnsureMax) return cudaErrorInvalidValue;
  const int per_cta = kEnsureThreads / 32;
  const int grid = (a.r.E + per_cta - 1) / per_cta;
  if (a.pf_n > 0 && a.r.T * a.r.k > kEnsureThreads) return cudaErrorInvalidValue;
  if (grid <= kClusterMaxCtas && a.r.T * a.r.E <= kClusterMaxLogits) {
    const int cgrid = a.pf_n > 0 ? max(grid, 2) : grid;  // CTA 1 runs the lookahead
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(cgrid);
    cfg.blockDim = dim3(kEnsureThreads);
    const int tc = a.r.T == 1 ? 1 : min(a.r.T, kTokChunk);
    cfg.dynamicSmemBytes = (size_t)tc * a.r.H * 2 + (size_t)(a.r.T * a.r.k) * 4 +
                           (a.pf_n > 0 ? (size_t)(2 * a.r.T * a.r.k) * 4 : 0);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cgrid;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 2 : 1;
    if (a.r.T == 1) return cudaLaunchKernelEx(&cfg, route_ensure_cluster_kernel<1>, a);
    return cudaLaunchKernelEx(&cfg, route_ensure_cluster_kernel<kTokChunk>, a);
  }
  RouteEnsureArgs b = a;
  b.pf_n = 0;  // this kernel has no predictor: the lookahead follows as two launches
  cudaError_t e = a.r.T == 1
                      ? launch_k(route_ensure_kernel<1>, dim3(grid), dim3(kEnsureThreads), 0, st, a.pdl != 0, b)
                      : launch_k(route_ensure_kernel<kTokChunk>, dim3(grid), dim3(kEnsureThreads), 0, st,
                                 a.pdl != 0, b);
  if (e != cudaSuccess || a.pf_n <= 0) return e;
  return launch_lookahead(a.r.x, a.wr_next, a.r.T, a.r.E, a.r.H, a.r.k, a.tab_next, a.S, a.pf_n, a.pf_bytes,
                          a.pred_logits, a.pred_ids, a.pred_w, a.pred_done, st);
}

cudaError_t launch_lookahead(const uint16_t* x, const uint16_t* wr_next, int T, int E, int H, int k,
                             LayerTables tab_next, int S, int N, unsigned long long bytes, float* pred_logits,
                             int32_t* pred_ids, float* pred_w, unsigned* pred_done, cudaStream_t st) {
  if (T <= 0 || N <= 0) return cudaSuccess;
  if (T * k > kEnsureThreads || E > kEnsureMax || S > kEnsureMax) return cudaErrorInvalidValue;
  RouteArgs r{};
  r.x = x;
  r.wr = wr_next;
  r.T = T;
  r.E = E;
  r.H = H;
  r.k = k;
  r.renorm = 1;
  r.ids = pred_ids;
  r.w = pred_w;
  r.logits = pred_logits;
  r.done = pred_done;
  cudaError_t e = launch_route(r, st);
  if (e != cudaSuccess) return e;
  return launch_prefetch_install(pred_ids, pred_logits, T, k, E, tab_next, S, N, bytes, st);
}

}  // namespace moe
