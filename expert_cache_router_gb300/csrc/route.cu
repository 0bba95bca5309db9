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
      const uint4 wv = ld_keep(row + c);
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
      asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(row + c));
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
          wv[u] = c < H ? ld_keep(row + c) : make_uint4(0u, 0u, 0u, 0u);
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
  ensure_call(sm, a.tab, r.ids, T * r.k, E, a.S, a.slot_ids, a.status, a.expert_bytes);
  if (threadIdx.x == 0) *r.done = 0u;
}

// Cluster variant of the fused head (E <= 256, T*E <= kClusterMaxLogits, T*k <=
// kHeadThreads): one thread-block cluster of up to 8 CTAs (16 where the device
// holds such a cluster), each owning a contiguous range of at least 16 and at
// most 32 experts, one warp per expert. Each warp copies
// its router row into shared memory (cp.async) before the dependency wait, so
// that once x is in the dot products read only shared memory (a CTA of this
// size cannot become resident beside the preceding kernel's CTAs, so the copy
// overlaps at least the launch and the wait). Each warp stores its logits
// straight into CTA 0's shared memory (distributed shared memory: no global
// round trip, fence or counter);
// after one cluster barrier CTA 0 takes each token's top-k (one warp per token)
// and updates the slot table (one warp for calls of up to 32 pairs on up to 64
// slots) while the other CTAs exit. Same picks, weights and table as the other
// head kernels.
//
// With the router lookahead on (a.pf_n > 0, at least two CTAs), each warp also
// dots the next layer's router rows of its experts with the same x (the
// predictor, rows pulled into L2 before the wait) and stores them into CTA 1's
// shared memory, and CTA 1 does the rest of the lookahead while CTA 0 does the
// demand side: it copies the next layer's table into its shared memory before
// the dependency wait, takes the predicted top-k (the same rule as the demand
// top-k), orders the candidates and installs them (lookahead_candidates_block,
// install_block). The two CTAs write different layers' tables. Dynamic shared
// memory: x of one token chunk [TC][H] (read once per CTA), routed ids,
// predicted ids and candidates [T][k] each, the CTA's router rows [32][H].
constexpr int kClusterMaxLogits = 2048;
constexpr int kHeadMaxE = 256;   // experts of the cluster head (eight keys per lane in the top-k)
constexpr int kRowSmemH = 2048;  // router rows staged in shared memory up to this hidden size
constexpr int kHeadThreads = 1024;
constexpr int kHeadWarps = kHeadThreads / 32;
constexpr int kHeadMaxEpc = 32;  // experts per CTA of the cluster head

// Largest cluster of the head: 16 CTAs (a non-portable size) where the device
// can hold such a cluster of this kernel, else 8. Set by route_init_attributes.
int g_head_cluster_max = 8;

// CTAs of the cluster head for E experts (one warp per expert, at least 16
// experts per CTA, up to g_head_cluster_max CTAs). The router dot products are
// bound by shared-memory bandwidth (each warp reads its router row and its own
// copy of x), so spreading the experts over more CTAs shortens them.
inline int head_ctas(int E) {
  const int c = (E + 15) / 16;
  return c < 1 ? 1 : (c > g_head_cluster_max ? g_head_cluster_max : c);
}

// Top-k of rows [T][E] of logits in shared memory with the rule of
// topk_row_warp and route_ensure_kernel (larger logit first, equal logits by
// lower expert id, NaN ranking as -inf). Each (logit, expert) pair becomes one
// 64-bit key whose unsigned order is that rule: the logit's bits mapped to an
// order-preserving unsigned integer (NaN read as -inf, -0 as +0) in the high
// word, the complement of the expert id in the low word; 0 (below every real
// key) pads. One warp per token holds the row's keys in registers (up to eight
// per lane) and takes the k largest one at a time: no block barrier and no
// shared-memory round trip between the logits and the picks.
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

// One token's row lg[0..E) (E <= 32*R), R keys per lane: k rounds of a
// warp-wide maximum, each two 32-bit reductions (the high words; then the low
// words of the keys whose high word is that maximum), after which the winning
// key leaves its lane. Lane j < k returns the key of pick j, other lanes 0.
// A short loop, not an unrolled network: this code runs once per call, and a
// long straight-line sequence would be fetched cold every time.
template <int R>
__device__ __forceinline__ unsigned long long topk_warp(const float* lg, int E, int k) {
  const int lane = threadIdx.x & 31;
  unsigned long long a[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int e = r * 32 + lane;
    a[r] = e < E ? rank_key(lg[e], e) : 0ull;
  }
  unsigned long long mine = 0ull;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    unsigned long long m[R];
#pragma unroll
    for (int r = 0; r < R; ++r) m[r] = a[r];
#pragma unroll
    for (int w = 1; w < R; w <<= 1)
#pragma unroll
      for (int r = 0; r + w < R; r += 2 * w) m[r] = m[r + w] > m[r] ? m[r + w] : m[r];
    const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(m[0] >> 32));
    const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(m[0] >> 32) == hi ? (uint32_t)m[0] : 0u);
    const unsigned long long win = ((unsigned long long)hi << 32) | lo;
    if (lane == j) mine = win;
#pragma unroll
    for (int r = 0; r < R; ++r) a[r] = a[r] == win ? 0ull : a[r];
  }
  return mine;
}

__device__ __forceinline__ unsigned long long topk_row(const float* lg, int E, int k) {
  if (E <= 32) return topk_warp<1>(lg, E, k);
  if (E <= 64) return topk_warp<2>(lg, E, k);
  if (E <= 128) return topk_warp<4>(lg, E, k);
  return topk_warp<8>(lg, E, k);
}

// TR: the decode-trace variant (stamps into a.tr); the plain one has none.
template <int TC, bool TR>
__global__ void __launch_bounds__(kHeadThreads)
route_ensure_cluster_kernel(RouteEnsureArgs a) {
  unsigned long long* const tr = TR ? a.tr : nullptr;
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ EnsureSmem sm;
  __shared__ float lall[kClusterMaxLogits];  // CTA 0: every logit [T][E]; CTA 1: every predicted logit
  extern __shared__ uint4 dyn[];
  const RouteArgs& r = a.r;
  const unsigned crank = cluster.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = r.H, E = r.E, T = r.T, k = r.k;
  const int epc = (E + (int)cluster.num_blocks() - 1) / (int)cluster.num_blocks();  // experts per CTA
  const int e0 = (int)crank * epc, e1 = min(E, e0 + epc);
  const bool pf = a.pf_n > 0;
  const int tc = T < TC ? T : TC;
  uint16_t* xs = reinterpret_cast<uint16_t*>(dyn);                  // [tc][H] bf16: this chunk's x
  int* ids_s = reinterpret_cast<int*>(xs + (size_t)tc * H);         // [T][k] routed ids (CTA 0)
  int* pid = ids_s + T * k;                                         // [T][k] predicted ids (CTA 1)
  int* cand = pid + T * k;                                          // [T][k] candidates (CTA 1)
  uint16_t* rows_s = reinterpret_cast<uint16_t*>(                   // [epc][H] router rows (H <= kRowSmemH)
      dyn + (((size_t)tc * H * 2 + (size_t)3 * T * k * 4 + 15) / 16));
  // Every CTA must have started before another writes into its shared memory:
  // arrive now, wait just before the first remote store.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  if (crank == 0) ensure_load_table(sm, a.tab, E, a.S);
  if (pf && crank == 1) ensure_load_table(sm, a.tab_next, E, a.S);
  // The router rows do not depend on the preceding kernel: with H <= kRowSmemH
  // each warp copies its rows into shared memory (cp.async, 16 bytes per lane
  // per step, each lane later reading only the chunks it copied) before the
  // dependency wait, kept in L2 with the evict-last hint; longer rows, and the
  // predictor's rows, are pulled into L2.
  const bool row_in_smem = H <= kRowSmemH;
  {
    const unsigned long long keep = l2_evict_last();
    for (int e = e0 + warp; e < e1; e += kHeadWarps) {
      const uint16_t* row = r.wr + (size_t)e * H;
      if (row_in_smem) {
        const uint32_t dst = (uint32_t)__cvta_generic_to_shared(rows_s + (size_t)(e - e0) * H);
        for (int c = lane * 8; c < H; c += 256)
          asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst + 2u * c),
                       "l"(row + c), "l"(keep) : "memory");
      } else {
        for (int c = lane * 64; c < H; c += 32 * 64) asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(row + c));
      }
      if (pf)
        for (int c = lane * 64; c < H; c += 32 * 64)
          asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(a.wr_next + (size_t)e * H + c));
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  pdl_wait();
  pdl_trigger();
  if (crank == 0 && threadIdx.x == 0) trace_max(tr, kTrHeadWait);
  float* to0 = cluster.map_shared_rank(lall, 0);
  float* to1 = cluster.map_shared_rank(lall, pf ? 1 : 0);
  bool waited = false;
  const int h8 = H >> 3;
  for (int t0 = 0; t0 < T; t0 += TC) {
    const int nt = min(TC, T - t0);
    // x rows of this chunk, read once per CTA into shared memory
    __syncthreads();
    for (int i = threadIdx.x; i < nt * h8; i += kHeadThreads)
      dyn[i] = __ldg(reinterpret_cast<const uint4*>(r.x + (size_t)t0 * H) + i);
    if (t0 == 0) asm volatile("cp.async.wait_all;" ::: "memory");  // this lane's row chunks
    __syncthreads();
    for (int e = e0 + warp; e < e1; e += kHeadWarps) {
      const uint16_t* rs = rows_s + (size_t)(e - e0) * H;
      for (int pass = 0; pass < (pf ? 2 : 1); ++pass) {
        const uint16_t* wrow = (pass ? a.wr_next : r.wr) + (size_t)e * H;
        float* dst = pass ? to1 : to0;
        float acc[TC];
#pragma unroll
        for (int t = 0; t < TC; ++t) acc[t] = 0.0f;
        for (int c0 = lane * 8; c0 < H; c0 += 256 * kRowUnroll) {
          uint4 wv[kRowUnroll];
          if (pass == 0 && row_in_smem) {
#pragma unroll
            for (int u = 0; u < kRowUnroll; ++u) {
              const int c = c0 + 256 * u;
              wv[u] = c < H ? *reinterpret_cast<const uint4*>(rs + c) : make_uint4(0u, 0u, 0u, 0u);
            }
          } else {
#pragma unroll
            for (int u = 0; u < kRowUnroll; ++u) {
              const int c = c0 + 256 * u;
              wv[u] = c < H ? ld_keep(wrow + c) : make_uint4(0u, 0u, 0u, 0u);
            }
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
  }
  if (!waited) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  cluster.sync();  // every logit is in CTA 0's (and predicted ones in CTA 1's) shared memory
  if (crank == 0 && threadIdx.x == 0) trace_max(tr, kTrHeadLogits);
  if (pf && crank == 1) {
    // Lookahead into the next layer: predicted top-k, candidates, install.
    for (int t = warp; t < T; t += kHeadWarps) {
      const unsigned long long key = topk_row(lall + t * E, E, k);
      if (lane < k) pid[t * k + lane] = key_expert(key);
    }
    __syncthreads();
    const int nc = lookahead_candidates_block(sm, pid, lall, T, k, E, cand);
    install_block(sm, a.tab_next, cand, nc, a.pf_n, E, a.S, a.pf_bytes, true);
    return;
  }
  if (crank != 0) return;

  // Top-k and weights of each token in one warp; the picks go to the caller's ids
  // and weights and, for the slot update, to shared memory.
  for (int t = warp; t < T; t += kHeadWarps) {
    const float* row = lall + t * E;
    const unsigned long long key = topk_row(row, E, k);
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
  if (threadIdx.x == 0) trace_max(tr, kTrHeadTopk);
  ensure_call(sm, a.tab, ids_s, T * k, E, a.S, a.slot_ids, a.status, a.expert_bytes);
  if (threadIdx.x == 0) trace_max(tr, kTrHeadDone);
}

}  // namespace

// Dynamic shared memory of the cluster head: x of one token chunk [TC][H] bf16,
// routed ids, predicted ids and candidates [T][k] each (T*k <= kHeadThreads),
// then (H <= kRowSmemH) the router rows of the CTA's experts [<= 32][H] bf16.
constexpr int kHeadSmemWide = kTokChunk * 8192 * 2 + 3 * kHeadThreads * 4 + 16;  // H = 8192
constexpr int kHeadSmemRows =
    kTokChunk * kRowSmemH * 2 + 3 * kHeadThreads * 4 + 16 + kHeadMaxEpc * kRowSmemH * 2;  // H <= 2048
constexpr int kHeadSmemAttr = kHeadSmemWide > kHeadSmemRows ? kHeadSmemWide : kHeadSmemRows;
static_assert(kHeadSmemAttr + (int)sizeof(EnsureSmem) + kClusterMaxLogits * 4 <= 227 * 1024, "head shared memory");

cudaError_t route_init_attributes() {
  cudaError_t e = cudaFuncSetAttribute(route_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemMax);
  for (auto kern : {route_ensure_cluster_kernel<1, false>, route_ensure_cluster_kernel<kTokChunk, false>,
                    route_ensure_cluster_kernel<1, true>})
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kHeadSmemAttr);
  if (e == cudaSuccess) {
    // 16-CTA head clusters where the device holds one (every instantiation).
    int fits = 1;
    for (auto kern : {route_ensure_cluster_kernel<1, false>, route_ensure_cluster_kernel<kTokChunk, false>,
                      route_ensure_cluster_kernel<1, true>}) {
      int n = 0;
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(16);
      cfg.blockDim = dim3(kHeadThreads);
      cfg.dynamicSmemBytes = kHeadSmemAttr;
      cudaLaunchAttribute at;
      at.id = cudaLaunchAttributeClusterDimension;
      at.val.clusterDim.x = 16;
      at.val.clusterDim.y = 1;
      at.val.clusterDim.z = 1;
      cfg.attrs = &at;
      cfg.numAttrs = 1;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
          cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1)
        fits = 0;
    }
    (void)cudaGetLastError();  // a refused query leaves the portable size, not an error
    g_head_cluster_max = fits ? 16 : 8;
  }
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
  if (a.pf_n > 0 && a.r.T * a.r.k > kEnsureThreads) return cudaErrorInvalidValue;
  const int T = a.r.T, E = a.r.E, k = a.r.k;
  if (E <= kHeadMaxE && T * E <= kClusterMaxLogits && T * k <= kHeadThreads) {
    const int cgrid = a.pf_n > 0 ? max(head_ctas(E), 2) : head_ctas(E);  // CTA 1 runs the lookahead
    if ((E + cgrid - 1) / cgrid > kHeadMaxEpc) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(cgrid);
    cfg.blockDim = dim3(kHeadThreads);
    const int tc = T == 1 ? 1 : min(T, kTokChunk);
    const int epc = (E + cgrid - 1) / cgrid;
    // x chunk, then the three [T][k] id arrays (all reserved, so the row area's
    // offset is the one the kernel computes), then the CTA's router rows
    cfg.dynamicSmemBytes = ((size_t)tc * a.r.H * 2 + (size_t)3 * T * k * 4 + 15) / 16 * 16 +
                           (a.r.H <= kRowSmemH ? (size_t)epc * a.r.H * 2 : 0);
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
    if (T == 1 && a.tr) return cudaLaunchKernelEx(&cfg, route_ensure_cluster_kernel<1, true>, a);
    if (T == 1) return cudaLaunchKernelEx(&cfg, route_ensure_cluster_kernel<1, false>, a);
    return cudaLaunchKernelEx(&cfg, route_ensure_cluster_kernel<kTokChunk, false>, a);
  }
  const int per_cta = kEnsureThreads / 32;
  const int grid = (E + per_cta - 1) / per_cta;
  RouteEnsureArgs b = a;
  b.pf_n = 0;  // this kernel has no predictor: the lookahead follows as two launches
  cudaError_t e = T == 1
                      ? launch_k(route_ensure_kernel<1>, dim3(grid), dim3(kEnsureThreads), 0, st, a.pdl != 0, b)
                      : launch_k(route_ensure_kernel<kTokChunk>, dim3(grid), dim3(kEnsureThreads), 0, st,
                                 a.pdl != 0, b);
  if (e != cudaSuccess || a.pf_n <= 0) return e;
  return launch_lookahead(a.r.x, a.wr_next, T, E, a.r.H, k, a.tab_next, a.S, a.pf_n, a.pf_bytes,
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
