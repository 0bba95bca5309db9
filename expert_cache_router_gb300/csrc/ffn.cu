// Grouped expert FFN for decode-sized calls, over the [num_slots, N, K] slot
// tensors ("MoE expert offload" page, "How it works": the GEMMs read slot
// tensors instead of [num_experts, N, K]). The expert FFN is the fused
// gate+up+SiLU form ("MoE-Infinity" page, feature list):
//   g, u = W13[slot] x   (fp32)      h = silu(g) * u      y = W2[slot] h   (fp32)
//   out_t = bf16( sum_{j=0..k-1} w[t,j] * y[t,j] [+ y_shared] )   in rank order
//
// Two launches. The gate/up grid is (T*k pairs [+1 shared-expert column] [+ copy
// columns]) x (row blocks); the CTA of pair p works only when p is the first
// pair routed to its slot, and then serves every pair of that slot, so each
// expert's weights cross HBM (or the host link, for a spilled expert) once per
// call. Each token's dot products are accumulated in the same order whatever
// else shares the expert, whichever slot holds it and whether it is read from a
// slot or from host memory, so the output is bit-identical for every slot
// count. The down launch owns disjoint output rows per CTA and sums the k
// ranks of each token in order inside the CTA (the shared expert last, weight 1).
//
// Copy-through (decode step): the experts the slot ensure of this call
// installed are not copied by a separate launch first. The CTAs that compute a
// newly installed expert read its W13 rows from mapped host memory and store
// every 16-byte chunk they load into the slot, and extra CTAs of the same
// launch copy its W2 (and FP8 block scales) into the slot, so the host-link
// stream of the misses overlaps the HBM stream of the hits. The down launch
// then reads W2 from the slot.
//
// Early down (decode step under programmatic dependent launch): the down launch
// does not wait for the whole gate/up grid. Each gate/up CTA of a serving column
// counts itself done once its h rows are written, each W2-copy CTA once its copies
// are; a down warp waits (bounded) only for the groups it computes, hits first, so
// the down work of the resident experts overlaps the host-link stream of the
// missed ones. The down grid can only start once every gate/up CTA has started
// (each triggers the dependent launch at its start), so no wait can hold a
// producer off the GPU. The last down CTA waits for the gate/up grid to complete
// and zeroes the counters for the next call.
//
// Weight formats: bf16 (8 elements per 16-byte load) or FP8 e4m3 with one fp32
// scale per 128 x 128 block (16 elements per load; a load never crosses a
// block, so each chunk's partial dot is scaled once).
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "kernels.h"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kGateRowsPerWarp = 2;                         // gate rows (and as many up rows)
constexpr int kGateRowsPerCta = kWarps * kGateRowsPerWarp;  // 16 rows of I per CTA
constexpr int kMaxPairs = 1024;
constexpr int kCopyCols = 4;  // copy-through: extra grid columns of W2 copy workers
constexpr int kSyncCopy = kSyncCopyLine * kSyncLine;  // early down: W2-copy CTAs done
constexpr int kSyncDone = kSyncDoneLine * kSyncLine;  // early down: down CTAs done
static_assert(kSyncColumns >= kMaxPairs + 1, "early-down counters");

template <int FMT>
struct Fmt;
template <>
struct Fmt<0> {  // bf16
  static constexpr int kElems = 8;
  static constexpr int kBytes = 2;
};
template <>
struct Fmt<1> {  // FP8 e4m3, 128 x 128 block scales
  static constexpr int kElems = 16;
  static constexpr int kBytes = 1;
};

struct Group {
  int leader;   // 1 when this CTA serves the slot of its pair
  int valid;    // slot id resolves to weights
  int n;        // pairs in the group
  const uint8_t* w13;
  const uint8_t* w2;
  const float* s13;   // FP8 scales (nullptr for bf16)
  const float* s2;
  uint8_t* w13_dst;  // copy-through: the slot this CTA also fills, else nullptr
};

__device__ __forceinline__ void fp8x16_to_f32(const uint4 w, float* f) {
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(words[i] & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(words[i] >> 16), __NV_E4M3);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    f[4 * i] = a.x;
    f[4 * i + 1] = a.y;
    f[4 * i + 2] = b.x;
    f[4 * i + 3] = b.y;
  }
}

// 16-byte load through L2 only, for slot bytes another CTA may have written during this call.
__device__ __forceinline__ uint4 ld_l2(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}

// Early down: this CTA's part of a gate/up column (or of the W2 copy) is written.
__device__ __forceinline__ void signal_done(uint32_t* sync, int word) {
  if (!sync) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(sync + word, 1u);
  }
}

__device__ __forceinline__ void load_x8(const uint16_t* p, float* xv) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  xv[0] = bf16lo(v.x); xv[1] = bf16hi(v.x); xv[2] = bf16lo(v.y); xv[3] = bf16hi(v.y);
  xv[4] = bf16lo(v.z); xv[5] = bf16hi(v.z); xv[6] = bf16lo(v.w); xv[7] = bf16hi(v.w);
}

// acc += (weight chunk . activation chunk) [* block scale], activations bf16 (x) or fp32 (h).
template <int FMT>
__device__ __forceinline__ float chunk_dot_x(const uint4 w, const uint16_t* x, float sc, float acc) {
  if constexpr (FMT == 0) {
    float xv[8];
    load_x8(x, xv);
    return dot8(w, xv, acc);
  } else {
    float wf[16], xv[16];
    fp8x16_to_f32(w, wf);
    load_x8(x, xv);
    load_x8(x + 8, xv + 8);
    float part = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) part = fmaf(wf[i], xv[i], part);
    return fmaf(part, sc, acc);
  }
}

template <int FMT>
__device__ __forceinline__ float chunk_dot_h(const uint4 w, const float* h, float sc, float acc) {
  if constexpr (FMT == 0) {
    const float4 h0 = __ldcg(reinterpret_cast<const float4*>(h));
    const float4 h1 = __ldcg(reinterpret_cast<const float4*>(h + 4));
    const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    return dot8(w, hv, acc);
  } else {
    float wf[16];
    fp8x16_to_f32(w, wf);
    float part = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 hq = __ldcg(reinterpret_cast<const float4*>(h + 4 * q));
      part = fmaf(wf[4 * q], hq.x, part);
      part = fmaf(wf[4 * q + 1], hq.y, part);
      part = fmaf(wf[4 * q + 2], hq.z, part);
      part = fmaf(wf[4 * q + 3], hq.w, part);
    }
    return fmaf(part, sc, acc);
  }
}

// Per-expert sizes in bytes (weights) and floats (FP8 scales).
struct ExpertSizes {
  size_t e13, e2, f13, f2;
};
template <int FMT>
__device__ __forceinline__ ExpertSizes sizes_of(const FfnArgs& a) {
  ExpertSizes z;
  z.e13 = (size_t)2 * a.I * a.H * Fmt<FMT>::kBytes;
  z.e2 = (size_t)a.H * a.I * Fmt<FMT>::kBytes;
  z.f13 = FMT ? (size_t)(2 * a.I / 128) * (a.H / 128) : 0;
  z.f2 = FMT ? (size_t)(a.H / 128) * (a.I / 128) : 0;
  return z;
}

// Shared-memory group of pair blockIdx.x: pairs routed to the same slot, in pair order.
// The slot ids and the pair's host source (the expert id when the call installed or spilled it,
// from the ensure that produced the slot ids) arrive in one round trip.
template <int FMT>
__device__ void form_group(const FfnArgs& a, int* sid, int* members, Group* g, bool copy_through) {
  __shared__ int s_src;
  const int Tk = a.T * a.k;
  const int p = blockIdx.x;
  const ExpertSizes z = sizes_of<FMT>(a);
  for (int q = threadIdx.x; q < Tk; q += kThreads) sid[q] = __ldcg(a.slot_ids + q);
  if (threadIdx.x == 0) s_src = a.pair_src ? __ldcg(a.pair_src + p) : -1;
  __syncthreads();
  const int s = sid[p];
  int dup = 0;
  for (int q = threadIdx.x; q < p; q += kThreads) dup |= (sid[q] == s);
  const int is_dup = __syncthreads_or(dup);
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int count = 0;
    if (!is_dup) {
      for (int base = p; base < Tk; base += 32) {
        const int q = base + lane;
        const bool m = q < Tk && sid[q] == s;
        const unsigned bal = __ballot_sync(0xffffffffu, m);
        if (m) members[count + __popc(bal & ((1u << lane) - 1u))] = q;
        count += __popc(bal);
      }
    }
    if (lane == 0) {
      g->leader = !is_dup;
      g->n = count;
      g->valid = 0;
      g->w13 = g->w2 = nullptr;
      g->s13 = g->s2 = nullptr;
      g->w13_dst = nullptr;
      const int e = s_src;  // expert read from host memory in this call, or -1
      if (!is_dup) {
        if (s >= 0 && s < a.S) {
          g->w13 = a.lw.slot_w13 + (size_t)s * z.e13;
          g->w2 = a.lw.slot_w2 + (size_t)s * z.e2;
          if (FMT) {
            g->s13 = a.lw.slot_s13 + (size_t)s * z.f13;
            g->s2 = a.lw.slot_s2 + (size_t)s * z.f2;
          }
          g->valid = 1;
          if (copy_through && e >= 0 && e < a.E) {  // installed by this call: read it from host, fill the slot
            g->w13 = a.lw.host_w13 + (size_t)e * z.e13;
            if (FMT) g->s13 = a.lw.host_s13 + (size_t)e * z.f13;
            g->w13_dst = a.lw.slot_w13 + (size_t)s * z.e13;
          }
        } else if (s >= a.S && e >= 0 && e < a.E) {  // spilled: read from host memory
          g->w13 = a.lw.host_w13 + (size_t)e * z.e13;
          g->w2 = a.lw.host_w2 + (size_t)e * z.e2;
          if (FMT) {
            g->s13 = a.lw.host_s13 + (size_t)e * z.f13;
            g->s2 = a.lw.host_s2 + (size_t)e * z.f2;
          }
          g->valid = 1;
        }
        if (!g->valid) atomicOr(a.status, kDevBadSlotId);
      }
    }
  }
  __syncthreads();
}

// Copy-through workers: W2 (and FP8 scales) of every expert installed by this call, host -> slot.
template <int FMT>
__device__ void copy_installed_rest(const FfnArgs& a, int worker, int workers) {
  const int n = min(__ldcg(a.counts + kCntInstall), a.S);
  if (n <= 0) return;
  const ExpertSizes z = sizes_of<FMT>(a);
  const unsigned long long u2 = z.e2 / 16;  // 16-byte units of W2 per expert
  const unsigned long long total = (unsigned long long)n * u2;
  const unsigned long long stride = (unsigned long long)workers * kThreads;
  const unsigned long long t0 = (unsigned long long)worker * kThreads + threadIdx.x;
  if (FMT) {
    const unsigned long long fpe = z.f13 + z.f2;
    for (unsigned long long v = t0; v < (unsigned long long)n * fpe; v += stride) {
      const int i = (int)(v / fpe);
      const unsigned long long o = v - (unsigned long long)i * fpe;
      const int e = __ldcg(a.miss_expert + i), sl = __ldcg(a.miss_slot + i);
      if ((unsigned)e >= (unsigned)a.E || (unsigned)sl >= (unsigned)a.S) continue;
      if (o < z.f13) a.lw.slot_s13[(size_t)sl * z.f13 + o] = a.lw.host_s13[(size_t)e * z.f13 + o];
      else a.lw.slot_s2[(size_t)sl * z.f2 + (o - z.f13)] = a.lw.host_s2[(size_t)e * z.f2 + (o - z.f13)];
    }
  }
  const uint4* src = reinterpret_cast<const uint4*>(a.lw.host_w2);
  uint4* dst = reinterpret_cast<uint4*>(a.lw.slot_w2);
  constexpr int U = 8;
  for (unsigned long long u0 = t0; u0 < total; u0 += stride * U) {
    uint4 v[U];
    uint4* d[U];
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const unsigned long long u = u0 + q * stride;
      d[q] = nullptr;
      if (u < total) {
        const int i = (int)(u / u2);
        const unsigned long long off = u - (unsigned long long)i * u2;
        const int e = __ldcg(a.miss_expert + i), sl = __ldcg(a.miss_slot + i);
        if ((unsigned)e < (unsigned)a.E && (unsigned)sl < (unsigned)a.S) {
          v[q] = ld_stream(src + (size_t)e * u2 + off);
          d[q] = dst + (size_t)sl * u2 + off;
        }
      }
    }
#pragma unroll
    for (int q = 0; q < U; ++q)
      if (d[q]) *d[q] = v[q];
  }
}

// One token (TC = 1): four CTAs per SM (64 registers), so that the batch-1 grid of
// 8 pairs + 4 copy columns x 48 row blocks is resident at once and the missed
// expert's row blocks all start with the launch.
// TR: the decode-trace variant (stamps into a.tr); the plain one has none.
template <int FMT, int TC, bool TR>
__global__ void __launch_bounds__(kThreads, TC == 1 ? 4 : 0)
ffn_gate_up_kernel(FfnArgs a) {
  __shared__ int sid[kMaxPairs];
  __shared__ int members[kMaxPairs];
  __shared__ Group g;
  unsigned long long* const tr = TR ? a.tr : nullptr;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) trace_min(tr, kTrGateFirst);
  const int Tk = a.T * a.k;
  const int cols = Tk + (a.shared ? 1 : 0);
  if ((int)blockIdx.x >= cols) {  // copy-through W2 workers
    copy_installed_rest<FMT>(a, (blockIdx.x - cols) * gridDim.y + blockIdx.y, (gridDim.x - cols) * gridDim.y);
    signal_done(a.sync, kSyncCopy);
    if (threadIdx.x == 0) {
      trace_max(tr, kTrCopyDone);
      trace_max(tr, kTrGateDone);
    }
    return;
  }
  if ((int)blockIdx.x < Tk) {
    form_group<FMT>(a, sid, members, &g, a.copy_through != 0);
  } else {  // the shared expert serves every token
    for (int t = threadIdx.x; t < a.T; t += kThreads) members[t] = Tk + t;
    if (threadIdx.x == 0) {
      g.leader = 1;
      g.n = a.T;
      g.w13 = a.lw.sh_w13;
      g.s13 = a.lw.sh_s13;
      g.w2 = a.lw.sh_w2;
      g.s2 = a.lw.sh_s2;
      g.w13_dst = nullptr;
      g.valid = g.w13 != nullptr && (FMT == 0 || g.s13 != nullptr);
      if (!g.valid) atomicOr(a.status, kDevBadSlotId);
    }
    __syncthreads();
  }
  if (!g.leader) return;
  const int col_word = blockIdx.x * kSyncLine;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i0 = blockIdx.y * kGateRowsPerCta + warp * kGateRowsPerWarp;
  const int H = a.H, I = a.I, k = a.k;
  if (!g.valid) {
    for (int m = 0; m < g.n; ++m)
      for (int r = lane; r < kGateRowsPerWarp; r += 32)
        if (i0 + r < I) a.hbuf[(size_t)members[m] * I + i0 + r] = 0.0f;
    signal_done(a.sync, col_word);
    return;
  }
  constexpr int CE = Fmt<FMT>::kElems, EB = Fmt<FMT>::kBytes;
  // chunks of 32*CE columns per lane-step; UNR chunks' loads are issued together
  constexpr int UNR = TC == 1 ? 2 : (TC <= 2 ? 4 : (TC <= 4 ? 2 : 1));
  constexpr int R2 = 2 * kGateRowsPerWarp;
  const int hb = H >> 7;
  for (int m0 = 0; m0 < g.n; m0 += TC) {
    const int nt = min(TC, g.n - m0);
    float acc[R2][TC];
#pragma unroll
    for (int r = 0; r < R2; ++r)
#pragma unroll
      for (int t = 0; t < TC; ++t) acc[r][t] = 0.0f;
    const uint16_t* xrow[TC];
#pragma unroll
    for (int t = 0; t < TC; ++t) {
      const int pm = members[m0 + min(t, nt - 1)];
      xrow[t] = a.x + (size_t)(pm < Tk ? pm / k : pm - Tk) * H;
    }
    // the first token chunk of a copy-through group also writes the slot
    uint8_t* dst = m0 == 0 ? g.w13_dst : nullptr;
    if (i0 < I) {
      for (int c0 = lane * CE; c0 < H; c0 += 32 * CE * UNR) {
        uint4 wv[UNR][R2];
        float sc[UNR][R2];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int c = c0 + 32 * CE * u;
#pragma unroll
          for (int r = 0; r < R2; ++r) {
            const int row = r < kGateRowsPerWarp ? i0 + r : I + i0 + r - kGateRowsPerWarp;
            wv[u][r] = c < H ? ld_stream(g.w13 + ((size_t)row * H + c) * EB) : make_uint4(0u, 0u, 0u, 0u);
            sc[u][r] = (FMT && c < H) ? __ldg(g.s13 + (row >> 7) * hb + (c >> 7)) : 1.0f;
          }
        }
        if (dst) {
#pragma unroll
          for (int u = 0; u < UNR; ++u) {
            const int c = c0 + 32 * CE * u;
            if (c < H) {
#pragma unroll
              for (int r = 0; r < R2; ++r) {
                const int row = r < kGateRowsPerWarp ? i0 + r : I + i0 + r - kGateRowsPerWarp;
                *reinterpret_cast<uint4*>(dst + ((size_t)row * H + c) * EB) = wv[u][r];
              }
            }
          }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int c = c0 + 32 * CE * u;
          if (c < H) {
#pragma unroll
            for (int t = 0; t < TC; ++t) {
              if (t < nt) {
#pragma unroll
                for (int r = 0; r < R2; ++r) acc[r][t] = chunk_dot_x<FMT>(wv[u][r], xrow[t] + c, sc[u][r], acc[r][t]);
              }
            }
          }
        }
        // first host chunk of an installed expert used: the test reads acc, so the
        // stamp follows the chunk's arrival (it is skipped only if acc hits that value)
        if (TR && dst && c0 == lane * CE && threadIdx.x == 0 && acc[0][0] != 1.2345e-7f)
          trace_min(tr, kTrGateHostFirst);
      }
    }
#pragma unroll
    for (int t = 0; t < TC; ++t) {
#pragma unroll
      for (int r = 0; r < kGateRowsPerWarp; ++r) {
        const float gs = warp_sum(acc[r][t]);
        const float us = warp_sum(acc[kGateRowsPerWarp + r][t]);
        if (lane == 0 && t < nt && i0 + r < I) {
          const float silu = gs / (1.0f + expf(-gs));
          a.hbuf[(size_t)members[m0 + t] * I + i0 + r] = silu * us;
        }
      }
    }
  }
  signal_done(a.sync, col_word);
  if (threadIdx.x == 0) {
    if (g.w13_dst) trace_max(tr, kTrGateHostDone);
    trace_max(tr, kTrGateDone);
  }
}

// Down projection + combine. CTA b owns output rows [8b, 8b+8) for every
// token: its warps take the call's distinct slots in turn (then the shared
// expert) and dot each of the 8 W2 rows with h of every pair routed to that
// slot; the CTA then sums the k ranks of each token in rank order (and the
// shared expert last, weight 1). No other CTA touches these rows.
// (The one-token variants are held to two CTAs per SM, 128 registers.)
template <int FMT, int TC, bool TR>
__global__ void __launch_bounds__(kThreads, TC == 1 ? 2 : 0)
ffn_down_combine_kernel(FfnArgs a) {
  unsigned long long* const tr = TR ? a.tr : nullptr;
  extern __shared__ float ys[];       // [parts][Tk (+T)][kDownRowsPerCta]
  __shared__ int sid[kMaxPairs];
  __shared__ int nxt[kMaxPairs];      // next pair routed to the same slot, -1 at the end
  __shared__ int glead[kMaxPairs];    // first pair of each distinct slot, in pair order
  __shared__ unsigned char lead[kMaxPairs];  // 1: first pair of a hit slot, 2: of a missed expert
  __shared__ float s_w[kMaxPairs];    // routing weights of the call
  __shared__ int s_src[kMaxPairs];    // host source of each pair (installed or spilled expert), else -1
  __shared__ int s_groups;
  __shared__ int s_last;              // early down: this CTA resets the counters at its end
  __shared__ int s_waited;            // early down: warps past their last wait
  const int Tk = a.T * a.k;
  const int H = a.H, I = a.I, k = a.k;
  constexpr int CE = Fmt<FMT>::kElems, EB = Fmt<FMT>::kBytes;
  const ExpertSizes z = sizes_of<FMT>(a);
  if (threadIdx.x == 0) trace_min(tr, kTrDownFirst);
  // The slot ids, weights and host sources come from the kernel two launches
  // back (the head), which has completed: read them once, together, into
  // shared memory. Early down reads only these before its per-group waits
  // (every gate/up CTA started after the head completed).
  for (int p = threadIdx.x; p < Tk; p += kThreads) {
    sid[p] = __ldcg(a.slot_ids + p);
    s_w[p] = __ldcg(a.w + p);
    s_src[p] = a.pair_src ? __ldcg(a.pair_src + p) : -1;
  }
  if (threadIdx.x == 0) {
    s_last = 0;
    s_waited = 0;
  }
  __syncthreads();
  if (a.pdl) {
    // Pull this CTA's W2 rows of every slot into L2 while the gate/up launch
    // still runs. (Lines of slots it is still filling are refreshed in L2 by
    // its stores; L1 is not filled.)
    const int lpr = (I * EB + 127) / 128;  // 128-byte lines per W2 row
    const int r0p = blockIdx.x * kDownRowsPerCta;
    const int rows = min(kDownRowsPerCta, H - r0p);
    for (int i = threadIdx.x; i < Tk * rows * lpr; i += kThreads) {
      const int p = i / (rows * lpr), rem = i - p * (rows * lpr);
      const int r = rem / lpr, line = rem - r * lpr;
      const int s = sid[p];
      if (s >= 0 && s < a.S)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a.lw.slot_w2 + (size_t)s * z.e2 +
                                                      ((size_t)(r0p + r) * I) * EB + line * 128));
    }
  }
  if (!a.sync) pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int p = threadIdx.x; p < Tk; p += kThreads) {
    const int s = sid[p];
    int first = 1, nx = -1;
    for (int q = 0; q < p; ++q)
      if (sid[q] == s) { first = 0; break; }
    for (int q = p + 1; q < Tk; ++q)
      if (sid[q] == s) { nx = q; break; }
    lead[p] = (unsigned char)(first ? (s_src[p] >= 0 ? 2 : 1) : 0);
    nxt[p] = nx;
  }
  __syncthreads();
  if (warp == 0) {  // groups in pair order, those of hit slots first
    int count = 0;
    for (int kind = 1; kind <= 2; ++kind) {
      for (int base = 0; base < Tk; base += 32) {
        const int p = base + lane;
        const bool m = p < Tk && lead[p] == kind;
        const unsigned bal = __ballot_sync(0xffffffffu, m);
        if (m) glead[count + __popc(bal & ((1u << lane) - 1u))] = p;
        count += __popc(bal);
      }
    }
    if (lane == 0) s_groups = count;
  }
  __syncthreads();
  const uint32_t gate_ctas = (uint32_t)((I + kGateRowsPerCta - 1) / kGateRowsPerCta);
  const unsigned long long wait_ns = a.wait_ns ? a.wait_ns : kDefaultWaitNs;
  const uint32_t copy_ctas = a.copy_through ? (uint32_t)kCopyCols * gate_ctas : 0u;
  const int r0 = blockIdx.x * kDownRowsPerCta;
  const int ib = I >> 7;
  const int ngroups = s_groups + (a.shared ? 1 : 0);
  // One token with fewer expert groups than warps (a small top-k, e.g. 2): each
  // group's I range is split over `parts` warps, whole loop steps each, and the
  // partial sums are added in part order in the combine. With one part this is
  // the plain per-group loop.
  const int parts = (TC == 1 && a.T == 1 && ngroups > 0 && ngroups < kWarps) ? kWarps / ngroups : 1;
  const int items = ngroups * parts;
  const int npairs = Tk + (a.shared ? a.T : 0);
  // Early down: the CTA counts itself done once every warp is past its last
  // wait, so that round trip overlaps the compute; the CTA that counts last
  // resets the counters at its end.
  auto waits_done = [&]() {
    if (a.sync && lane == 0 && atomicAdd(&s_waited, 1) == kWarps - 1) {
      s_last = atomicAdd(a.sync + kSyncDone, 1u) == gridDim.x - 1;
      trace_max(tr, kTrDownWaits);
    }
  };
  if (warp >= items) waits_done();
  for (int item = warp; item < items; item += kWarps) {
    const int d = parts == 1 ? item : item % ngroups, part = parts == 1 ? 0 : item / ngroups;
    float* ysp = ys + (size_t)part * npairs * kDownRowsPerCta;  // this part's partial sums
    const uint8_t* w2 = nullptr;
    const float* s2 = nullptr;
    int p0;
    bool filled = false;  // slot filled by this call's copy CTAs
    if (d < s_groups) {
      p0 = glead[d];
      const int s = sid[p0];
      if (s >= 0 && s < a.S) {
        w2 = a.lw.slot_w2 + (size_t)s * z.e2;
        if (FMT) s2 = a.lw.slot_s2 + (size_t)s * z.f2;
        filled = a.copy_through && lead[p0] == 2;
      } else if (s >= a.S && a.pair_src) {  // spilled: read from host memory
        const int e = s_src[p0];
        if (e >= 0 && e < a.E) {
          w2 = a.lw.host_w2 + (size_t)e * z.e2;
          if (FMT) s2 = a.lw.host_s2 + (size_t)e * z.f2;
        }
      }
    } else {  // the shared expert: virtual pairs Tk..Tk+T-1
      p0 = Tk;
      w2 = a.lw.sh_w2;
      s2 = a.lw.sh_s2;
      if (FMT && !s2) w2 = nullptr;
    }
    if (!w2 && lane == 0) atomicOr(a.status, kDevBadSlotId);
    if (a.sync) {
      // (a.stall: the first group's target is one more CTA than its column has, so it runs out)
      const uint32_t target = gate_ctas + (a.stall && d == 0 ? 1u : 0u);
      if (lane == 0 && wait_at_least(a.sync + (d < s_groups ? p0 : Tk) * kSyncLine, target, a.status, wait_ns) &&
          filled)
        wait_at_least(a.sync + kSyncCopy, copy_ctas, a.status, wait_ns);
      __syncwarp();
      if (item + kWarps >= items) waits_done();
    }
    const bool coh = a.sync && filled;
    for (int p = p0; p >= 0;) {
      int mem[TC];
      int nt = 0;
#pragma unroll
      for (int t = 0; t < TC; ++t) {
        mem[t] = p >= 0 ? p : mem[t > 0 ? t - 1 : 0];
        if (p >= 0) {
          ++nt;
          p = p < Tk ? nxt[p] : (p + 1 < Tk + a.T ? p + 1 : -1);
        }
      }
      if (!w2) {
        for (int t = 0; t < nt; ++t)
          if (lane < kDownRowsPerCta) ysp[mem[t] * kDownRowsPerCta + lane] = 0.0f;
        continue;
      }
      float acc[kDownRowsPerCta][TC];
#pragma unroll
      for (int r = 0; r < kDownRowsPerCta; ++r)
#pragma unroll
        for (int t = 0; t < TC; ++t) acc[r][t] = 0.0f;
      constexpr int UNR = FMT == 1 ? 1 : (TC <= 2 ? 3 : 1);
      constexpr int kStep = 32 * CE * UNR;  // columns of one loop step
      const int span = (I + parts * kStep - 1) / (parts * kStep) * kStep;
      const int i_lo = part * span, i_hi = min(I, i_lo + span);
      for (int c0 = i_lo + lane * CE; c0 < i_hi; c0 += kStep) {
        uint4 wv[UNR][kDownRowsPerCta];
        float sc[UNR][kDownRowsPerCta];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int c = c0 + 32 * CE * u;
#pragma unroll
          for (int r = 0; r < kDownRowsPerCta; ++r) {
            const bool in = c < I && r0 + r < H;
            const uint8_t* wp = w2 + ((size_t)(r0 + r) * I + c) * EB;
            wv[u][r] = in ? (coh ? ld_l2(wp) : ld_stream(wp)) : make_uint4(0u, 0u, 0u, 0u);
            if (FMT) {
              const float* sp = s2 + ((r0 + r) >> 7) * ib + (c >> 7);
              sc[u][r] = in ? (coh ? __ldcg(sp) : __ldg(sp)) : 1.0f;
            } else {
              sc[u][r] = 1.0f;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int c = c0 + 32 * CE * u;
          if (c < I) {
#pragma unroll
            for (int t = 0; t < TC; ++t) {
              if (t < nt) {
                const float* hr = a.hbuf + (size_t)mem[t] * I + c;
#pragma unroll
                for (int r = 0; r < kDownRowsPerCta; ++r) acc[r][t] = chunk_dot_h<FMT>(wv[u][r], hr, sc[u][r], acc[r][t]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < TC; ++t) {
#pragma unroll
        for (int r = 0; r < kDownRowsPerCta; ++r) {
          const float yv = warp_sum(acc[r][t]);
          if (lane == 0 && t < nt) ysp[mem[t] * kDownRowsPerCta + r] = yv;
        }
      }
    }
  }
  __syncthreads();
  const int rows = min(kDownRowsPerCta, H - r0);
  for (int idx = threadIdx.x; idx < a.T * rows; idx += kThreads) {
    const int t = idx / rows, r = idx - t * rows;
    auto y_of = [&](int pair) {  // the pair's y row, its parts added in order
      float y = ys[pair * kDownRowsPerCta + r];
      for (int q = 1; q < parts; ++q) y = __fadd_rn(y, ys[((size_t)q * npairs + pair) * kDownRowsPerCta + r]);
      return y;
    };
    float acc = 0.0f;
    for (int j = 0; j < k; ++j) acc = __fadd_rn(acc, __fmul_rn(s_w[t * k + j], y_of(t * k + j)));
    if (a.shared) acc = __fadd_rn(acc, y_of(Tk + t));
    const __nv_bfloat16 b = __float2bfloat16_rn(acc);
    a.out[(size_t)t * H + r0 + r] = *reinterpret_cast<const uint16_t*>(&b);
  }
  if (threadIdx.x == 0) trace_max(tr, kTrDownOut);  // thread 0's rows written
  if (a.sync && s_last) {  // every down CTA is past its waits: let the gate/up grid complete, reset
    if (threadIdx.x == 0) {
      if (copy_ctas) wait_at_least(a.sync + kSyncCopy, copy_ctas, a.status, wait_ns);
      pdl_wait();
    }
    __syncthreads();
    {
      const int cols = Tk + (a.shared ? 1 : 0);
      for (int c = threadIdx.x; c < cols; c += kThreads) a.sync[c * kSyncLine] = 0u;
      if (threadIdx.x == 0) {
        a.sync[kSyncCopy] = 0u;
        a.sync[kSyncDone] = 0u;
      }
    }
  }
  if (threadIdx.x == 0) trace_max(tr, kTrDownDone);
}

template <int FMT, int TC>
cudaError_t launch_tc(const FfnArgs& a, int phase, cudaStream_t st) {
  const int Tk = a.T * a.k;
  if (phase == 0) {
    dim3 g1(Tk + (a.shared ? 1 : 0) + (a.copy_through ? kCopyCols : 0),
            (a.I + kGateRowsPerCta - 1) / kGateRowsPerCta);
    if (TC == 1 && a.tr) return launch_k(ffn_gate_up_kernel<FMT, 1, true>, g1, dim3(kThreads), 0, st, a.pdl != 0, a);
    return launch_k(ffn_gate_up_kernel<FMT, TC, false>, g1, dim3(kThreads), 0, st, a.pdl != 0, a);
  }
  // one token: room for the partial sums of up to kWarps parts per group
  const size_t smem = (size_t)(Tk + (a.shared ? a.T : 0)) * kDownRowsPerCta * sizeof(float) * (a.T == 1 ? kWarps : 1);
  const dim3 g2((a.H + kDownRowsPerCta - 1) / kDownRowsPerCta);
  if (TC == 1 && a.tr)
    return launch_k(ffn_down_combine_kernel<FMT, 1, true>, g2, dim3(kThreads), smem, st, a.pdl != 0, a);
  return launch_k(ffn_down_combine_kernel<FMT, TC, false>, g2, dim3(kThreads), smem, st, a.pdl != 0, a);
}

// Largest dynamic shared memory of a down launch: ys of kMaxPairs pairs.
constexpr int kDownSmemMax = kMaxPairs * kDownRowsPerCta * (int)sizeof(float);

template <int FMT, int TC, bool TR = false>
cudaError_t down_attr() {
  return cudaFuncSetAttribute(ffn_down_combine_kernel<FMT, TC, TR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kDownSmemMax);
}

template <int FMT>
cudaError_t launch_fmt(const FfnArgs& a, int phase, cudaStream_t st) {
  if (a.T >= 8) return launch_tc<FMT, 8>(a, phase, st);
  if (a.T >= 4) return launch_tc<FMT, 4>(a, phase, st);
  if (a.T >= 2) return launch_tc<FMT, 2>(a, phase, st);
  return launch_tc<FMT, 1>(a, phase, st);
}

}  // namespace

cudaError_t ffn_init_attributes() {
  cudaError_t e = cudaSuccess;
  for (cudaError_t r : {down_attr<0, 1>(), down_attr<0, 2>(), down_attr<0, 4>(), down_attr<0, 8>(),
                        down_attr<1, 1>(), down_attr<1, 2>(), down_attr<1, 4>(), down_attr<1, 8>(),
                        down_attr<0, 1, true>(), down_attr<1, 1, true>()})
    if (e == cudaSuccess) e = r;
  return e;
}

cudaError_t launch_grouped_ffn_phase(const FfnArgs& a, int phase, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  if (a.T * a.k + (a.shared ? a.T : 0) > kMaxPairs) return cudaErrorInvalidValue;
  if (a.fmt == 1) {
    if (a.H % 128 != 0 || a.I % 128 != 0) return cudaErrorInvalidValue;
    return launch_fmt<1>(a, phase, st);
  }
  return launch_fmt<0>(a, phase, st);
}

cudaError_t launch_grouped_ffn(const FfnArgs& a, cudaStream_t st) {
  cudaError_t e = launch_grouped_ffn_phase(a, 0, st);
  return e != cudaSuccess ? e : launch_grouped_ffn_phase(a, 1, st);
}

}  // namespace moe
