// Prefill path ("MoE expert offload" page, "How it works", Prefill): when a call
// touches more distinct experts than the layer has slots, the whole expert layer
// is copied into a staging buffer (asynchronously, from the pinned mapped store,
// by SM loads — see stage_copy_kernel) and the grouped GEMM runs there; the slot
// table is left alone. Otherwise the call goes through the
// slot table like a decode call. The host learns the distinct count (one
// synchronisation), so this path is never captured in a graph.
//
// Grouped GEMM: the (token, rank) pairs are bucketed by expert (or slot); each
// bucket is a dense GEMM [M_e, H] x [H, 2I] with the SiLU(g)*u epilogue, then
// [M_e, I] x [I, H]; the expert outputs are combined per token in rank order.
// Every output row depends only on its own row of inputs, so the order of the
// pairs inside a bucket never changes a result.
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <string>

#include "kernels.h"
#include "prefill.h"
#include "prefill_tc.h"

namespace moe {
namespace {

constexpr int kMaxGroups = 1024;
// meta layout (int32): counts[G] | offsets[G+1] | cursor[G] | tile_off[G+1]
constexpr int kMetaCounts = 0;
constexpr int kMetaOffsets = kMaxGroups;
constexpr int kMetaCursor = 2 * kMaxGroups + 1;
constexpr int kMetaTiles = 3 * kMaxGroups + 1;
constexpr int kMetaInts = 4 * kMaxGroups + 2;

constexpr int BM = 64;   // pair rows per tile
constexpr int BK = 32;

__global__ void __launch_bounds__(1024) distinct_kernel(const int32_t* __restrict__ ids, int Tk, int E,
                                                        int* host_distinct, uint32_t* status) {
  __shared__ unsigned char present[kMaxGroups];
  __shared__ int total;
  if (threadIdx.x < E) present[threadIdx.x] = 0;
  if (threadIdx.x == 0) total = 0;
  __syncthreads();
  int bad = 0;
  for (int p = threadIdx.x; p < Tk; p += blockDim.x) {
    const int e = ids[p];
    if (e >= 0 && e < E) present[e] = 1;
    else bad = 1;
  }
  __syncthreads();
  if (threadIdx.x < E && present[threadIdx.x]) atomicAdd(&total, 1);
  if (bad) atomicOr(status, kDevBadExpertId);
  __syncthreads();
  if (threadIdx.x == 0) *host_distinct = total;
}

// Whole-layer staging copy by SM loads from mapped host memory. On GB300 the
// copy engine reads cudaHostRegister'ed pageable memory at ~36 GB/s while SM
// loads of the same memory run at the NVLink-C2C rate (~200 GB/s), so the
// pinned async memcpy of the page becomes this grid-stride kernel: two
// contiguous ranges (W13 and W2 of all experts), eight 16-byte loads in
// flight per thread before their stores.
__global__ void __launch_bounds__(512) stage_copy_kernel(const uint4* __restrict__ s13, uint4* __restrict__ d13,
                                                         unsigned long long n13, const uint4* __restrict__ s2,
                                                         uint4* __restrict__ d2, unsigned long long n2) {
  const unsigned long long total = n13 + n2;
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  for (unsigned long long u0 = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; u0 < total;
       u0 += stride * 8) {
    uint4 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const unsigned long long u = u0 + q * stride;
      if (u < total) v[q] = ld_stream(u < n13 ? s13 + u : s2 + (u - n13));
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const unsigned long long u = u0 + q * stride;
      if (u < total) {
        if (u < n13) d13[u] = v[q];
        else d2[u - n13] = v[q];
      }
    }
  }
}

__global__ void stage_stats_kernel(unsigned long long* stats, unsigned long long bytes) {
  stats[kStatStagedCalls] += 1ull;
  stats[kStatStagedBytes] += bytes;
}

// Staging of FP8 experts: nexp matrices [rows, cols] of e4m3 codes with fp32 scales
// [rows/128, cols/128] each become bf16 matrices: bf16(f32(code) * scale), round to
// nearest even. Sixteen codes (one 16-byte load, inside one 128-column block) a step.
__global__ void __launch_bounds__(512) stage_dequant_kernel(const uint8_t* __restrict__ q,
                                                            const float* __restrict__ sc, int nexp, int rows,
                                                            int cols, uint16_t* __restrict__ dst) {
  const unsigned long long per = (unsigned long long)rows * cols / 16;  // 16-code units per expert
  const unsigned long long total = per * nexp;
  const int cb = cols >> 7, units_per_row = cols >> 4;
  for (unsigned long long u = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; u < total;
       u += (unsigned long long)gridDim.x * blockDim.x) {
    const unsigned long long e = u / per, r0 = u - e * per;
    const int r = (int)(r0 / units_per_row), c = (int)(r0 - (unsigned long long)r * units_per_row) * 16;
    const uint4 w = ld_stream(q + u * 16);
    const float s = __ldg(sc + e * (unsigned long long)(rows >> 7) * cb + (r >> 7) * cb + (c >> 7));
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(words[i] & 0xFFFFu), __NV_E4M3);
      const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(words[i] >> 16), __NV_E4M3);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
      const __nv_bfloat162 pa = __floats2bfloat162_rn(a.x * s, a.y * s);
      const __nv_bfloat162 pb = __floats2bfloat162_rn(b.x * s, b.y * s);
      o[2 * i] = *reinterpret_cast<const uint32_t*>(&pa);
      o[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&pb);
    }
    uint4* d = reinterpret_cast<uint4*>(dst + u * 16);
    d[0] = make_uint4(o[0], o[1], o[2], o[3]);
    d[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// Group index of every pair with a shared expert: the routed pairs keep their expert,
// token t's shared pair (Tk + t) goes to group E.
__global__ void shared_pairs_kernel(const int32_t* __restrict__ ids, int Tk, int T, int E, int32_t* __restrict__ gidx) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p < Tk) gidx[p] = ids[p];
  else if (p < Tk + T) gidx[p] = E;
}

__global__ void group_count_kernel(const int32_t* __restrict__ gidx, int Tk, int G, int32_t* meta) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p < Tk) {
    const int g = gidx[p];
    if (g >= 0 && g < G) atomicAdd(meta + kMetaCounts + g, 1);
  }
}

// One CTA: bucket offsets and tile offsets (exclusive scans over G <= 1024 groups)
// for tiles of bm rows.
__global__ void __launch_bounds__(1024) group_scan_kernel(int G, int bm, int32_t* meta) {
  __shared__ int a[kMaxGroups], b[kMaxGroups];
  const int g = threadIdx.x;
  const int c = g < G ? meta[kMetaCounts + g] : 0;
  a[g] = c;
  b[g] = (c + bm - 1) / bm;
  __syncthreads();
  for (int o = 1; o < kMaxGroups; o <<= 1) {
    const int av = g >= o ? a[g - o] : 0, bv = g >= o ? b[g - o] : 0;
    __syncthreads();
    a[g] += av;
    b[g] += bv;
    __syncthreads();
  }
  if (g < G) {
    meta[kMetaOffsets + g + 1] = a[g];
    meta[kMetaTiles + g + 1] = b[g];
    meta[kMetaCursor + g] = 0;
  }
  if (g == 0) {
    meta[kMetaOffsets] = 0;
    meta[kMetaTiles] = 0;
  }
}

__global__ void group_place_kernel(const int32_t* __restrict__ gidx, int Tk, int G, int32_t* meta,
                                   int32_t* __restrict__ perm) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p < Tk) {
    const int g = gidx[p];
    if (g >= 0 && g < G) perm[meta[kMetaOffsets + g] + atomicAdd(meta + kMetaCursor + g, 1)] = p;
  }
}

// Tile t -> (group, first row); returns false for tiles past the last group's.
__device__ bool find_tile(const int32_t* meta, int G, int t, int* g_out, int* m0, int* rows) {
  const int* tiles = meta + kMetaTiles;
  if (t >= tiles[G]) return false;
  int lo = 0, hi = G - 1;
  while (lo < hi) {  // largest g with tiles[g] <= t
    const int mid = (lo + hi + 1) >> 1;
    if (tiles[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  // skip empty groups that share the same tile offset
  while (lo + 1 <= G - 1 && tiles[lo + 1] <= t) ++lo;
  const int g = lo;
  *g_out = g;
  *m0 = (t - tiles[g]) * BM;
  *rows = min(BM, meta[kMetaCounts + g] - *m0);
  return *rows > 0;
}

__device__ __forceinline__ void unpack8(const uint4 v, float* f) {
  f[0] = bf16lo(v.x); f[1] = bf16hi(v.x); f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  f[4] = bf16lo(v.z); f[5] = bf16hi(v.z); f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

// GEMM 1: rows = pairs of one bucket (x of their token), cols = 32 gate rows and
// the 32 matching up rows of W13; epilogue h = silu(g) * u stored as bf16.
__global__ void __launch_bounds__(256)
gemm_gate_up_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm,
                    const int32_t* __restrict__ meta, int G, const uint16_t* __restrict__ w13_base,
                    size_t w13_elems, int k, int Tr, int H, int I, uint16_t* __restrict__ hb) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][64 + 4];
  int g, m0, rows;
  if (!find_tile(meta, G, blockIdx.x, &g, &m0, &rows)) return;
  const int pos0 = meta[kMetaOffsets + g] + m0;
  const int i0 = blockIdx.y * 32;
  const uint16_t* W = w13_base + (size_t)g * w13_elems;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int lr = tid >> 2, lk = (tid & 3) * 8;
  const int pair = lr < rows ? perm[pos0 + lr] : -1;
  // routed pair p is token p / k; pair Tr + t (shared expert) is token t
  const uint16_t* arow = pair >= 0 ? x + (size_t)(pair < Tr ? pair / k : pair - Tr) * H : nullptr;
  const int wr = lr < 32 ? i0 + lr : I + i0 + (lr - 32);
  const uint16_t* brow = W + (size_t)wr * H;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += BK) {
    float fa[8], fb[8];
    if (arow) unpack8(*reinterpret_cast<const uint4*>(arow + k0 + lk), fa);
    else for (int q = 0; q < 8; ++q) fa[q] = 0.0f;
    unpack8(*reinterpret_cast<const uint4*>(brow + k0 + lk), fb);
    for (int q = 0; q < 8; ++q) {
      As[lk + q][lr] = fa[q];
      Bs[lk + q][lr] = fb[q];
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float av[4], bv[4];
      for (int r = 0; r < 4; ++r) av[r] = As[kk][ty * 4 + r];
      bv[0] = Bs[kk][tx * 2];
      bv[1] = Bs[kk][tx * 2 + 1];
      bv[2] = Bs[kk][32 + tx * 2];
      bv[3] = Bs[kk][32 + tx * 2 + 1];
      for (int r = 0; r < 4; ++r)
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
    }
    __syncthreads();
  }
  for (int r = 0; r < 4; ++r) {
    const int row = ty * 4 + r;
    if (row >= rows) continue;
    for (int c = 0; c < 2; ++c) {
      const float gs = acc[r][c], us = acc[r][2 + c];
      const float h = gs / (1.0f + expf(-gs)) * us;
      const __nv_bfloat16 b = __float2bfloat16_rn(h);
      hb[(size_t)(pos0 + row) * I + i0 + tx * 2 + c] = *reinterpret_cast<const uint16_t*>(&b);
    }
  }
}

// GEMM 2: rows = the bucket's h rows, cols = 64 rows of W2; fp32 y scattered by pair.
__global__ void __launch_bounds__(256)
gemm_down_kernel(const uint16_t* __restrict__ hb, const int32_t* __restrict__ perm,
                 const int32_t* __restrict__ meta, int G, const uint16_t* __restrict__ w2_base,
                 size_t w2_elems, int H, int I, float* __restrict__ yb) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][64 + 4];
  int g, m0, rows;
  if (!find_tile(meta, G, blockIdx.x, &g, &m0, &rows)) return;
  const int pos0 = meta[kMetaOffsets + g] + m0;
  const int n0 = blockIdx.y * 64;
  const uint16_t* W = w2_base + (size_t)g * w2_elems;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int lr = tid >> 2, lk = (tid & 3) * 8;
  const uint16_t* arow = lr < rows ? hb + (size_t)(pos0 + lr) * I : nullptr;
  const uint16_t* brow = W + (size_t)(n0 + lr) * I;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < I; k0 += BK) {
    float fa[8], fb[8];
    if (arow) unpack8(*reinterpret_cast<const uint4*>(arow + k0 + lk), fa);
    else for (int q = 0; q < 8; ++q) fa[q] = 0.0f;
    unpack8(*reinterpret_cast<const uint4*>(brow + k0 + lk), fb);
    for (int q = 0; q < 8; ++q) {
      As[lk + q][lr] = fa[q];
      Bs[lk + q][lr] = fb[q];
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float av[4], bv[4];
      for (int r = 0; r < 4; ++r) av[r] = As[kk][ty * 4 + r];
      for (int c = 0; c < 4; ++c) bv[c] = Bs[kk][tx * 4 + c];
      for (int r = 0; r < 4; ++r)
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
    }
    __syncthreads();
  }
  for (int r = 0; r < 4; ++r) {
    const int row = ty * 4 + r;
    if (row >= rows) continue;
    const int pair = perm[pos0 + row];
    float4 v = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    *reinterpret_cast<float4*>(yb + (size_t)pair * H + n0 + tx * 4) = v;
  }
}

__global__ void combine_kernel(const float* __restrict__ yb, const float* __restrict__ w,
                               const int32_t* __restrict__ gidx, int T, int k, int H, int shared,
                               uint16_t* __restrict__ out) {
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (size_t)T * H) return;
  const int t = (int)(idx / H), n = (int)(idx - (size_t)t * H);
  float acc = 0.0f;
  for (int j = 0; j < k; ++j) {
    if (gidx[t * k + j] < 0) continue;
    acc = __fadd_rn(acc, __fmul_rn(w[t * k + j], yb[(size_t)(t * k + j) * H + n]));
  }
  if (shared) acc = __fadd_rn(acc, yb[((size_t)T * k + t) * H + n]);  // the shared expert, weight 1, last
  const __nv_bfloat16 b = __float2bfloat16_rn(acc);
  out[idx] = *reinterpret_cast<const uint16_t*>(&b);
}

template <typename T>
cudaError_t grow(T** p, size_t count, size_t* bytes) {
  if (*p) cudaFree(*p);
  *p = nullptr;
  void* q = nullptr;
  cudaError_t e = cudaMalloc(&q, count * sizeof(T) + 16);
  if (e == cudaSuccess) {
    *p = static_cast<T*>(q);
    *bytes += count * sizeof(T);
  }
  return e;
}

}  // namespace

cudaError_t prefill_init_attributes() { return tc_gemm_init_attributes(); }

cudaError_t prefill_create(PrefillState* ps, int E, int extra, int H, int I, size_t w13_elems, size_t w2_elems,
                           size_t* dev_bytes) {
  ps->E = E;
  ps->H = H;
  ps->I = I;
  cudaError_t e = cudaSuccess;
  const size_t ne = (size_t)E + (extra > 0 ? extra : 0);
  for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
    e = cudaMalloc(&ps->stage_w13[b], ne * w13_elems * 2);
    if (e == cudaSuccess) e = cudaMalloc(&ps->stage_w2[b], ne * w2_elems * 2);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ps->ready[b], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ps->freed[b], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&ps->stage_stream, cudaStreamNonBlocking);
  if (e != cudaSuccess) return e;
  e = cudaMalloc(&ps->meta, sizeof(int32_t) * kMetaInts);
  if (e != cudaSuccess) return e;
  e = cudaHostAlloc(&ps->host_distinct, sizeof(int), cudaHostAllocMapped);
  if (e != cudaSuccess) return e;
  for (auto& ev : ps->ev)
    if ((e = cudaEventCreate(&ev)) != cudaSuccess) return e;
  ps->bytes = 2 * ne * (w13_elems + w2_elems) * 2 + sizeof(int32_t) * kMetaInts;
  *dev_bytes += ps->bytes;
  return cudaSuccess;
}

cudaError_t prefill_reserve(PrefillState* ps, int T, int k, int E, size_t* dev_bytes) {
  if (T <= ps->cap_T) return cudaSuccess;
  const size_t pairs = (size_t)T * (k + 1);  // routed pairs and one shared-expert pair per token
  cudaError_t e;
  if ((e = grow(&ps->ids, pairs, dev_bytes)) != cudaSuccess) return e;
  if ((e = grow(&ps->w, pairs, dev_bytes)) != cudaSuccess) return e;
  if ((e = grow(&ps->gidx, pairs, dev_bytes)) != cudaSuccess) return e;
  if ((e = grow(&ps->perm, pairs, dev_bytes)) != cudaSuccess) return e;
  if ((e = grow(&ps->logits, (size_t)T * E, dev_bytes)) != cudaSuccess) return e;
  if ((e = grow(&ps->hb, pairs * ps->I, dev_bytes)) != cudaSuccess) return e;
  if ((e = grow(&ps->xp, pairs * ps->H, dev_bytes)) != cudaSuccess) return e;
  if ((e = grow(&ps->yb, pairs * ps->H, dev_bytes)) != cudaSuccess) return e;
  // one counter per 128-row tensor-core tile (tiles <= ceil(pairs / 128) + groups)
  if ((e = grow(&ps->tile_done, (pairs + 127) / 128 + kMaxGroups + 2, dev_bytes)) != cudaSuccess) return e;
  ps->cap_T = T;
  ps->cap_pairs = (int)pairs;
  return cudaSuccess;
}

cudaError_t prefill_layer(PrefillState* ps, const PrefillLayer& pl, const uint16_t* x, int T,
                          uint16_t* out, cudaStream_t st, size_t* dev_bytes, std::string* why) {
  cudaError_t e = prefill_reserve(ps, T, pl.k, pl.E, dev_bytes);
  if (e != cudaSuccess) { *why = "prefill scratch"; return e; }
  const int Tk = T * pl.k;
  cudaEventRecord(ps->ev[0], st);
  RouteArgs ra{};
  ra.x = x; ra.wr = pl.router; ra.T = T; ra.E = pl.E; ra.H = pl.H; ra.k = pl.k;
  ra.renorm = pl.renorm; ra.ids = ps->ids; ra.w = ps->w; ra.logits = ps->logits; ra.done = pl.route_done;
  if ((e = launch_route(ra, st)) != cudaSuccess) { *why = "route"; return e; }
  distinct_kernel<<<1, 1024, 0, st>>>(ps->ids, Tk, pl.E, ps->host_distinct, pl.status);
  if ((e = cudaGetLastError()) != cudaSuccess) { *why = "distinct"; return e; }
  cudaEventRecord(ps->ev[1], st);
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) { *why = "sync"; return e; }
  const int D = *reinterpret_cast<volatile int*>(ps->host_distinct);

  const uint16_t* base13;
  const uint16_t* base2;
  const int32_t* gidx;
  int G;
  cudaEventRecord(ps->ev[2], st);
  // FP8 experts and the shared expert always stage (the GEMMs take bf16 groups of one buffer)
  const bool stage = D > pl.S || pl.frozen || pl.fmt == 1 || pl.shared;
  ps->last_staged = stage ? 1 : 0;
  int used = -1;  // staging buffer this call's GEMMs read
  if (stage) {
    const size_t b13 = (size_t)pl.E * pl.w13_elems * 2, b2 = (size_t)pl.E * pl.w2_elems * 2;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    for (int b = 0; b < 2; ++b)
      if (ps->spec_layer[b] == pl.layer) used = b;
    if (used >= 0) {
      // staged while the previous layer computed: wait for that copy
      if ((e = cudaStreamWaitEvent(st, ps->ready[used], 0)) != cudaSuccess) { *why = "staging wait"; return e; }
    } else {
      used = ps->spec_layer[0] == -1 ? 0 : (ps->spec_layer[1] == -1 ? 1 : 0);
      if (ps->freed_recorded[used] && (e = cudaStreamWaitEvent(st, ps->freed[used], 0)) != cudaSuccess) {
        *why = "staging buffer";
        return e;
      }
      // a speculative copy still writing this buffer is ordered before this one
      if ((e = cudaStreamWaitEvent(st, ps->ready[used], 0)) != cudaSuccess) { *why = "staging buffer"; return e; }
      if (pl.fmt == 1) {
        stage_dequant_kernel<<<2 * sms, 512, 0, st>>>(reinterpret_cast<const uint8_t*>(pl.host_w13_ptr), pl.host_s13,
                                                      pl.E, 2 * pl.I, pl.H, ps->stage_w13[used]);
        stage_dequant_kernel<<<2 * sms, 512, 0, st>>>(reinterpret_cast<const uint8_t*>(pl.host_w2_ptr), pl.host_s2,
                                                      pl.E, pl.H, pl.I, ps->stage_w2[used]);
      } else {
        stage_copy_kernel<<<2 * sms, 512, 0, st>>>(reinterpret_cast<const uint4*>(pl.host_w13_ptr),
                                                   reinterpret_cast<uint4*>(ps->stage_w13[used]), b13 / 16,
                                                   reinterpret_cast<const uint4*>(pl.host_w2_ptr),
                                                   reinterpret_cast<uint4*>(ps->stage_w2[used]), b2 / 16);
      }
      if ((e = cudaGetLastError()) != cudaSuccess) {
        *why = "staging copy";
        return e;
      }
      if ((e = cudaEventRecord(ps->ready[used], st)) != cudaSuccess) { *why = "staging event"; return e; }
    }
    ps->spec_layer[used] = -1;
    stage_stats_kernel<<<1, 1, 0, st>>>(pl.tab.stats, pl.stage_bytes);
    if (pl.shared) {  // the shared expert is group E of the buffer
      if (pl.fmt == 1) {
        stage_dequant_kernel<<<sms, 512, 0, st>>>(pl.sh_w13, pl.sh_s13, 1, 2 * pl.I, pl.H,
                                                  ps->stage_w13[used] + (size_t)pl.E * pl.w13_elems);
        stage_dequant_kernel<<<sms, 512, 0, st>>>(pl.sh_w2, pl.sh_s2, 1, pl.H, pl.I,
                                                  ps->stage_w2[used] + (size_t)pl.E * pl.w2_elems);
        e = cudaGetLastError();
      } else {
        e = cudaMemcpyAsync(ps->stage_w13[used] + (size_t)pl.E * pl.w13_elems, pl.sh_w13, pl.w13_elems * 2,
                            cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess)
          e = cudaMemcpyAsync(ps->stage_w2[used] + (size_t)pl.E * pl.w2_elems, pl.sh_w2, pl.w2_elems * 2,
                              cudaMemcpyDeviceToDevice, st);
      }
      if (e != cudaSuccess) { *why = "shared expert staging"; return e; }
    }
    // Speculative staging of the next layer into the other buffer, on the staging
    // stream: after this layer's copy (one stream on the host link at a time) and
    // after the last GEMM that read the other buffer. SM loads, not the copy engine:
    // on GB300 the copy engine read this store at 85-117 GB/s after runs of other
    // host copies (200 GB/s in a fresh process), SM loads at ~150 GB/s or more.
    const int other = 1 - used;
    if (pl.next_host_w13 && pl.next_host_w2) {
      if ((e = cudaStreamWaitEvent(ps->stage_stream, ps->ready[used], 0)) != cudaSuccess ||
          (ps->freed_recorded[other] && (e = cudaStreamWaitEvent(ps->stage_stream, ps->freed[other], 0)) != cudaSuccess) ||
          (e = cudaStreamWaitEvent(ps->stage_stream, ps->ready[other], 0)) != cudaSuccess) {
        *why = "speculative staging";
        return e;
      }
      if (pl.fmt == 1) {
        stage_dequant_kernel<<<2 * sms, 512, 0, ps->stage_stream>>>(
            reinterpret_cast<const uint8_t*>(pl.next_host_w13), pl.next_host_s13, pl.E, 2 * pl.I, pl.H,
            ps->stage_w13[other]);
        stage_dequant_kernel<<<2 * sms, 512, 0, ps->stage_stream>>>(
            reinterpret_cast<const uint8_t*>(pl.next_host_w2), pl.next_host_s2, pl.E, pl.H, pl.I, ps->stage_w2[other]);
        e = cudaGetLastError();
      } else {
        stage_copy_kernel<<<2 * sms, 512, 0, ps->stage_stream>>>(
            reinterpret_cast<const uint4*>(pl.next_host_w13), reinterpret_cast<uint4*>(ps->stage_w13[other]),
            b13 / 16, reinterpret_cast<const uint4*>(pl.next_host_w2), reinterpret_cast<uint4*>(ps->stage_w2[other]),
            b2 / 16);
        e = cudaGetLastError();
      }
      if (e != cudaSuccess || (e = cudaEventRecord(ps->ready[other], ps->stage_stream)) != cudaSuccess) {
        *why = "speculative staging";
        return e;
      }
      ps->spec_layer[other] = pl.layer + 1;
    }
    base13 = ps->stage_w13[used];
    base2 = ps->stage_w2[used];
    gidx = ps->ids;
    G = pl.E;
    if (pl.shared) {
      shared_pairs_kernel<<<(Tk + T + 255) / 256, 256, 0, st>>>(ps->ids, Tk, T, pl.E, ps->gidx);
      gidx = ps->gidx;
      G = pl.E + 1;
    }
  } else {
    EnsureArgs ea{};
    ea.tab = pl.tab; ea.ids = ps->ids; ea.Tk = Tk; ea.E = pl.E; ea.S = pl.S; ea.slot_ids = ps->gidx;
    ea.status = pl.status; ea.expert_bytes = (unsigned long long)(pl.w13_elems + pl.w2_elems) * 2ull;
    if ((e = launch_slot_ensure(ea, st)) != cudaSuccess) { *why = "slot ensure"; return e; }
    CopyArgs ca{};
    ca.lw = pl.lw; ca.counts = pl.tab.counts; ca.miss_expert = pl.tab.miss_expert;
    ca.miss_slot = pl.tab.miss_slot; ca.E = pl.E; ca.S = pl.S;
    ca.u13 = pl.w13_elems * 2 / 16; ca.u2 = pl.w2_elems * 2 / 16; ca.status = pl.status;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if ((e = launch_miss_copy(ca, 2 * sms, st)) != cudaSuccess) { *why = "miss copy"; return e; }
    base13 = reinterpret_cast<const uint16_t*>(pl.lw.slot_w13);
    base2 = reinterpret_cast<const uint16_t*>(pl.lw.slot_w2);
    gidx = ps->gidx;
    G = pl.S;
  }
  cudaEventRecord(ps->ev[3], st);
  if ((e = cudaMemsetAsync(ps->meta, 0, sizeof(int32_t) * kMetaInts, st)) != cudaSuccess) {
    *why = "meta";
    return e;
  }
  const bool tc = tc_gemm_supported(pl.H, pl.I);
  ps->last_tc = tc ? 1 : 0;
  const int P = Tk + (stage && pl.shared ? T : 0);  // pairs: routed, then one shared-expert pair per token
  group_count_kernel<<<(P + 255) / 256, 256, 0, st>>>(gidx, P, G, ps->meta);
  group_scan_kernel<<<1, kMaxGroups, 0, st>>>(G, tc ? tc_gemm_tile_rows() : BM, ps->meta);
  group_place_kernel<<<(P + 255) / 256, 256, 0, st>>>(gidx, P, G, ps->meta, ps->perm);
  if (tc) {
    // tensor-core path: tcgen05 grouped GEMMs over the bucket-ordered rows
    TcPrefillArgs ta{};
    ta.x = x; ta.perm = ps->perm; ta.counts = ps->meta + kMetaCounts; ta.offsets = ps->meta + kMetaOffsets;
    ta.tiles = ps->meta + kMetaTiles; ta.Tk = P; ta.k = pl.k; ta.Tr = Tk; ta.G = G; ta.H = pl.H; ta.I = pl.I;
    ta.w13 = base13; ta.w2 = base2; ta.xp = ps->xp; ta.hp = ps->hb; ta.y = ps->yb; ta.status = pl.status;
    ta.tile_done = pl.early_down ? ps->tile_done : nullptr;
    ta.wait_ns = pl.wait_ns;
    ta.stall = pl.stall;
    ta.ev_gemm_begin = ps->ev[6];
    ta.ev_gemm_end = ps->ev[7];
    if ((e = launch_tc_prefill(ta, st)) != cudaSuccess) { *why = "tensor-core grouped GEMM"; return e; }
  } else {
    // shapes the 128x256 tensor-core tiling does not cover: CUDA-core tiles
    const int max_tiles = (P + BM - 1) / BM + G;
    gemm_gate_up_kernel<<<dim3(max_tiles, pl.I / 32), 256, 0, st>>>(x, ps->perm, ps->meta, G, base13,
                                                                     pl.w13_elems, pl.k, Tk, pl.H, pl.I, ps->hb);
    gemm_down_kernel<<<dim3(max_tiles, pl.H / 64), 256, 0, st>>>(ps->hb, ps->perm, ps->meta, G, base2,
                                                                  pl.w2_elems, pl.H, pl.I, ps->yb);
  }
  cudaEventRecord(ps->ev[4], st);
  const size_t n = (size_t)T * pl.H;
  combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(ps->yb, ps->w, gidx, T, pl.k, pl.H,
                                                              stage && pl.shared ? 1 : 0, out);
  if ((e = cudaGetLastError()) != cudaSuccess) { *why = "grouped GEMM"; return e; }
  if (used >= 0) {
    if ((e = cudaEventRecord(ps->freed[used], st)) != cudaSuccess) { *why = "staging event"; return e; }
    ps->freed_recorded[used] = true;
  }
  cudaEventRecord(ps->ev[5], st);
  return cudaSuccess;
}

cudaError_t prefill_gemm_ms(PrefillState* ps, float* ms) {
  if (ps->last_staged < 0 || !ps->last_tc) return cudaErrorInvalidValue;
  cudaError_t e = cudaEventSynchronize(ps->ev[7]);
  return e != cudaSuccess ? e : cudaEventElapsedTime(ms, ps->ev[6], ps->ev[7]);
}

cudaError_t prefill_times(PrefillState* ps, float* ms4, int* staged) {
  *staged = ps->last_staged;
  if (ps->last_staged < 0) return cudaErrorInvalidValue;
  cudaError_t e = cudaEventSynchronize(ps->ev[5]);
  if (e != cudaSuccess) return e;
  const int from[4] = {0, 2, 3, 4}, to[4] = {1, 3, 4, 5};
  for (int i = 0; i < 4; ++i)
    if ((e = cudaEventElapsedTime(&ms4[i], ps->ev[from[i]], ps->ev[to[i]])) != cudaSuccess) return e;
  return cudaSuccess;
}

void prefill_forget(PrefillState* ps) {
  ps->spec_layer[0] = ps->spec_layer[1] = -1;
}

void prefill_destroy(PrefillState* ps) {
  if (ps->stage_stream) cudaStreamSynchronize(ps->stage_stream);
  cudaFree(ps->ids); cudaFree(ps->w); cudaFree(ps->gidx); cudaFree(ps->perm); cudaFree(ps->logits);
  cudaFree(ps->hb); cudaFree(ps->xp); cudaFree(ps->yb); cudaFree(ps->meta); cudaFree(ps->tile_done);
  for (int b = 0; b < 2; ++b) {
    cudaFree(ps->stage_w13[b]);
    cudaFree(ps->stage_w2[b]);
    if (ps->ready[b]) cudaEventDestroy(ps->ready[b]);
    if (ps->freed[b]) cudaEventDestroy(ps->freed[b]);
  }
  if (ps->stage_stream) cudaStreamDestroy(ps->stage_stream);
  if (ps->host_distinct) cudaFreeHost(ps->host_distinct);
  for (auto& ev : ps->ev)
    if (ev) cudaEventDestroy(ev);
  *ps = PrefillState();
}

}  // namespace moe
