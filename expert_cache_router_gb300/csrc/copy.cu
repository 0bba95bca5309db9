// Miss copy: the experts the last slot_ensure installed are copied from mapped
// host memory into their slots by SM loads ("MoE expert offload" page, "How it
// works": a second kernel copies the missing experts straight from device-mapped
// pinned host memory; it reads the miss count from device memory, so the launch
// shape is fixed and decode needs no host synchronisation).
//
// The installed experts form one virtual array of 16-byte units
// (expert i's W13 units, then its W2 units, for i = 0..installs-1). A fixed,
// persistent grid walks it with a grid-wide stride, eight independent 16-byte
// loads in flight per thread before their stores, so the host link sees a deep
// queue of coalesced reads. With no installs the kernel exits after reading the
// count.
#include <stdint.h>

#include "kernels.h"

namespace moe {
namespace {

constexpr int kThreads = 512;
constexpr int kUnroll = 8;

__global__ void __launch_bounds__(kThreads)
miss_copy_kernel(LayerWeights lw, const int32_t* __restrict__ counts, int count_idx,
                 const int32_t* __restrict__ miss_expert, const int32_t* __restrict__ miss_slot,
                 int E, int S, unsigned long long u13, unsigned long long u2, unsigned long long f13,
                 unsigned long long f2, uint32_t* status) {
  const int n = counts[count_idx];
  if (n <= 0) return;
  if (n > S) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, kDevBadCount);
    return;
  }
  const unsigned long long upe = u13 + u2;
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  const unsigned long long u0 = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
  // FP8 block scales (a few hundred bytes per expert), 4 bytes at a time
  if (f13 + f2 > 0) {
    const unsigned long long fpe = f13 + f2;
    for (unsigned long long v = u0; v < (unsigned long long)n * fpe; v += stride) {
      const int i = (int)(v / fpe);
      const unsigned long long o = v - (unsigned long long)i * fpe;
      const int e = miss_expert[i], s = miss_slot[i];
      if ((unsigned)e >= (unsigned)E || (unsigned)s >= (unsigned)S) continue;
      if (o < f13) lw.slot_s13[(size_t)s * f13 + o] = lw.host_s13[(size_t)e * f13 + o];
      else lw.slot_s2[(size_t)s * f2 + (o - f13)] = lw.host_s2[(size_t)e * f2 + (o - f13)];
    }
  }
  if (u0 >= (unsigned long long)n * upe) return;
  int i = (int)(u0 / upe);
  unsigned long long off = u0 - (unsigned long long)i * upe;
  const uint4* hw13 = reinterpret_cast<const uint4*>(lw.host_w13);
  const uint4* hw2 = reinterpret_cast<const uint4*>(lw.host_w2);
  uint4* sw13 = reinterpret_cast<uint4*>(lw.slot_w13);
  uint4* sw2 = reinterpret_cast<uint4*>(lw.slot_w2);
  bool bad = false;
  while (i < n) {
    uint4 v[kUnroll];
    uint4* dst[kUnroll];
#pragma unroll
    for (int q = 0; q < kUnroll; ++q) {
      dst[q] = nullptr;
      if (i < n) {
        const int e = miss_expert[i];
        const int s = miss_slot[i];
        if ((unsigned)e < (unsigned)E && (unsigned)s < (unsigned)S) {
          if (off < u13) {
            v[q] = ld_stream(hw13 + (size_t)e * u13 + off);
            dst[q] = sw13 + (size_t)s * u13 + off;
          } else {
            v[q] = ld_stream(hw2 + (size_t)e * u2 + (off - u13));
            dst[q] = sw2 + (size_t)s * u2 + (off - u13);
          }
        } else {
          bad = true;
        }
        off += stride;
        while (off >= upe && i < n) {
          off -= upe;
          ++i;
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kUnroll; ++q)
      if (dst[q]) *dst[q] = v[q];
  }
  if (bad) atomicOr(status, kDevBadCount);
}

// One read of every 16-byte unit (or 4-byte unit, for arrays that are not
// 16-byte aligned and sized) of a mapped host array. The OR of what was read
// goes to *sink so the loads are kept.
__global__ void __launch_bounds__(kThreads)
host_touch_kernel(const uint8_t* __restrict__ p, unsigned long long bytes, int wide, unsigned* sink) {
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  const unsigned long long i0 = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
  unsigned acc = 0;
  if (wide) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
    const unsigned long long n = bytes / 16;
    for (unsigned long long i = i0; i < n; i += stride * kUnroll) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const unsigned long long j = i + u * stride;
        v[u] = j < n ? ld_stream(q + j) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) acc |= v[u].x | v[u].y | v[u].z | v[u].w;
    }
  } else {
    const unsigned* q = reinterpret_cast<const unsigned*>(p);
    const unsigned long long n = bytes / 4;
    for (unsigned long long i = i0; i < n; i += stride) acc |= __ldg(q + i);
  }
  if (acc == 0x5eed5eedu) atomicOr(sink, 1u);  // practically never taken; keeps the loads
}

}  // namespace

cudaError_t launch_host_touch(const void* p, unsigned long long bytes, unsigned* sink, int grid, cudaStream_t st) {
  if (bytes == 0) return cudaSuccess;
  const int wide = ((reinterpret_cast<uintptr_t>(p) & 15u) == 0 && bytes % 16 == 0) ? 1 : 0;
  if (!wide && ((reinterpret_cast<uintptr_t>(p) & 3u) != 0 || bytes % 4 != 0)) return cudaErrorInvalidValue;
  host_touch_kernel<<<grid, kThreads, 0, st>>>(static_cast<const uint8_t*>(p), bytes, wide, sink);
  return cudaGetLastError();
}

cudaError_t launch_miss_copy(const CopyArgs& a, int grid, cudaStream_t st) {
  if (a.count_idx < 0 || a.count_idx >= kNumCounts) return cudaErrorInvalidValue;
  miss_copy_kernel<<<grid, kThreads, 0, st>>>(a.lw, a.counts, a.count_idx, a.miss_expert, a.miss_slot, a.E,
                                              a.S, a.u13, a.u2, a.f13, a.f2, a.status);
  return cudaGetLastError();
}

}  // namespace moe
