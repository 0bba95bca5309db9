// Shared device helpers and the per-layer device state of the offloaded MoE library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {

// Device status bits (mirror the MOE_DEV_* values of the public header).
constexpr uint32_t kDevBadExpertId = 1u << 0;
constexpr uint32_t kDevBadSlotId = 1u << 1;
constexpr uint32_t kDevAuditFailed = 1u << 2;
constexpr uint32_t kDevBadCount = 1u << 3;
constexpr uint32_t kDevTimeout = 1u << 4;

// Per-layer counters kept on the device (indices into LayerTables::stats).
enum StatIdx { kStatCalls = 0, kStatHits, kStatMisses, kStatSpills, kStatBytesCopied,
               kStatStagedCalls, kStatStagedBytes, kStatPrefetchInstalls, kStatPrefetchHits,
               kStatPrefetchBytes, kNumStats };

// Indices into LayerTables::counts (results of the last slot_ensure, and of the
// last prefetch install into this layer).
// kCntFrozen (written by the host only): 1 while the layer holds a static placement.
enum CountIdx { kCntMiss = 0, kCntSpill, kCntInstall, kCntDistinct, kCntPrefetch, kCntCandidates, kCntFrozen,
                kNumCounts };

// Device-resident LRU slot table and miss list of one layer.
struct LayerTables {
  int32_t* slot_expert;   // [S], -1 = empty
  int32_t* expert_slot;   // [E], -1 = not resident
  uint32_t* stamp;        // [S]
  uint32_t* clock;        // [1]
  int32_t* miss_expert;   // [E]: installs first (ascending id), then spills
  int32_t* miss_slot;     // [E]: slot, or S + spill index
  int32_t* counts;        // [kNumCounts]
  unsigned long long* stats;  // [kNumStats]
  int32_t* pf_expert;     // [E]: experts the last prefetch install put in this layer, in install order
  int32_t* pf_slot;       // [E]: their slots
  int32_t* pf_cand;       // [E]: that install's candidates (descending predicted logit)
  unsigned long long* route_counts;  // [E]: routed (token, rank) pairs per expert, cumulative
  int32_t* pair_src;      // [kMaxCallPairs]: per pair of the last ensure, the expert id when it
                          // missed (installed by that call or spilled), else -1
};
constexpr int kMaxCallPairs = 1024;  // T*k of one ensure call

// Where layer l's expert weights live. Weight pointers are byte addresses:
// bf16 experts take 2 bytes per element, FP8 (e4m3) experts 1 byte plus one fp32
// scale per 128 x 128 block.
struct LayerWeights {
  const uint8_t* host_w13;    // device-usable alias of the mapped host array [E,2I,H]
  const uint8_t* host_w2;     // [E,H,I]
  uint8_t* slot_w13;          // [S,2I,H] device
  uint8_t* slot_w2;           // [S,H,I] device
  const float* host_s13;      // FP8: [E, 2I/128, H/128] block scales (mapped host), else nullptr
  const float* host_s2;       // FP8: [E, H/128, I/128]
  float* slot_s13;            // FP8: [S, 2I/128, H/128] device
  float* slot_s2;             // FP8: [S, H/128, I/128]
  const uint8_t* sh_w13;      // always-resident shared expert (device), or nullptr
  const uint8_t* sh_w2;
  const float* sh_s13;        // its FP8 scales
  const float* sh_s2;
};

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// L2 eviction policy for router loads: the routers of all layers (tens of MB)
// are read every decode step and should survive the expert weights streaming
// through L2 (gigabytes per step; an evict-first hint on those measured slower).
__device__ __forceinline__ unsigned long long l2_evict_last() {
  unsigned long long p;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 16-byte read-only load that does not allocate in L1 (streamed weights).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// 16-byte read-only load of router weights: no L1 allocation, kept in L2 across steps.
__device__ __forceinline__ uint4 ld_keep(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(l2_evict_last()));
  return v;
}

// Eight bf16 weights (one uint4) dotted with eight fp32 values, accumulated in order.
__device__ __forceinline__ float dot8(const uint4 w, const float* x, float acc) {
  acc = fmaf(bf16lo(w.x), x[0], acc);
  acc = fmaf(bf16hi(w.x), x[1], acc);
  acc = fmaf(bf16lo(w.y), x[2], acc);
  acc = fmaf(bf16hi(w.y), x[3], acc);
  acc = fmaf(bf16lo(w.z), x[4], acc);
  acc = fmaf(bf16hi(w.z), x[5], acc);
  acc = fmaf(bf16lo(w.w), x[6], acc);
  acc = fmaf(bf16hi(w.w), x[7], acc);
  return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) {
  atomicOr(status, bit);
}

// Programmatic dependent launch. pdl_wait blocks until the preceding kernel of
// the stream has completed and its writes are visible (a no-op when this launch
// did not ask for programmatic serialization); pdl_trigger lets the next kernel
// start launching. Kernels here trigger only after their own wait, so when a
// kernel starts, the kernel two places before it has completed.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Decode trace (moe_offload_trace_enable): per layer, kTraceFields globaltimer
// stamps, each the earliest (trace_min) or latest (trace_max) time a kernel
// passed a point of the step. tr == nullptr: off. Fire-and-forget atomics.
enum TraceField {
  kTrHeadWait = 0,      // head, CTA 0 past its dependency wait
  kTrHeadLogits,        // head, every logit in CTA 0 (after the cluster barrier)
  kTrHeadTopk,          // head, top-k and weights written
  kTrHeadDone,          // head, slot table updated
  kTrGateFirst,         // gate/up, first CTA past its dependency wait        (min)
  kTrGateHostFirst,     // gate/up, first W13 chunk of an installed expert used (min)
  kTrGateHostDone,      // gate/up, last CTA of an installed expert done      (max)
  kTrCopyDone,          // gate/up, last W2-copy CTA done                     (max)
  kTrGateDone,          // gate/up, last CTA done                             (max)
  kTrDownFirst,         // down, first CTA started                            (min)
  kTrDownWaits,         // down, last CTA past its waits                      (max)
  kTrDownDone,          // down, last CTA done (counter resets included)      (max)
  kTrDownOut,           // down, latest CTA past writing its output rows      (max)
  kTraceFields = 16
};
constexpr unsigned kTraceMinFields =
    (1u << kTrGateFirst) | (1u << kTrGateHostFirst) | (1u << kTrDownFirst);  // reset to ~0

__device__ __forceinline__ void trace_min(unsigned long long* tr, int f) {
  if (tr) atomicMin(tr + f, globaltimer_ns());
}
__device__ __forceinline__ void trace_max(unsigned long long* tr, int f) {
  if (tr) atomicMax(tr + f, globaltimer_ns());
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait of one thread until *ctr >= target. Gives up (false) after
// limit_ns, setting kDevTimeout, or at once when an earlier wait already timed out.
__device__ __forceinline__ bool wait_at_least(const uint32_t* ctr, uint32_t target, uint32_t* status,
                                              unsigned long long limit_ns) {
  if (ld_acquire(ctr) >= target) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (ld_acquire(ctr) < target) {
    if (*reinterpret_cast<volatile uint32_t*>(status) & kDevTimeout) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(status, kDevTimeout);
      return false;
    }
    __nanosleep(100);
  }
  return true;
}

}  // namespace moe
