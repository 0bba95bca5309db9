// Launchers of the device kernels (host side, internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "common.cuh"

namespace moe {

// Launch with optional programmatic stream serialization (PDL).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct RouteArgs {
  const uint16_t* x;    // [T,H] bf16
  const uint16_t* wr;   // [E,H] bf16
  int T, E, H, k, renorm;
  int32_t* ids;         // [T,k]
  float* w;             // [T,k]
  float* logits;        // [T,E] scratch
  unsigned* done;       // one counter, zero between launches
};
// Router logits + top-k + weights. Decode-sized T (<= kRouteFuseT) runs as one
// launch (the last CTA does the top-k); larger T adds a top-k launch.
constexpr int kRouteFuseT = 8;
cudaError_t launch_route(const RouteArgs& a, cudaStream_t st);
// Opt-in shared-memory limits; called once per device before the first launch.
cudaError_t route_init_attributes();

// Decode step head in one launch: router logits (one warp per expert), then the
// last CTA to finish runs the top-k of every token and the slot-table update
// (ensure_block). ids/w/slot_ids are [T,k]; T <= kRouteEnsureMaxT.
constexpr int kRouteEnsureMaxT = 64;
struct RouteEnsureArgs {
  RouteArgs r;
  LayerTables tab;
  int S;
  int32_t* slot_ids;
  uint32_t* status;
  unsigned long long expert_bytes;
  int pdl;  // launched with programmatic serialization after the previous kernel
  // Router lookahead into the next layer (pf_n = 0: off): its router on this x,
  // then up to pf_n predicted non-resident experts installed at stamp 0 in tab_next.
  const uint16_t* wr_next;
  LayerTables tab_next;
  int pf_n;
  unsigned long long pf_bytes;  // bytes of one expert (prefetch statistics)
  // scratch of the two-launch lookahead (heads without the in-kernel predictor)
  float* pred_logits;           // [T,E]
  int32_t* pred_ids;            // [T,k]
  float* pred_w;                // [T,k]
  unsigned* pred_done;          // [1], zero between calls
  unsigned long long* tr;       // decode trace of this layer ([kTraceFields]) or nullptr
};
cudaError_t launch_route_ensure(const RouteEnsureArgs& a, cudaStream_t st);
// Router lookahead as its own launches: the next layer's router on x (logits and
// per-token top-k into the scratch), then the prefetch install into tab_next.
cudaError_t launch_lookahead(const uint16_t* x, const uint16_t* wr_next, int T, int E, int H, int k,
                             LayerTables tab_next, int S, int N, unsigned long long bytes, float* pred_logits,
                             int32_t* pred_ids, float* pred_w, unsigned* pred_done, cudaStream_t st);
// The prefetch install alone (one CTA): candidates from predicted ids [T,k] and logits [T,E].
cudaError_t launch_prefetch_install(const int32_t* pred_ids, const float* pred_logits, int T, int k, int E,
                                    LayerTables tab, int S, int N, unsigned long long bytes, cudaStream_t st);

struct EnsureArgs {
  LayerTables tab;
  const int32_t* ids;   // [Tk]
  int Tk, E, S;
  int32_t* slot_ids;    // [Tk]
  uint32_t* status;
  unsigned long long expert_bytes;
};
cudaError_t launch_slot_ensure(const EnsureArgs& a, cudaStream_t st);
// ffn_sync: the FFN's early-down counters to check for zero (between calls), or nullptr.
cudaError_t launch_audit(const LayerTables& tab, int E, int S, uint32_t* status, const uint32_t* ffn_sync,
                         cudaStream_t st);

struct CopyArgs {
  LayerWeights lw;
  const int32_t* counts;
  const int32_t* miss_expert;
  const int32_t* miss_slot;
  int E, S;
  unsigned long long u13, u2;  // 16-byte units per expert of W13 and W2
  unsigned long long f13, f2;  // FP8 block scales per expert (4-byte units), 0 for bf16
  uint32_t* status;
  int count_idx;               // counts[count_idx] experts of the lists are copied (kCntInstall,
                               // or kCntPrefetch with the prefetch lists)
};
cudaError_t launch_miss_copy(const CopyArgs& a, int grid, cudaStream_t st);
// Reads every byte of a mapped host array once from the GPU (p 4-byte aligned, bytes a multiple of 4).
cudaError_t launch_host_touch(const void* p, unsigned long long bytes, unsigned* sink, int grid, cudaStream_t st);

struct FfnArgs {
  LayerWeights lw;
  const uint16_t* x;        // [T,H]
  const int32_t* slot_ids;  // [T,k]: slot, or S + spill index
  const float* w;           // [T,k]
  int T, k, H, I, E, S;
  const int32_t* counts;    // layer counts (spill resolution)
  const int32_t* miss_expert;
  float* hbuf;              // [T*k (+T with a shared expert), I] scratch
  uint16_t* out;            // [T,H]
  uint32_t* status;
  int copy_through;         // 1: fill the slots the current call installed (no separate copy)
  const int32_t* miss_slot; // layer miss list slots (copy-through)
  int pdl;                  // launched with programmatic serialization after the previous kernel
  const int32_t* pair_src;  // per pair: expert id when installed or spilled by the ensure behind
                            // slot_ids (host source), else -1; nullptr: no spills, no copy-through
  int fmt;                  // 0: bf16 experts, 1: FP8 e4m3 experts with 128x128 block scales
  int shared;               // 1: add the shared expert (lw.sh_*) to every token, weight 1, after the k ranks
  uint32_t* sync;           // early down: [kFfnSyncWords] zeroed counters, or nullptr (down waits for
                            // the whole gate/up grid)
  unsigned long long* tr;    // decode trace of this layer ([kTraceFields]) or nullptr
  unsigned long long wait_ns;  // bound of one early-down wait (0: kDefaultWaitNs)
  int stall;                // debug: the first group's wait of every down warp targets one CTA more
                            // than its column has, so it runs out (tests of the bounded wait)
};
// Counters of the early-down hand-off of a decode step, one 128-byte line each
// (so that pollers of different counters do not queue on one L2 line): line
// c < 1025 counts the finished gate/up CTAs of column c (pair, or the shared
// expert); then the finished W2-copy CTAs and the finished down CTAs. All are
// zero between calls; the last down CTA resets them.
constexpr int kSyncLine = 32;  // words per line
constexpr int kSyncColumns = 1025;
constexpr int kSyncCopyLine = kSyncColumns;
constexpr int kSyncDoneLine = kSyncColumns + 1;
constexpr int kFfnSyncWords = (kSyncDoneLine + 1) * kSyncLine;
constexpr int kDownRowsPerCta = 8;  // output rows per CTA of the down + combine launch
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // bound of one early-down wait
cudaError_t launch_grouped_ffn(const FfnArgs& a, cudaStream_t st);
// Opt the down launch into the dynamic shared memory of its largest calls (T*k up to 1024 pairs);
// once per device, before the first launch with more than 64 pairs.
cudaError_t ffn_init_attributes();
// One of the two launches of launch_grouped_ffn: phase 0 gate/up (+ copy-through), 1 down + combine.
cudaError_t launch_grouped_ffn_phase(const FfnArgs& a, int phase, cudaStream_t st);

// Sets the reason moe_offload_last_error(NULL) returns (calls that take no handle).
void set_handleless_error(const char* msg);

}  // namespace moe
