// Prefill path of the offloaded MoE layer (calls above the graph token bound).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "common.cuh"

namespace moe {

struct PrefillState {
  int cap_pairs = 0;          // T*k capacity of the scratch below
  int cap_T = 0;
  int E = 0, H = 0, I = 0;
  int32_t* ids = nullptr;     // [T,k] routed expert ids
  float* w = nullptr;         // [T,k]
  int32_t* gidx = nullptr;    // [T,k] group index per pair (slot id or expert id)
  float* logits = nullptr;    // [T,E]
  int32_t* perm = nullptr;    // [T*k] pair index by group order
  int32_t* meta = nullptr;    // group counts, offsets, cursors, tile offsets, flags
  uint16_t* hb = nullptr;     // [T*k, I] bf16 SiLU(g)*u, in group order
  uint16_t* xp = nullptr;     // [T*k, H] bf16 x rows in group order (tensor-core path)
  float* yb = nullptr;        // [T*k, H] fp32 expert outputs, by pair
  uint32_t* tile_done = nullptr;  // tensor-core path: per-tile gate/up completion counts (early down)
  // Two whole-layer staging buffers: while one serves a layer's GEMMs, the next
  // layer is staged into the other (speculatively: used if that layer stages too).
  uint16_t* stage_w13[2] = {nullptr, nullptr};  // [E,2I,H]
  uint16_t* stage_w2[2] = {nullptr, nullptr};   // [E,H,I]
  int spec_layer[2] = {-1, -1};   // layer whose copy the buffer holds or is receiving, -1 none
  cudaEvent_t ready[2] = {nullptr, nullptr};  // after the copy into the buffer
  cudaEvent_t freed[2] = {nullptr, nullptr};  // after the last GEMM that read the buffer
  bool freed_recorded[2] = {false, false};
  cudaStream_t stage_stream = nullptr;        // speculative copies
  int* host_distinct = nullptr;   // pinned: distinct experts of the call
  size_t bytes = 0;
  // events of the last call: route start, route end, copy start, copy end, GEMMs end, combine end,
  // and (tensor-core path) before the gate/up launch and after the down launch
  cudaEvent_t ev[8] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  int last_staged = -1;           // 1 staged, 0 slot path, -1 no call yet
  int last_tc = 0;                // the last call ran the tensor-core GEMMs
};

struct PrefillLayer {
  int layer;                       // index of this layer (speculative staging of layer + 1)
  const uint16_t* next_host_w13;   // the next layer's store (nullptr: last layer)
  const uint16_t* next_host_w2;
  // FP8 experts (fmt 1): the store holds e4m3 codes (host_w13_ptr/host_w2_ptr as bytes) and
  // these fp32 block scales; staging dequantises them to bf16 for the bf16 GEMMs.
  int fmt;
  const float* host_s13;
  const float* host_s2;
  const float* next_host_s13;
  const float* next_host_s2;
  // shared expert (device, the handle's format): staged as group E, one pair per token
  int shared;
  const uint8_t* sh_w13;
  const uint8_t* sh_w2;
  const float* sh_s13;
  const float* sh_s2;
  unsigned long long stage_bytes;  // host bytes of one staged layer (statistics)
  LayerWeights lw;
  LayerTables tab;
  const uint16_t* router;
  int E, S, k, H, I, renorm;
  size_t w13_elems, w2_elems;
  const uint16_t* host_w13_ptr;  // device-usable alias of the mapped host store
  const uint16_t* host_w2_ptr;
  unsigned* route_done;
  uint32_t* status;
  int frozen;  // the layer holds a static placement: always stage (its table takes no installs)
  int early_down;  // tensor-core GEMMs: the down launch starts under gate/up (per-tile counts)
  unsigned long long wait_ns;  // bound of that per-tile wait (0: the default)
  int stall;                   // debug: the per-tile wait targets one CTA more than a tile has
};

cudaError_t prefill_init_attributes();
// Staging buffers hold E + extra experts (extra = 1 with a shared expert).
cudaError_t prefill_create(PrefillState* ps, int E, int extra, int H, int I, size_t w13_elems, size_t w2_elems,
                           size_t* dev_bytes);
// Grows the per-call scratch to T tokens (allocates; never under capture).
cudaError_t prefill_reserve(PrefillState* ps, int T, int k, int E, size_t* dev_bytes);
cudaError_t prefill_layer(PrefillState* ps, const PrefillLayer& pl, const uint16_t* x, int T,
                          uint16_t* out, cudaStream_t st, size_t* dev_bytes, std::string* why);
// Forgets the speculative staging (the caller has synchronised the device).
void prefill_forget(PrefillState* ps);
// Times of the last call (route, copy or staging, grouping + GEMMs, combine), in ms.
cudaError_t prefill_times(PrefillState* ps, float* ms4, int* staged);
// Time of the last call's two tensor-core GEMM launches, in ms (cudaErrorInvalidValue when
// the last call did not run them).
cudaError_t prefill_gemm_ms(PrefillState* ps, float* ms);
void prefill_destroy(PrefillState* ps);

}  // namespace moe
