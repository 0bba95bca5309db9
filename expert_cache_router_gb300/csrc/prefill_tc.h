// Tensor-core (tcgen05) grouped GEMM of the prefill path.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

struct TcGemmArgs {
  const int32_t* counts;   // rows per bucket [G]
  const int32_t* offsets;  // first row of each bucket [G+1]
  const int32_t* tiles;    // first 128-row tile of each bucket [G+1]
  int G, K, I, H;
  int cb;                  // column blocks of this GEMM (grid x)
  const int32_t* perm;     // bucket-order row -> pair
  uint16_t* hp;            // [Tk, I] bf16 (gate/up output)
  float* y;                // [Tk, H] fp32, by pair (down output)
  uint32_t* status;
  // Early down: gate/up CTAs count themselves into tile_done[tile] once their h rows
  // are written; a down CTA starts under the gate/up launch and loads its tile's h
  // rows once the count reaches tile_need. nullptr: the down launch follows gate/up.
  uint32_t* tile_done;
  uint32_t tile_need;
  unsigned long long wait_ns;  // bound of the tile-count wait (0: kDefaultWaitNs)
};

struct TcPrefillArgs {
  const uint16_t* x;       // [T, H]
  const int32_t* perm;     // [Tk]
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* tiles;
  int Tk, k, G, H, I;
  int Tr;                  // routed pairs (token p / k); pairs Tr.. are shared-expert pairs (token p - Tr)
  const uint16_t* w13;     // [G, 2I, H]
  const uint16_t* w2;      // [G, H, I]
  uint16_t* xp;            // [Tk, H] scratch: x rows in bucket order
  uint16_t* hp;            // [Tk, I] scratch
  float* y;                // [Tk, H]
  uint32_t* status;
  uint32_t* tile_done;     // [ceil(Tk/128) + G] scratch, zeroed here each call; nullptr: no early down
  unsigned long long wait_ns;  // bound of the down CTAs' tile-count wait (0: the 2 s default)
  int stall;                   // debug: the tile-count target is one gate/up CTA above the tile's
  cudaEvent_t ev_gemm_begin;  // recorded before the gate/up launch (nullptr: none)
  cudaEvent_t ev_gemm_end;    // recorded after the down launch (nullptr: none)
};

bool tc_gemm_supported(int H, int I);
int tc_gemm_tile_rows();
cudaError_t tc_gemm_init_attributes();
cudaError_t launch_tc_prefill(const TcPrefillArgs& a, cudaStream_t st);

}  // namespace moe
