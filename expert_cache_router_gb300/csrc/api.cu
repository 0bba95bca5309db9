// C ABI of the offloaded MoE layer: handle life cycle, memory ownership and the
// launch sequence of each entry point. See include/moe_offload.h for the contract.
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/moe_offload.h"
#include "kernels.h"
#include "prefill.h"

using namespace moe;

struct moe_offload {
  moe_offload_config_t cfg{};
  int device = 0;
  int sm_count = 0;
  std::string err;
  size_t dev_bytes = 0;

  size_t w13_elems = 0, w2_elems = 0;  // per expert
  int fmt = 0;                         // 0 bf16, 1 FP8 e4m3 with 128 x 128 block scales
  size_t e13_bytes = 0, e2_bytes = 0;  // weight bytes per expert
  size_t f13 = 0, f2 = 0;              // fp32 block scales per expert (FP8 only)
  std::vector<int> shared_set;         // per layer: shared expert installed
  std::vector<int> frozen;             // per layer: static placement installed (host mirror)
  std::vector<void*> registered;       // host ranges this handle registered
  std::vector<LayerWeights> lw;
  std::vector<LayerTables> tab;
  std::vector<const uint16_t*> router;
  std::vector<void*> allocations;

  // decode scratch (T <= max_tokens_graph)
  int32_t* ids_buf = nullptr;
  float* w_buf = nullptr;
  int32_t* slot_buf = nullptr;
  float* logits = nullptr;
  float* hbuf = nullptr;
  unsigned* route_done = nullptr;  // [L]
  uint32_t* status = nullptr;
  int copy_grid = 0;
  int pdl = 1;  // programmatic dependent launch in the decode chain (env MOE_OFFLOAD_PDL=0 turns it off)
  int audit_each = 0;  // env MOE_OFFLOAD_AUDIT=1: audit a layer's table after every update of it
  int early_down = 1;  // env MOE_OFFLOAD_EARLY_DOWN=0: the down launch (decode and prefill) waits for the whole gate/up grid
  unsigned long long* trace = nullptr;  // [L, kTraceFields] decode trace records (moe_offload_trace_enable)
  int trace_on = 0;
  uint32_t* ffn_sync = nullptr;  // [kFfnSyncWords] counters of the early-down hand-off
  int last_tk = 0;               // T * k of the last decode-path call (ids_buf, w_buf, slot_buf)
  // Bound of the early-down waits, and the debug stall that plants a target no
  // counter reaches (moe_offload_debug_wait).
  unsigned long long wait_ns = kDefaultWaitNs;
  int stall = 0;
  size_t auto_free = 0;          // num_slots = 0 at create: free device bytes the sizing saw

  // Eager decode profile (env MOE_OFFLOAD_PROFILE=1): events before the head, after the head,
  // after gate/up and after down of every decode_layer call outside stream capture; folded into
  // per-layer sums when read (or when many are pending) and printed at destroy.
  struct ProfileRec {
    int layer;
    std::array<cudaEvent_t, 4> ev;
  };
  int profile = 0;
  std::vector<ProfileRec> prof_pending;
  std::vector<cudaEvent_t> prof_pool;
  std::vector<std::array<double, 4>> prof_sum;  // per layer: calls, head, gate/up, down (ms)
  // Host-side fault injection (env MOE_OFFLOAD_FAIL_ALLOC=n): create's n-th allocation
  // (device allocation or host registration, counted from 0) reports out-of-memory
  // without being attempted. -1 = off.
  int fail_alloc_at = -1;
  int alloc_seq = 0;

  // Router lookahead (cfg.prefetch_n > 0): the copies of prefetched experts run on
  // a high-priority stream; layer l's copy is joined before layer l's FFN.
  cudaStream_t pf_stream = nullptr;
  std::vector<cudaEvent_t> pf_ready, pf_done;  // per layer receiving a prefetch
  std::vector<int> pf_pending;                 // 0: none, 1: issued eagerly, 2: issued under capture
  float* pred_logits = nullptr;                // scratch of the two-launch lookahead
  int32_t* pred_ids = nullptr;
  float* pred_w = nullptr;
  unsigned* pred_done = nullptr;
  int pf_grid = 32;                            // CTAs of a prefetch copy (leaves the SMs to the FFN)

  PrefillState prefill;
};

namespace {

thread_local std::string g_create_error;
constexpr size_t kAutoReserveBytes = (size_t)5 << 29;  // 2.5 GiB, the page's default reserve

moe_status_t fail(moe_offload* h, moe_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (h) h->err = buf;
  else g_create_error = buf;
  return st;
}

moe_status_t cuda_fail(moe_offload* h, cudaError_t e, const char* what) {
  moe_status_t st = (e == cudaErrorMemoryAllocation) ? MOE_ERR_OOM : MOE_ERR_CUDA;
  return fail(h, st, "%s: %s", what, cudaGetErrorString(e));
}

#define CK(h, call)                                        \
  do {                                                     \
    cudaError_t e_ = (call);                               \
    if (e_ != cudaSuccess) return cuda_fail((h), e_, #call); \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// What one slot holds: the expert's weights and, for FP8, its block scales.
unsigned long long slot_bytes(const moe_offload* h) {
  return (unsigned long long)(h->e13_bytes + h->e2_bytes + sizeof(float) * (h->f13 + h->f2));
}

moe_status_t check_shared(moe_offload* h, int l0, int l1) {
  if (!h->cfg.shared_expert) return MOE_OK;
  for (int l = l0; l < l1; ++l)
    if (!h->shared_set[l]) return fail(h, MOE_ERR_INVALID, "shared expert of layer %d not set", l);
  return MOE_OK;
}

// True when this allocation is the one MOE_OFFLOAD_FAIL_ALLOC names.
bool injected_failure(moe_offload* h) { return h->alloc_seq++ == h->fail_alloc_at; }

template <typename T>
moe_status_t dev_alloc(moe_offload* h, T** p, size_t bytes) {
  if (injected_failure(h))
    return fail(h, MOE_ERR_OOM, "cudaMalloc of %zu bytes: injected failure (MOE_OFFLOAD_FAIL_ALLOC=%d)", bytes,
                h->fail_alloc_at);
  void* q = nullptr;
  cudaError_t e = cudaMalloc(&q, bytes ? bytes : 16);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaMalloc");
  h->allocations.push_back(q);
  h->dev_bytes += bytes;
  *p = static_cast<T*>(q);
  return MOE_OK;
}

// Pins and maps the host ranges (merged where they touch) unless already pinned.
moe_status_t register_host(moe_offload* h, std::vector<std::pair<uintptr_t, size_t>> ranges) {
  std::sort(ranges.begin(), ranges.end());
  std::vector<std::pair<uintptr_t, size_t>> merged;
  for (auto& r : ranges) {
    if (!merged.empty() && r.first <= merged.back().first + merged.back().second) {
      const uintptr_t end = std::max(merged.back().first + merged.back().second, r.first + r.second);
      merged.back().second = end - merged.back().first;
    } else {
      merged.push_back(r);
    }
  }
  for (auto& r : merged) {
    void* p = reinterpret_cast<void*>(r.first);
    cudaPointerAttributes at{};
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e == cudaSuccess && at.type == cudaMemoryTypeHost) continue;  // already pinned
    (void)cudaGetLastError();
    if (injected_failure(h))
      return fail(h, MOE_ERR_OOM, "cudaHostRegister of the host expert store: injected failure "
                  "(MOE_OFFLOAD_FAIL_ALLOC=%d)", h->fail_alloc_at);
    e = cudaHostRegister(p, r.second, cudaHostRegisterMapped | cudaHostRegisterPortable);
    if (e == cudaErrorHostMemoryAlreadyRegistered) {
      (void)cudaGetLastError();
      continue;
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaHostRegister of the host expert store");
    h->registered.push_back(p);
  }
  return MOE_OK;
}

moe_status_t init_tables(moe_offload* h) {
  const int E = h->cfg.num_experts, S = h->cfg.num_slots;
  for (auto& t : h->tab) {
    std::vector<int32_t> neg_s(S, -1), neg_e(E, -1);
    CK(h, cudaMemcpy(t.slot_expert, neg_s.data(), sizeof(int32_t) * S, cudaMemcpyHostToDevice));
    CK(h, cudaMemcpy(t.expert_slot, neg_e.data(), sizeof(int32_t) * E, cudaMemcpyHostToDevice));
    CK(h, cudaMemset(t.stamp, 0, sizeof(uint32_t) * S));
    CK(h, cudaMemset(t.clock, 0, sizeof(uint32_t)));
    CK(h, cudaMemset(t.miss_expert, 0, sizeof(int32_t) * E));
    CK(h, cudaMemset(t.miss_slot, 0, sizeof(int32_t) * E));
    CK(h, cudaMemset(t.counts, 0, sizeof(int32_t) * kNumCounts));
    CK(h, cudaMemset(t.stats, 0, sizeof(unsigned long long) * kNumStats));
    CK(h, cudaMemset(t.route_counts, 0, sizeof(unsigned long long) * E));
    CK(h, cudaMemset(t.pair_src, 0xff, sizeof(int32_t) * kMaxCallPairs));
  }
  std::fill(h->frozen.begin(), h->frozen.end(), 0);
  CK(h, cudaMemset(h->status, 0, sizeof(uint32_t)));
  return MOE_OK;
}

moe_status_t check_layer(moe_offload* h, int layer) {
  if (!h) return MOE_ERR_INVALID;
  if (layer < 0 || layer >= h->cfg.num_layers)
    return fail(h, MOE_ERR_INVALID, "layer %d outside [0, %d)", layer, h->cfg.num_layers);
  return MOE_OK;
}

moe_status_t set_device(moe_offload* h) {
  CK(h, cudaSetDevice(h->device));
  return MOE_OK;
}

bool capturing(cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return cs != cudaStreamCaptureStatusNone;
}

// Copy of the experts the last prefetch install put into `layer`, on the
// prefetch stream after the work enqueued so far on st (which made the install).
moe_status_t pf_fork(moe_offload* h, int layer, cudaStream_t st) {
  if (h->pf_pending[layer]) return fail(h, MOE_ERR_INVALID, "prefetch of layer %d issued twice without a join", layer);
  CK(h, cudaEventRecord(h->pf_ready[layer], st));
  CK(h, cudaStreamWaitEvent(h->pf_stream, h->pf_ready[layer], 0));
  CopyArgs a{};
  a.lw = h->lw[layer];
  a.counts = h->tab[layer].counts;
  a.count_idx = kCntPrefetch;
  a.miss_expert = h->tab[layer].pf_expert;
  a.miss_slot = h->tab[layer].pf_slot;
  a.E = h->cfg.num_experts;
  a.S = h->cfg.num_slots;
  a.u13 = (unsigned long long)h->e13_bytes / 16ull;
  a.u2 = (unsigned long long)h->e2_bytes / 16ull;
  a.f13 = h->f13;
  a.f2 = h->f2;
  a.status = h->status;
  CK(h, launch_miss_copy(a, h->pf_grid, h->pf_stream));
  CK(h, cudaEventRecord(h->pf_done[layer], h->pf_stream));
  h->pf_pending[layer] = capturing(st) ? 2 : 1;
  return MOE_OK;
}

// Work enqueued on st after this waits for the prefetch copy into `layer`.
moe_status_t pf_join(moe_offload* h, int layer, cudaStream_t st) {
  if (h->pf_pending.empty() || !h->pf_pending[layer]) return MOE_OK;
  const bool cap = capturing(st);
  if ((h->pf_pending[layer] == 2) != cap)
    return fail(h, MOE_ERR_CAPTURE, "prefetch copy of layer %d was issued %s stream capture and is joined %s it",
                layer, h->pf_pending[layer] == 2 ? "under" : "outside", cap ? "under" : "outside");
  CK(h, cudaStreamWaitEvent(st, h->pf_done[layer], 0));
  h->pf_pending[layer] = 0;
  return MOE_OK;
}

FfnArgs ffn_args(moe_offload* h, int layer, const void* x, const int32_t* slot_ids, const float* w,
                 int T, void* out) {
  FfnArgs a{};
  a.lw = h->lw[layer];
  a.x = static_cast<const uint16_t*>(x);
  a.slot_ids = slot_ids;
  a.w = w;
  a.T = T;
  a.k = h->cfg.top_k;
  a.H = h->cfg.hidden;
  a.I = h->cfg.inter;
  a.E = h->cfg.num_experts;
  a.S = h->cfg.num_slots;
  a.counts = h->tab[layer].counts;
  a.miss_expert = h->tab[layer].miss_expert;
  a.hbuf = h->hbuf;
  a.out = static_cast<uint16_t*>(out);
  a.status = h->status;
  a.copy_through = 0;
  a.miss_slot = h->tab[layer].miss_slot;
  a.pdl = 0;
  a.fmt = h->fmt;
  a.shared = h->cfg.shared_expert ? 1 : 0;
  a.pair_src = h->tab[layer].pair_src;
  a.wait_ns = h->wait_ns;
  a.stall = h->stall;
  a.tr = h->trace_on ? h->trace + (size_t)layer * kTraceFields : nullptr;
  return a;
}

moe_status_t do_route(moe_offload* h, int layer, const void* x, int T, int32_t* ids, float* w,
                      float* logits, cudaStream_t st) {
  RouteArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.wr = h->router[layer];
  a.T = T;
  a.E = h->cfg.num_experts;
  a.H = h->cfg.hidden;
  a.k = h->cfg.top_k;
  a.renorm = h->cfg.renormalize;
  a.ids = ids;
  a.w = w;
  a.logits = logits;
  a.done = h->route_done + layer;
  CK(h, launch_route(a, st));
  return MOE_OK;
}

moe_status_t do_ensure(moe_offload* h, int layer, const int32_t* ids, int T, int32_t* slot_ids,
                       cudaStream_t st) {
  EnsureArgs a{};
  a.tab = h->tab[layer];
  a.ids = ids;
  a.Tk = T * h->cfg.top_k;
  a.E = h->cfg.num_experts;
  a.S = h->cfg.num_slots;
  a.slot_ids = slot_ids;
  a.status = h->status;
  a.expert_bytes = slot_bytes(h);
  CK(h, launch_slot_ensure(a, st));
  return MOE_OK;
}

// Counters for the early down of a decode step (launches under programmatic
// dependent launch only; otherwise the down launch starts after gate/up completes).
uint32_t* early_down_sync(const moe_offload* h, int pdl) {
  return (h->early_down && pdl) ? h->ffn_sync : nullptr;
}

// Decode step of one layer in three launches: route + top-k + slot ensure, then
// the grouped FFN whose gate/up launch also fills the slots this call installed
// (copy-through), then down projection + combine. No host synchronisation.
moe_status_t do_decode_head(moe_offload* h, int layer, const void* x, int T, cudaStream_t st, bool pdl = true) {
  RouteEnsureArgs a{};
  a.r.x = static_cast<const uint16_t*>(x);
  a.r.wr = h->router[layer];
  a.r.T = T;
  a.r.E = h->cfg.num_experts;
  a.r.H = h->cfg.hidden;
  a.r.k = h->cfg.top_k;
  a.r.renorm = h->cfg.renormalize;
  a.r.ids = h->ids_buf;
  a.r.w = h->w_buf;
  a.r.logits = h->logits;
  a.r.done = h->route_done + layer;
  a.tab = h->tab[layer];
  a.S = h->cfg.num_slots;
  a.slot_ids = h->slot_buf;
  a.status = h->status;
  a.expert_bytes = slot_bytes(h);
  a.pdl = (pdl && h->pdl) ? 1 : 0;
  a.tr = h->trace_on ? h->trace + (size_t)layer * kTraceFields : nullptr;
  const bool pf = h->cfg.prefetch_n > 0 && layer + 1 < h->cfg.num_layers;
  if (pf) {
    // a copy into the next layer still in flight must finish before its slots change hands
    moe_status_t js = pf_join(h, layer + 1, st);
    if (js != MOE_OK) return js;
    a.wr_next = h->router[layer + 1];
    a.tab_next = h->tab[layer + 1];
    a.pf_n = h->cfg.prefetch_n;
    a.pf_bytes = slot_bytes(h);
    a.pred_logits = h->pred_logits;
    a.pred_ids = h->pred_ids;
    a.pred_w = h->pred_w;
    a.pred_done = h->pred_done;
  }
  CK(h, launch_route_ensure(a, st));
  if (h->audit_each) {  // the layer's table, and the next layer's after a prefetch install
    CK(h, launch_audit(h->tab[layer], h->cfg.num_experts, h->cfg.num_slots, h->status, h->ffn_sync, st));
    if (pf)
      CK(h, launch_audit(h->tab[layer + 1], h->cfg.num_experts, h->cfg.num_slots, h->status, h->ffn_sync, st));
  }
  return MOE_OK;
}

// Whether the decode step of `layer` prefetches into the next layer.
bool lookahead_on(const moe_offload* h, int layer) {
  return h->cfg.prefetch_n > 0 && layer + 1 < h->cfg.num_layers;
}

// Launches of this library per decode layer (head, gate/up, down, audits).
int launches_per_layer(const moe_offload* h, int layer) {
  return 3 + (h->audit_each ? 1 + (lookahead_on(h, layer) ? 1 : 0) : 0);
}

moe_status_t do_decode_ffn(moe_offload* h, int layer, const void* x, int T, void* out, cudaStream_t st,
                           cudaEvent_t after_gate_up = nullptr) {
  moe_status_t js = pf_join(h, layer, st);
  if (js != MOE_OK) return js;
  FfnArgs a = ffn_args(h, layer, x, h->slot_buf, h->w_buf, T, out);
  a.copy_through = 1;
  a.pdl = h->pdl;
  a.sync = early_down_sync(h, a.pdl);
  CK(h, launch_grouped_ffn_phase(a, 0, st));
  // The next layer's prefetch copy starts once this layer's own copies (done by
  // the gate/up launch) are through, so it uses the host link while down +
  // combine and the next head run instead of competing with demand copies.
  if (lookahead_on(h, layer) && (js = pf_fork(h, layer + 1, st)) != MOE_OK) return js;
  if (after_gate_up) CK(h, cudaEventRecord(after_gate_up, st));
  CK(h, launch_grouped_ffn_phase(a, 1, st));
  return MOE_OK;
}

// Profile: adds the elapsed times of every pending record to the per-layer sums
// (waits for their last events) and returns the events to the pool.
moe_status_t profile_fold(moe_offload* h) {
  moe_status_t st = MOE_OK;
  for (auto& r : h->prof_pending) {
    float ms[3] = {0.0f, 0.0f, 0.0f};
    cudaError_t e = cudaEventSynchronize(r.ev[3]);
    for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaEventElapsedTime(&ms[i], r.ev[i], r.ev[i + 1]);
    if (e != cudaSuccess) {  // a record whose launches failed: report it, clear the runtime's error
      (void)cudaGetLastError();
      st = cuda_fail(h, e, "profile events");
    } else {
      auto& acc = h->prof_sum[r.layer];
      acc[0] += 1.0;
      for (int i = 0; i < 3; ++i) acc[i + 1] += ms[i];
    }
    for (cudaEvent_t ev : r.ev) h->prof_pool.push_back(ev);
  }
  h->prof_pending.clear();
  return st;
}

moe_status_t profile_event(moe_offload* h, cudaEvent_t* ev) {
  if (!h->prof_pool.empty()) {
    *ev = h->prof_pool.back();
    h->prof_pool.pop_back();
    return MOE_OK;
  }
  CK(h, cudaEventCreate(ev));
  return MOE_OK;
}

// One profiled decode step of a layer: the three launches with events between them.
moe_status_t profiled_decode(moe_offload* h, int layer, const void* x, int T, void* out, cudaStream_t s) {
  constexpr size_t kMaxPending = 1 << 16;
  moe_status_t st;
  if (h->prof_pending.size() >= kMaxPending && (st = profile_fold(h)) != MOE_OK) return st;
  moe_offload::ProfileRec r{layer, {}};
  for (auto& ev : r.ev)
    if ((st = profile_event(h, &ev)) != MOE_OK) return st;
  h->prof_pending.push_back(r);  // recorded or not, its events go back to the pool at the next fold
  CK(h, cudaEventRecord(r.ev[0], s));
  if ((st = do_decode_head(h, layer, x, T, s)) != MOE_OK) return st;
  CK(h, cudaEventRecord(r.ev[1], s));
  if ((st = do_decode_ffn(h, layer, x, T, out, s, r.ev[2])) != MOE_OK) return st;
  CK(h, cudaEventRecord(r.ev[3], s));
  return MOE_OK;
}

moe_status_t do_copy(moe_offload* h, int layer, cudaStream_t st) {
  CopyArgs a{};
  a.lw = h->lw[layer];
  a.counts = h->tab[layer].counts;
  a.miss_expert = h->tab[layer].miss_expert;
  a.miss_slot = h->tab[layer].miss_slot;
  a.E = h->cfg.num_experts;
  a.S = h->cfg.num_slots;
  a.u13 = (unsigned long long)h->e13_bytes / 16ull;
  a.u2 = (unsigned long long)h->e2_bytes / 16ull;
  a.f13 = h->f13;
  a.f2 = h->f2;
  a.status = h->status;
  a.count_idx = kCntInstall;
  CK(h, launch_miss_copy(a, h->copy_grid, st));
  return MOE_OK;
}

}  // namespace

void moe::set_handleless_error(const char* msg) { g_create_error = msg; }

extern "C" {

int moe_offload_slots_for_fraction(double fraction, int num_experts, int top_k) {
  if (!(fraction > 0.0 && fraction <= 1.0) || num_experts < 1 || top_k < 1) return -1;
  const int s = (int)std::floor(fraction * (double)num_experts + 1e-9);
  return std::max(top_k, s);
}

int moe_offload_slots_auto(size_t free_bytes, size_t reserve_bytes, int num_layers, int num_experts, int top_k,
                           size_t expert_bytes) {
  if (num_layers < 1 || num_experts < 1 || top_k < 1 || top_k > num_experts || expert_bytes == 0) return -1;
  if (free_bytes <= reserve_bytes) return -1;
  const unsigned long long per_slot = (unsigned long long)num_layers * expert_bytes;
  const unsigned long long s = (unsigned long long)(free_bytes - reserve_bytes) / per_slot;
  if (s < (unsigned long long)top_k) return -1;
  return s > (unsigned long long)num_experts ? num_experts : (int)s;
}

moe_status_t moe_offload_create(const moe_offload_config_t* cfg, int device, void* const* host_w13,
                                void* const* host_w2, const float* const* host_scales13,
                                const float* const* host_scales2, const void* const* dev_router,
                                moe_offload_t* out) {
  if (!out) return fail(nullptr, MOE_ERR_INVALID, "out is NULL");
  *out = nullptr;
  if (!cfg || !host_w13 || !host_w2 || !dev_router)
    return fail(nullptr, MOE_ERR_INVALID, "NULL config or weight table");
  const moe_offload_config_t c = *cfg;
  if (c.num_layers < 1 || c.num_experts < 1 || c.num_experts > 1024 || c.top_k < 1 || c.top_k > 16 ||
      c.top_k > c.num_experts || c.hidden < 256 || c.hidden % 256 != 0 || c.hidden > 8192 ||
      c.inter < 64 || c.inter % 64 != 0 ||
      (c.num_slots != 0 && (c.num_slots < c.top_k || c.num_slots > c.num_experts)) ||
      c.max_tokens_graph < 1 || c.max_tokens_graph > 64 || c.max_tokens_graph * c.top_k > 1024)
    return fail(nullptr, MOE_ERR_INVALID,
                "invalid configuration (L=%d E=%d k=%d H=%d I=%d S=%d Tmax=%d)", c.num_layers,
                c.num_experts, c.top_k, c.hidden, c.inter, c.num_slots, c.max_tokens_graph);
  if (c.dtype != MOE_DTYPE_BF16 && c.dtype != MOE_DTYPE_FP8_E4M3_B128)
    return fail(nullptr, MOE_ERR_INVALID, "unsupported dtype %d", c.dtype);
  const bool fp8 = c.dtype == MOE_DTYPE_FP8_E4M3_B128;
  if (c.shared_expert != 0 && c.shared_expert != 1)
    return fail(nullptr, MOE_ERR_INVALID, "shared_expert must be 0 or 1");
  const int s_bound = c.num_slots ? c.num_slots : c.num_experts;  // auto: checked again once S is known
  if (c.prefetch_n < 0 || c.prefetch_n > s_bound)
    return fail(nullptr, MOE_ERR_INVALID, "prefetch_n=%d outside [0, num_slots=%d]", c.prefetch_n, s_bound);
  if (c.max_tokens_graph * (c.top_k + c.shared_expert) > 1024)
    return fail(nullptr, MOE_ERR_INVALID, "max_tokens_graph * (top_k + shared_expert) above 1024");
  if (fp8) {
    if (c.hidden % 128 != 0 || c.inter % 128 != 0)
      return fail(nullptr, MOE_ERR_INVALID, "FP8 block scales need hidden and inter multiples of 128");
    if (!host_scales13 || !host_scales2)
      return fail(nullptr, MOE_ERR_INVALID, "FP8 experts need both scale tables");
  } else if (host_scales13 || host_scales2) {
    return fail(nullptr, MOE_ERR_INVALID, "scale tables are only for block-scaled formats");
  }
  for (int l = 0; l < c.num_layers; ++l) {
    if (!host_w13[l] || !host_w2[l] || !dev_router[l])
      return fail(nullptr, MOE_ERR_INVALID, "NULL weight pointer at layer %d", l);
    if (!aligned16(host_w13[l]) || !aligned16(host_w2[l]) || !aligned16(dev_router[l]))
      return fail(nullptr, MOE_ERR_INVALID, "weight pointer of layer %d not 16-byte aligned", l);
    if (fp8 && (!host_scales13[l] || !host_scales2[l] || !aligned4(host_scales13[l]) || !aligned4(host_scales2[l])))
      return fail(nullptr, MOE_ERR_INVALID, "NULL or unaligned scale table at layer %d", l);
  }

  moe_offload* h = new (std::nothrow) moe_offload();
  if (!h) return fail(nullptr, MOE_ERR_OOM, "out of host memory");
  h->cfg = c;
  h->device = device;
  const int L = c.num_layers, E = c.num_experts, H = c.hidden, I = c.inter;
  const int Tmax = c.max_tokens_graph, k = c.top_k;
  h->w13_elems = (size_t)2 * I * H;
  h->w2_elems = (size_t)H * I;
  h->fmt = fp8 ? 1 : 0;
  h->e13_bytes = h->w13_elems * (fp8 ? 1 : 2);
  h->e2_bytes = h->w2_elems * (fp8 ? 1 : 2);
  h->f13 = fp8 ? (size_t)(2 * I / 128) * (H / 128) : 0;
  h->f2 = fp8 ? (size_t)(H / 128) * (I / 128) : 0;
  h->shared_set.assign(L, 0);
  h->frozen.assign(L, 0);
  auto bail = [&](moe_status_t st) {
    g_create_error = h->err;
    moe_offload_destroy(h);
    return st;
  };
  moe_status_t st = set_device(h);
  if (st != MOE_OK) return bail(st);
  cudaDeviceProp prop{};
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) {
    cuda_fail(h, cudaGetLastError(), "cudaGetDeviceProperties");
    return bail(MOE_ERR_CUDA);
  }
  h->sm_count = prop.multiProcessorCount;
  h->copy_grid = 2 * h->sm_count;
  if (const char* v = getenv("MOE_OFFLOAD_PDL")) h->pdl = atoi(v) != 0;
  if (const char* v = getenv("MOE_OFFLOAD_AUDIT")) h->audit_each = atoi(v) != 0;
  if (const char* v = getenv("MOE_OFFLOAD_EARLY_DOWN")) h->early_down = atoi(v) != 0;
  if (const char* v = getenv("MOE_OFFLOAD_PROFILE")) h->profile = atoi(v) != 0;
  h->prof_sum.assign(c.num_layers, std::array<double, 4>{0.0, 0.0, 0.0, 0.0});
  if (const char* v = getenv("MOE_OFFLOAD_FAIL_ALLOC")) h->fail_alloc_at = atoi(v);
  {
    cudaError_t e = route_init_attributes();
    if (e == cudaSuccess) e = prefill_init_attributes();
    if (e == cudaSuccess) e = ffn_init_attributes();
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "kernel attributes"));
  }

  // Host expert store: pin and map (never copied).
  std::vector<std::pair<uintptr_t, size_t>> ranges;
  for (int l = 0; l < L; ++l) {
    ranges.push_back({reinterpret_cast<uintptr_t>(host_w13[l]), (size_t)E * h->e13_bytes});
    ranges.push_back({reinterpret_cast<uintptr_t>(host_w2[l]), (size_t)E * h->e2_bytes});
    if (fp8) {
      ranges.push_back({reinterpret_cast<uintptr_t>(host_scales13[l]), (size_t)E * h->f13 * sizeof(float)});
      ranges.push_back({reinterpret_cast<uintptr_t>(host_scales2[l]), (size_t)E * h->f2 * sizeof(float)});
    }
  }
  st = register_host(h, ranges);
  if (st != MOE_OK) return bail(st);

  h->lw.resize(L);
  h->tab.resize(L);
  h->router.resize(L);
  for (int l = 0; l < L; ++l) {
    void* d13 = nullptr;
    void* d2 = nullptr;
    cudaError_t e = cudaHostGetDevicePointer(&d13, host_w13[l], 0);
    if (e == cudaSuccess) e = cudaHostGetDevicePointer(&d2, host_w2[l], 0);
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "cudaHostGetDevicePointer"));
    h->lw[l].host_w13 = static_cast<const uint8_t*>(d13);
    h->lw[l].host_w2 = static_cast<const uint8_t*>(d2);
    if (fp8) {
      void* q13 = nullptr;
      void* q2 = nullptr;
      e = cudaHostGetDevicePointer(&q13, const_cast<float*>(host_scales13[l]), 0);
      if (e == cudaSuccess) e = cudaHostGetDevicePointer(&q2, const_cast<float*>(host_scales2[l]), 0);
      if (e != cudaSuccess) return bail(cuda_fail(h, e, "cudaHostGetDevicePointer (scales)"));
      h->lw[l].host_s13 = static_cast<const float*>(q13);
      h->lw[l].host_s2 = static_cast<const float*>(q2);
    }
    h->router[l] = static_cast<const uint16_t*>(dev_router[l]);
  }

  // Decode scratch.
  const size_t tk = (size_t)Tmax * k;
  if ((st = dev_alloc(h, &h->ids_buf, sizeof(int32_t) * tk)) != MOE_OK ||
      (st = dev_alloc(h, &h->w_buf, sizeof(float) * tk)) != MOE_OK ||
      (st = dev_alloc(h, &h->slot_buf, sizeof(int32_t) * tk)) != MOE_OK ||
      (st = dev_alloc(h, &h->logits, sizeof(float) * (size_t)Tmax * E)) != MOE_OK ||
      (st = dev_alloc(h, &h->hbuf, sizeof(float) * (tk + (size_t)Tmax * c.shared_expert) * I)) != MOE_OK ||
      (st = dev_alloc(h, &h->route_done, sizeof(unsigned) * L)) != MOE_OK ||
      (st = dev_alloc(h, &h->status, sizeof(uint32_t))) != MOE_OK ||
      (st = dev_alloc(h, &h->ffn_sync, sizeof(uint32_t) * kFfnSyncWords)) != MOE_OK)
    return bail(st);
  {
    cudaError_t e = cudaMemset(h->route_done, 0, sizeof(unsigned) * L);
    if (e == cudaSuccess) e = cudaMemset(h->ffn_sync, 0, sizeof(uint32_t) * kFfnSyncWords);
    if (e == cudaSuccess) e = cudaMemset(h->ids_buf, 0, sizeof(int32_t) * tk);
    if (e == cudaSuccess) e = cudaMemset(h->w_buf, 0, sizeof(float) * tk);
    if (e == cudaSuccess) e = cudaMemset(h->slot_buf, 0, sizeof(int32_t) * tk);
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "cudaMemset"));
  }
  h->pf_pending.assign(L, 0);
  if (c.prefetch_n > 0) {
    if ((st = dev_alloc(h, &h->pred_logits, sizeof(float) * (size_t)Tmax * E)) != MOE_OK ||
        (st = dev_alloc(h, &h->pred_ids, sizeof(int32_t) * tk)) != MOE_OK ||
        (st = dev_alloc(h, &h->pred_w, sizeof(float) * tk)) != MOE_OK ||
        (st = dev_alloc(h, &h->pred_done, sizeof(unsigned))) != MOE_OK)
      return bail(st);
    cudaError_t e = cudaMemset(h->pred_done, 0, sizeof(unsigned));
    int lo = 0, hi = 0;
    if (e == cudaSuccess) e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&h->pf_stream, cudaStreamNonBlocking, hi);
    h->pf_ready.assign(L, nullptr);
    h->pf_done.assign(L, nullptr);
    for (int l = 0; l < L && e == cudaSuccess; ++l) {
      e = cudaEventCreateWithFlags(&h->pf_ready[l], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->pf_done[l], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "prefetch stream and events"));
  }
  {
    cudaError_t e = prefill_create(&h->prefill, E, c.shared_expert, H, I, h->w13_elems, h->w2_elems, &h->dev_bytes);
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "prefill buffers"));
  }

  // `auto` slot count: every other allocation is made; the layers' slots grow
  // evenly into what is free, less the reserve ("MoE expert offload" page,
  // Options table: auto sizing after loading, XINFER_MOE_OFFLOAD_RESERVE_GB).
  if (c.num_slots == 0) {
    size_t free_b = 0, total_b = 0;
    cudaError_t e = cudaMemGetInfo(&free_b, &total_b);
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "cudaMemGetInfo"));
    const size_t reserve = c.auto_reserve_bytes ? (size_t)c.auto_reserve_bytes : kAutoReserveBytes;
    const int s_auto = moe_offload_slots_auto(free_b, reserve, L, E, k, (size_t)slot_bytes(h));
    h->auto_free = free_b;
    if (s_auto < 0)
      return bail(fail(h, MOE_ERR_OOM, "auto slots: %zu free bytes less a %zu-byte reserve hold fewer than "
                       "top_k=%d slots per layer of %llu bytes x %d layers", free_b, reserve, k,
                       slot_bytes(h), L));
    if (c.prefetch_n > s_auto)
      return bail(fail(h, MOE_ERR_INVALID, "prefetch_n=%d above the %d auto slots", c.prefetch_n, s_auto));
    h->cfg.num_slots = s_auto;
  }
  const int S = h->cfg.num_slots;

  // Slot tensors.
  for (int l = 0; l < L; ++l) {
    if ((st = dev_alloc(h, &h->lw[l].slot_w13, (size_t)S * h->e13_bytes)) != MOE_OK) return bail(st);
    if ((st = dev_alloc(h, &h->lw[l].slot_w2, (size_t)S * h->e2_bytes)) != MOE_OK) return bail(st);
    if (fp8) {
      if ((st = dev_alloc(h, &h->lw[l].slot_s13, sizeof(float) * S * h->f13)) != MOE_OK) return bail(st);
      if ((st = dev_alloc(h, &h->lw[l].slot_s2, sizeof(float) * S * h->f2)) != MOE_OK) return bail(st);
    }
  }

  // Slot tables: one block, a 256-byte-aligned record per layer.
  auto up = [](size_t b) { return (b + 255) & ~(size_t)255; };
  const size_t rec = up(sizeof(int32_t) * S) + up(sizeof(int32_t) * E) + up(sizeof(uint32_t) * S) +
                     up(sizeof(uint32_t)) + up(sizeof(int32_t) * E) * 5 + up(sizeof(int32_t) * kNumCounts) +
                     up(sizeof(unsigned long long) * kNumStats) + up(sizeof(unsigned long long) * E) +
                     up(sizeof(int32_t) * kMaxCallPairs);
  char* block = nullptr;
  if ((st = dev_alloc(h, &block, rec * L)) != MOE_OK) return bail(st);
  for (int l = 0; l < L; ++l) {
    char* p = block + rec * l;
    LayerTables& t = h->tab[l];
    t.slot_expert = reinterpret_cast<int32_t*>(p); p += up(sizeof(int32_t) * S);
    t.expert_slot = reinterpret_cast<int32_t*>(p); p += up(sizeof(int32_t) * E);
    t.stamp = reinterpret_cast<uint32_t*>(p); p += up(sizeof(uint32_t) * S);
    t.clock = reinterpret_cast<uint32_t*>(p); p += up(sizeof(uint32_t));
    t.miss_expert = reinterpret_cast<int32_t*>(p); p += up(sizeof(int32_t) * E);
    t.miss_slot = reinterpret_cast<int32_t*>(p); p += up(sizeof(int32_t) * E);
    t.counts = reinterpret_cast<int32_t*>(p); p += up(sizeof(int32_t) * kNumCounts);
    t.pf_expert = reinterpret_cast<int32_t*>(p); p += up(sizeof(int32_t) * E);
    t.pf_slot = reinterpret_cast<int32_t*>(p); p += up(sizeof(int32_t) * E);
    t.pf_cand = reinterpret_cast<int32_t*>(p); p += up(sizeof(int32_t) * E);
    t.route_counts = reinterpret_cast<unsigned long long*>(p); p += up(sizeof(unsigned long long) * E);
    t.pair_src = reinterpret_cast<int32_t*>(p); p += up(sizeof(int32_t) * kMaxCallPairs);
    t.stats = reinterpret_cast<unsigned long long*>(p);
  }
  if ((st = init_tables(h)) != MOE_OK) return bail(st);
  // First GPU read of the host store: on GB300 the first pass of GPU reads over
  // host pages the CPU had just written ran well below the link rate (a
  // 256-token decode pass at 189 tok/s where later passes ran at 262), so the
  // store is read once here, at load time, rather than inside the first decode
  // steps. About 0.3 s per 54 GiB.
  {
    unsigned* sink = nullptr;
    if ((st = dev_alloc(h, &sink, sizeof(unsigned))) != MOE_OK) return bail(st);
    cudaError_t e = cudaSuccess;
    for (int l = 0; l < L && e == cudaSuccess; ++l) {
      const LayerWeights& w = h->lw[l];
      e = launch_host_touch(w.host_w13, (unsigned long long)E * h->e13_bytes, sink, h->copy_grid, 0);
      if (e == cudaSuccess) e = launch_host_touch(w.host_w2, (unsigned long long)E * h->e2_bytes, sink, h->copy_grid, 0);
      if (e == cudaSuccess && fp8)
        e = launch_host_touch(w.host_s13, (unsigned long long)E * h->f13 * sizeof(float), sink, h->copy_grid, 0);
      if (e == cudaSuccess && fp8)
        e = launch_host_touch(w.host_s2, (unsigned long long)E * h->f2 * sizeof(float), sink, h->copy_grid, 0);
    }
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "first read of the host store"));
  }
  {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return bail(cuda_fail(h, e, "cudaDeviceSynchronize"));
  }
  *out = h;
  g_create_error.clear();
  return MOE_OK;
}

moe_status_t moe_offload_route_topk(moe_offload_t h, int layer, const void* x, int T, int32_t* ids,
                                    float* w, moe_stream_t stream) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  if (T < 0) return fail(h, MOE_ERR_INVALID, "T < 0");
  if (T == 0) return MOE_OK;
  if (!x || !ids || !w || !aligned16(x)) return fail(h, MOE_ERR_INVALID, "NULL or unaligned pointer");
  if ((st = set_device(h)) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* logits = h->logits;
  if (T > h->cfg.max_tokens_graph) {
    if (capturing(s)) return fail(h, MOE_ERR_CAPTURE, "T above max_tokens_graph under capture");
    cudaError_t e = prefill_reserve(&h->prefill, T, h->cfg.top_k, h->cfg.num_experts, &h->dev_bytes);
    if (e != cudaSuccess) return cuda_fail(h, e, "prefill scratch");
    logits = h->prefill.logits;
  }
  return do_route(h, layer, x, T, ids, w, logits, s);
}

moe_status_t moe_offload_slot_ensure(moe_offload_t h, int layer, const int32_t* ids, int T,
                                     int32_t* slot_ids, moe_stream_t stream) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  if (T < 0 || T > h->cfg.max_tokens_graph)
    return fail(h, MOE_ERR_INVALID, "T=%d outside [0, max_tokens_graph=%d]", T, h->cfg.max_tokens_graph);
  if (T == 0) return MOE_OK;
  if (!ids || !slot_ids) return fail(h, MOE_ERR_INVALID, "NULL pointer");
  if ((st = set_device(h)) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = do_ensure(h, layer, ids, T, slot_ids, s)) != MOE_OK) return st;
  if (h->audit_each)
    CK(h, launch_audit(h->tab[layer], h->cfg.num_experts, h->cfg.num_slots, h->status, h->ffn_sync, s));
  return MOE_OK;
}

moe_status_t moe_offload_miss_copy(moe_offload_t h, int layer, moe_stream_t stream) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  if ((st = set_device(h)) != MOE_OK) return st;
  if ((st = pf_join(h, layer, reinterpret_cast<cudaStream_t>(stream))) != MOE_OK) return st;
  return do_copy(h, layer, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_offload_grouped_ffn(moe_offload_t h, int layer, const void* x, const int32_t* slot_ids,
                                     const float* w, int T, void* out, moe_stream_t stream) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  if (T < 0 || T > h->cfg.max_tokens_graph)
    return fail(h, MOE_ERR_INVALID, "T=%d outside [0, max_tokens_graph=%d]", T, h->cfg.max_tokens_graph);
  if (T == 0) return MOE_OK;
  if (!x || !slot_ids || !w || !out || !aligned16(x) || !aligned16(out))
    return fail(h, MOE_ERR_INVALID, "NULL or unaligned pointer");
  if ((st = check_shared(h, layer, layer + 1)) != MOE_OK) return st;
  if ((st = set_device(h)) != MOE_OK) return st;
  if ((st = pf_join(h, layer, reinterpret_cast<cudaStream_t>(stream))) != MOE_OK) return st;
  FfnArgs a = ffn_args(h, layer, x, slot_ids, w, T, out);
  CK(h, launch_grouped_ffn(a, reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status_t moe_offload_decode_layer(moe_offload_t h, int layer, const void* x, int T, void* out,
                                      moe_stream_t stream) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  if (T < 0) return fail(h, MOE_ERR_INVALID, "T < 0");
  if (T == 0) return MOE_OK;
  if (!x || !out || !aligned16(x) || !aligned16(out))
    return fail(h, MOE_ERR_INVALID, "NULL or unaligned pointer");
  if ((st = check_shared(h, layer, layer + 1)) != MOE_OK) return st;
  if ((st = set_device(h)) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T <= h->cfg.max_tokens_graph) {
    h->last_tk = T * h->cfg.top_k;
    if (h->profile && !capturing(s)) return profiled_decode(h, layer, x, T, out, s);
    if ((st = do_decode_head(h, layer, x, T, s)) != MOE_OK) return st;
    return do_decode_ffn(h, layer, x, T, out, s);
  }
  if (h->cfg.shared_expert && h->cfg.num_experts >= 1024)
    return fail(h, MOE_ERR_INVALID, "prefill with a shared expert takes at most 1023 routed experts");
  if (capturing(s)) return fail(h, MOE_ERR_CAPTURE, "prefill path (T=%d) under stream capture", T);
  if ((st = pf_join(h, layer, s)) != MOE_OK) return st;
  PrefillLayer pl{};
  pl.lw = h->lw[layer];
  pl.tab = h->tab[layer];
  pl.router = h->router[layer];
  pl.E = h->cfg.num_experts;
  pl.S = h->cfg.num_slots;
  pl.k = h->cfg.top_k;
  pl.H = h->cfg.hidden;
  pl.I = h->cfg.inter;
  pl.renorm = h->cfg.renormalize;
  pl.w13_elems = h->w13_elems;
  pl.w2_elems = h->w2_elems;
  pl.host_w13_ptr = reinterpret_cast<const uint16_t*>(h->lw[layer].host_w13);
  pl.host_w2_ptr = reinterpret_cast<const uint16_t*>(h->lw[layer].host_w2);
  pl.route_done = h->route_done + layer;
  pl.status = h->status;
  pl.frozen = h->frozen[layer];
  pl.early_down = h->early_down;
  pl.wait_ns = h->wait_ns;
  pl.stall = h->stall;
  pl.layer = layer;
  pl.next_host_w13 = nullptr;
  pl.next_host_w2 = nullptr;
  if (layer + 1 < h->cfg.num_layers) {
    pl.next_host_w13 = reinterpret_cast<const uint16_t*>(h->lw[layer + 1].host_w13);
    pl.next_host_w2 = reinterpret_cast<const uint16_t*>(h->lw[layer + 1].host_w2);
  }
  pl.fmt = h->fmt;
  pl.host_s13 = h->lw[layer].host_s13;
  pl.host_s2 = h->lw[layer].host_s2;
  pl.next_host_s13 = layer + 1 < h->cfg.num_layers ? h->lw[layer + 1].host_s13 : nullptr;
  pl.next_host_s2 = layer + 1 < h->cfg.num_layers ? h->lw[layer + 1].host_s2 : nullptr;
  pl.shared = h->cfg.shared_expert ? 1 : 0;
  pl.sh_w13 = h->lw[layer].sh_w13;
  pl.sh_w2 = h->lw[layer].sh_w2;
  pl.sh_s13 = h->lw[layer].sh_s13;
  pl.sh_s2 = h->lw[layer].sh_s2;
  pl.stage_bytes = (unsigned long long)h->cfg.num_experts * slot_bytes(h);
  std::string why;
  cudaError_t e = prefill_layer(&h->prefill, pl, static_cast<const uint16_t*>(x), T,
                                static_cast<uint16_t*>(out), s, &h->dev_bytes, &why);
  if (e != cudaSuccess) return cuda_fail(h, e, why.empty() ? "prefill" : why.c_str());
  if (h->audit_each)
    CK(h, launch_audit(h->tab[layer], h->cfg.num_experts, h->cfg.num_slots, h->status, h->ffn_sync, s));
  return MOE_OK;
}

moe_status_t moe_offload_audit(moe_offload_t h, int layer, moe_stream_t stream) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  if ((st = set_device(h)) != MOE_OK) return st;
  CK(h, launch_audit(h->tab[layer], h->cfg.num_experts, h->cfg.num_slots, h->status, h->ffn_sync,
                     reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status_t moe_offload_get_stats(moe_offload_t h, int layer, moe_offload_stats_t* stats) {
  if (!h || !stats) return MOE_ERR_INVALID;
  if (layer >= h->cfg.num_layers) return fail(h, MOE_ERR_INVALID, "layer %d out of range", layer);
  moe_status_t st = set_device(h);
  if (st != MOE_OK) return st;
  CK(h, cudaDeviceSynchronize());
  memset(stats, 0, sizeof(*stats));
  const int l0 = layer < 0 ? 0 : layer, l1 = layer < 0 ? h->cfg.num_layers : layer + 1;
  for (int l = l0; l < l1; ++l) {
    unsigned long long v[kNumStats];
    CK(h, cudaMemcpy(v, h->tab[l].stats, sizeof(v), cudaMemcpyDeviceToHost));
    stats->calls += v[kStatCalls];
    stats->hits += v[kStatHits];
    stats->misses += v[kStatMisses];
    stats->spills += v[kStatSpills];
    stats->bytes_copied += v[kStatBytesCopied];
    stats->staged_calls += v[kStatStagedCalls];
    stats->staged_bytes += v[kStatStagedBytes];
    stats->prefetch_installs += v[kStatPrefetchInstalls];
    stats->prefetch_hits += v[kStatPrefetchHits];
    stats->prefetch_bytes += v[kStatPrefetchBytes];
  }
  uint32_t s = 0;
  CK(h, cudaMemcpy(&s, h->status, sizeof(s), cudaMemcpyDeviceToHost));
  stats->device_status = s;
  if (s != 0) return fail(h, MOE_ERR_DEVICE_STATUS, "device status 0x%x", s);
  return MOE_OK;
}

moe_status_t moe_offload_read_table(moe_offload_t h, int layer, int32_t* slot_expert,
                                    int32_t* expert_slot, uint32_t* stamp, uint32_t* clock) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  if ((st = set_device(h)) != MOE_OK) return st;
  CK(h, cudaDeviceSynchronize());
  const LayerTables& t = h->tab[layer];
  const int E = h->cfg.num_experts, S = h->cfg.num_slots;
  if (slot_expert) CK(h, cudaMemcpy(slot_expert, t.slot_expert, sizeof(int32_t) * S, cudaMemcpyDeviceToHost));
  if (expert_slot) CK(h, cudaMemcpy(expert_slot, t.expert_slot, sizeof(int32_t) * E, cudaMemcpyDeviceToHost));
  if (stamp) CK(h, cudaMemcpy(stamp, t.stamp, sizeof(uint32_t) * S, cudaMemcpyDeviceToHost));
  if (clock) CK(h, cudaMemcpy(clock, t.clock, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status_t moe_offload_debug_write_table(moe_offload_t h, int layer, int table, int index, int64_t value) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  const int E = h->cfg.num_experts, S = h->cfg.num_slots;
  const LayerTables& t = h->tab[layer];
  void* dst = nullptr;
  switch (table) {
    case MOE_TABLE_SLOT_EXPERT:
      if (index < 0 || index >= S || value < -1 || value >= E)
        return fail(h, MOE_ERR_INVALID, "slot_expert[%d] = %lld out of range", index, (long long)value);
      dst = t.slot_expert + index;
      break;
    case MOE_TABLE_EXPERT_SLOT:
      if (index < 0 || index >= E || value < -1 || value >= S)
        return fail(h, MOE_ERR_INVALID, "expert_slot[%d] = %lld out of range", index, (long long)value);
      dst = t.expert_slot + index;
      break;
    case MOE_TABLE_STAMP:
      if (index < 0 || index >= S || value < 0 || value > 0xffffffffll)
        return fail(h, MOE_ERR_INVALID, "stamp[%d] = %lld out of range", index, (long long)value);
      dst = t.stamp + index;
      break;
    case MOE_TABLE_CLOCK:
      if (index != 0 || value < 0 || value > 0xffffffffll)
        return fail(h, MOE_ERR_INVALID, "clock = %lld out of range", (long long)value);
      dst = t.clock;
      break;
    default:
      return fail(h, MOE_ERR_INVALID, "unknown table %d", table);
  }
  if ((st = set_device(h)) != MOE_OK) return st;
  CK(h, cudaDeviceSynchronize());
  const uint32_t word = static_cast<uint32_t>(static_cast<int32_t>(value));
  CK(h, cudaMemcpy(dst, &word, sizeof(word), cudaMemcpyHostToDevice));
  return MOE_OK;
}

moe_status_t moe_offload_read_misses(moe_offload_t h, int layer, int32_t* miss_expert, int32_t* miss_slot,
                                     int cap, int* miss_count, int* spill_count) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  if (cap < 0) return fail(h, MOE_ERR_INVALID, "cap < 0");
  if ((st = set_device(h)) != MOE_OK) return st;
  CK(h, cudaDeviceSynchronize());
  const LayerTables& t = h->tab[layer];
  int32_t c[kNumCounts];
  CK(h, cudaMemcpy(c, t.counts, sizeof(c), cudaMemcpyDeviceToHost));
  if (miss_count) *miss_count = c[kCntMiss];
  if (spill_count) *spill_count = c[kCntSpill];
  const int n = std::min(std::max(c[kCntMiss], 0), std::min(cap, h->cfg.num_experts));
  if (n > 0 && miss_expert) CK(h, cudaMemcpy(miss_expert, t.miss_expert, sizeof(int32_t) * n, cudaMemcpyDeviceToHost));
  if (n > 0 && miss_slot) CK(h, cudaMemcpy(miss_slot, t.miss_slot, sizeof(int32_t) * n, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status_t moe_offload_prefetch(moe_offload_t h, int layer, const void* x, int T, moe_stream_t stream) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  if (h->cfg.prefetch_n <= 0) return fail(h, MOE_ERR_INVALID, "handle was created with prefetch_n = 0");
  if (layer < 1) return fail(h, MOE_ERR_INVALID, "layer 0 has no previous layer to predict it from");
  if (T < 0 || T > h->cfg.max_tokens_graph)
    return fail(h, MOE_ERR_INVALID, "T=%d outside [0, max_tokens_graph=%d]", T, h->cfg.max_tokens_graph);
  if (T == 0) return MOE_OK;
  if (!x || !aligned16(x)) return fail(h, MOE_ERR_INVALID, "NULL or unaligned pointer");
  if ((st = set_device(h)) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // a copy into this layer still in flight must finish before its slots change hands
  if ((st = pf_join(h, layer, s)) != MOE_OK) return st;
  CK(h, launch_lookahead(static_cast<const uint16_t*>(x), h->router[layer], T, h->cfg.num_experts,
                         h->cfg.hidden, h->cfg.top_k, h->tab[layer], h->cfg.num_slots, h->cfg.prefetch_n,
                         slot_bytes(h), h->pred_logits, h->pred_ids, h->pred_w, h->pred_done, s));
  if (h->audit_each)
    CK(h, launch_audit(h->tab[layer], h->cfg.num_experts, h->cfg.num_slots, h->status, h->ffn_sync, s));
  return pf_fork(h, layer, s);
}

moe_status_t moe_offload_read_prefetch(moe_offload_t h, int layer, int32_t* cand, int* n_cand, int32_t* experts,
                                       int32_t* slots, int* n_installed, int cap) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  if (cap < 0) return fail(h, MOE_ERR_INVALID, "cap < 0");
  if ((st = set_device(h)) != MOE_OK) return st;
  CK(h, cudaDeviceSynchronize());
  const LayerTables& t = h->tab[layer];
  int32_t c[kNumCounts];
  CK(h, cudaMemcpy(c, t.counts, sizeof(c), cudaMemcpyDeviceToHost));
  if (n_cand) *n_cand = c[kCntCandidates];
  if (n_installed) *n_installed = c[kCntPrefetch];
  const int E = h->cfg.num_experts;
  const int nc = std::min(std::max(c[kCntCandidates], 0), std::min(cap, E));
  const int ni = std::min(std::max(c[kCntPrefetch], 0), std::min(cap, E));
  if (nc > 0 && cand) CK(h, cudaMemcpy(cand, t.pf_cand, sizeof(int32_t) * nc, cudaMemcpyDeviceToHost));
  if (ni > 0 && experts) CK(h, cudaMemcpy(experts, t.pf_expert, sizeof(int32_t) * ni, cudaMemcpyDeviceToHost));
  if (ni > 0 && slots) CK(h, cudaMemcpy(slots, t.pf_slot, sizeof(int32_t) * ni, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

int moe_offload_plan_static(const uint64_t* counts, int num_experts, int num_slots, int32_t* experts_out) {
  if (!counts || !experts_out || num_experts < 1 || num_slots < 1) return -1;
  std::vector<int> order(num_experts);
  for (int e = 0; e < num_experts; ++e) order[e] = e;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return counts[a] > counts[b]; });
  const int n = std::min(num_slots, num_experts);
  for (int i = 0; i < n; ++i) experts_out[i] = order[i];
  return n;
}

moe_status_t moe_offload_set_placement(moe_offload_t h, int layer, const int32_t* experts, int n,
                                       moe_stream_t stream) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  const int E = h->cfg.num_experts, S = h->cfg.num_slots;
  if (n < 1 || n > S || !experts) return fail(h, MOE_ERR_INVALID, "placement of %d experts into %d slots", n, S);
  std::vector<int32_t> se(S, -1), es(E, -1), ms(E, 0), me(E, 0);
  for (int i = 0; i < n; ++i) {
    const int e = experts[i];
    if (e < 0 || e >= E || es[e] >= 0) return fail(h, MOE_ERR_INVALID, "placement entry %d (expert %d) out of range or repeated", i, e);
    se[i] = e;
    es[e] = i;
    me[i] = e;
    ms[i] = i;
  }
  if ((st = set_device(h)) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (capturing(s)) return fail(h, MOE_ERR_CAPTURE, "set_placement under stream capture");
  CK(h, cudaDeviceSynchronize());  // nothing in flight may still use this layer's slots
  h->pf_pending[layer] = 0;
  const LayerTables& t = h->tab[layer];
  std::vector<uint32_t> zero(S, 0u);
  // The placement is installed as one call's miss list (slot i <- experts[i]) and copied by the
  // miss-copy kernel; then the layer is frozen: later calls hit or spill, never install.
  int32_t c[kNumCounts] = {0};
  c[kCntMiss] = n;
  c[kCntInstall] = n;
  c[kCntDistinct] = n;
  c[kCntFrozen] = 1;
  CK(h, cudaMemcpy(t.slot_expert, se.data(), sizeof(int32_t) * S, cudaMemcpyHostToDevice));
  CK(h, cudaMemcpy(t.expert_slot, es.data(), sizeof(int32_t) * E, cudaMemcpyHostToDevice));
  CK(h, cudaMemcpy(t.stamp, zero.data(), sizeof(uint32_t) * S, cudaMemcpyHostToDevice));
  CK(h, cudaMemcpy(t.miss_expert, me.data(), sizeof(int32_t) * E, cudaMemcpyHostToDevice));
  CK(h, cudaMemcpy(t.miss_slot, ms.data(), sizeof(int32_t) * E, cudaMemcpyHostToDevice));
  CK(h, cudaMemcpy(t.counts, c, sizeof(c), cudaMemcpyHostToDevice));
  if ((st = do_copy(h, layer, s)) != MOE_OK) return st;
  CK(h, cudaStreamSynchronize(s));
  h->frozen[layer] = 1;
  return MOE_OK;
}

moe_status_t moe_offload_read_route_counts(moe_offload_t h, int layer, uint64_t* counts) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  if (!counts) return fail(h, MOE_ERR_INVALID, "counts is NULL");
  if ((st = set_device(h)) != MOE_OK) return st;
  CK(h, cudaDeviceSynchronize());
  CK(h, cudaMemcpy(counts, h->tab[layer].route_counts, sizeof(uint64_t) * h->cfg.num_experts,
                   cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status_t moe_offload_read_slot(moe_offload_t h, int layer, int slot, void* w13_out, void* w2_out) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  if (slot < 0 || slot >= h->cfg.num_slots)
    return fail(h, MOE_ERR_INVALID, "slot %d outside [0, %d)", slot, h->cfg.num_slots);
  if ((st = set_device(h)) != MOE_OK) return st;
  CK(h, cudaDeviceSynchronize());
  if (w13_out)
    CK(h, cudaMemcpy(w13_out, h->lw[layer].slot_w13 + (size_t)slot * h->e13_bytes, h->e13_bytes,
                     cudaMemcpyDeviceToHost));
  if (w2_out)
    CK(h, cudaMemcpy(w2_out, h->lw[layer].slot_w2 + (size_t)slot * h->e2_bytes, h->e2_bytes,
                     cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status_t moe_offload_read_slot_scales(moe_offload_t h, int layer, int slot, float* s13_out, float* s2_out) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  if (h->fmt != 1) return fail(h, MOE_ERR_INVALID, "slot scales exist for block-scaled formats only");
  if (slot < 0 || slot >= h->cfg.num_slots)
    return fail(h, MOE_ERR_INVALID, "slot %d outside [0, %d)", slot, h->cfg.num_slots);
  if ((st = set_device(h)) != MOE_OK) return st;
  CK(h, cudaDeviceSynchronize());
  if (s13_out)
    CK(h, cudaMemcpy(s13_out, h->lw[layer].slot_s13 + (size_t)slot * h->f13, sizeof(float) * h->f13,
                     cudaMemcpyDeviceToHost));
  if (s2_out)
    CK(h, cudaMemcpy(s2_out, h->lw[layer].slot_s2 + (size_t)slot * h->f2, sizeof(float) * h->f2,
                     cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status_t moe_offload_set_shared_expert(moe_offload_t h, int layer, const void* w13, const float* s13,
                                           const void* w2, const float* s2) {
  moe_status_t st = check_layer(h, layer);
  if (st != MOE_OK) return st;
  if (!h->cfg.shared_expert) return fail(h, MOE_ERR_INVALID, "handle was created without a shared expert");
  if (!w13 || !w2 || !aligned16(w13) || !aligned16(w2))
    return fail(h, MOE_ERR_INVALID, "NULL or unaligned shared expert weights");
  if (h->fmt == 1 && (!s13 || !s2 || !aligned4(s13) || !aligned4(s2)))
    return fail(h, MOE_ERR_INVALID, "FP8 shared expert needs both scale tables");
  if (h->fmt == 0 && (s13 || s2)) return fail(h, MOE_ERR_INVALID, "scale tables are only for block-scaled formats");
  LayerWeights& lw = h->lw[layer];
  lw.sh_w13 = static_cast<const uint8_t*>(w13);
  lw.sh_w2 = static_cast<const uint8_t*>(w2);
  lw.sh_s13 = s13;
  lw.sh_s2 = s2;
  h->shared_set[layer] = 1;
  return MOE_OK;
}

moe_status_t moe_offload_reset(moe_offload_t h) {
  if (!h) return MOE_ERR_INVALID;
  moe_status_t st = set_device(h);
  if (st != MOE_OK) return st;
  CK(h, cudaDeviceSynchronize());
  std::fill(h->pf_pending.begin(), h->pf_pending.end(), 0);
  prefill_forget(&h->prefill);
  CK(h, cudaMemset(h->ffn_sync, 0, sizeof(uint32_t) * kFfnSyncWords));
  return init_tables(h);
}

moe_status_t moe_offload_host_alloc(size_t bytes, void** ptr) {
  if (!ptr) return fail(nullptr, MOE_ERR_INVALID, "ptr is NULL");
  *ptr = nullptr;
  void* p = nullptr;
  cudaError_t e = cudaHostAlloc(&p, bytes ? bytes : 16, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(nullptr, MOE_ERR_OOM, "cudaHostAlloc of %zu bytes: %s", bytes, cudaGetErrorString(e));
  }
  *ptr = p;
  return MOE_OK;
}

void moe_offload_host_free(void* ptr) {
  if (ptr) cudaFreeHost(ptr);
}

moe_status_t moe_offload_prefill_gemm_ms(moe_offload_t h, float* gemm_kernels_ms) {
  if (!h || !gemm_kernels_ms) return MOE_ERR_INVALID;
  moe_status_t st = set_device(h);
  if (st != MOE_OK) return st;
  if (h->prefill.last_staged < 0) return fail(h, MOE_ERR_INVALID, "no prefill call on this handle yet");
  if (!h->prefill.last_tc) return fail(h, MOE_ERR_INVALID, "the last prefill call did not run the tensor-core GEMMs");
  cudaError_t e = prefill_gemm_ms(&h->prefill, gemm_kernels_ms);
  if (e != cudaSuccess) return cuda_fail(h, e, "prefill GEMM events");
  return MOE_OK;
}

moe_status_t moe_offload_prefill_times(moe_offload_t h, float* route_ms, float* copy_ms, float* gemm_ms,
                                       float* combine_ms, int* staged) {
  if (!h) return MOE_ERR_INVALID;
  moe_status_t st = set_device(h);
  if (st != MOE_OK) return st;
  float ms[4] = {0, 0, 0, 0};
  int stg = -1;
  cudaError_t e = prefill_times(&h->prefill, ms, &stg);
  if (stg < 0) return fail(h, MOE_ERR_INVALID, "no prefill call on this handle yet");
  if (e != cudaSuccess) return cuda_fail(h, e, "prefill events");
  if (route_ms) *route_ms = ms[0];
  if (copy_ms) *copy_ms = ms[1];
  if (gemm_ms) *gemm_ms = ms[2];
  if (combine_ms) *combine_ms = ms[3];
  if (staged) *staged = stg;
  return MOE_OK;
}

size_t moe_offload_device_bytes(moe_offload_t h) { return h ? h->dev_bytes : 0; }

moe_status_t moe_offload_get_config(moe_offload_t h, moe_offload_config_t* cfg, size_t* auto_free_bytes) {
  if (!h) return MOE_ERR_INVALID;
  if (cfg) *cfg = h->cfg;
  if (auto_free_bytes) *auto_free_bytes = h->auto_free;
  return MOE_OK;
}

moe_status_t moe_offload_read_routing(moe_offload_t h, int32_t* ids, float* w, int32_t* slot_ids, int cap,
                                      int* n_pairs) {
  if (!h) return MOE_ERR_INVALID;
  if (cap < 0) return fail(h, MOE_ERR_INVALID, "cap < 0");
  moe_status_t st = set_device(h);
  if (st != MOE_OK) return st;
  CK(h, cudaDeviceSynchronize());
  if (n_pairs) *n_pairs = h->last_tk;
  const int n = std::min(cap, h->last_tk);
  if (n > 0 && ids) CK(h, cudaMemcpy(ids, h->ids_buf, sizeof(int32_t) * n, cudaMemcpyDeviceToHost));
  if (n > 0 && w) CK(h, cudaMemcpy(w, h->w_buf, sizeof(float) * n, cudaMemcpyDeviceToHost));
  if (n > 0 && slot_ids) CK(h, cudaMemcpy(slot_ids, h->slot_buf, sizeof(int32_t) * n, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

moe_status_t moe_offload_host_read_gbs(int device, const void* host_ptr, size_t bytes, int reps, double* best_gbs) {
  if (!host_ptr || !best_gbs || reps < 1 || bytes < 16 || bytes % 16 != 0 || !aligned16(host_ptr))
    return fail(nullptr, MOE_ERR_INVALID, "host_read_gbs: NULL, unaligned or empty buffer, or reps < 1");
  *best_gbs = 0.0;
  cudaError_t e = cudaSetDevice(device);
  void* dp = nullptr;
  if (e == cudaSuccess) e = cudaHostGetDevicePointer(&dp, const_cast<void*>(host_ptr), 0);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return fail(nullptr, MOE_ERR_INVALID, "host_read_gbs: not pinned, mapped host memory: %s", cudaGetErrorString(e));
  }
  int sms = 0;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess)
    return fail(nullptr, MOE_ERR_CUDA, "host_read_gbs: %s", cudaGetErrorString(e));
  unsigned* sink = nullptr;
  cudaEvent_t a = nullptr, b = nullptr;
  cudaStream_t st = nullptr;
  e = cudaMalloc(&sink, sizeof(unsigned));
  if (e == cudaSuccess) e = cudaEventCreate(&a);
  if (e == cudaSuccess) e = cudaEventCreate(&b);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
  float best = 0.0f;
  for (int r = 0; r <= reps && e == cudaSuccess; ++r) {  // the first read is a warm-up
    e = cudaEventRecord(a, st);
    if (e == cudaSuccess) e = launch_host_touch(dp, bytes, sink, 2 * sms, st);
    if (e == cudaSuccess) e = cudaEventRecord(b, st);
    if (e == cudaSuccess) e = cudaEventSynchronize(b);
    float ms = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
    if (e == cudaSuccess && r > 0 && (best == 0.0f || ms < best)) best = ms;
  }
  if (st) cudaStreamDestroy(st);
  if (a) cudaEventDestroy(a);
  if (b) cudaEventDestroy(b);
  if (sink) cudaFree(sink);
  if (e != cudaSuccess) return fail(nullptr, MOE_ERR_CUDA, "host_read_gbs: %s", cudaGetErrorString(e));
  *best_gbs = (double)bytes / ((double)best * 1e-3) / 1e9;
  return MOE_OK;
}

moe_status_t moe_offload_debug_wait(moe_offload_t h, long long limit_ns, int stall) {
  if (!h) return MOE_ERR_INVALID;
  if (limit_ns < 0 || (stall != 0 && stall != 1))
    return fail(h, MOE_ERR_INVALID, "debug_wait: limit_ns=%lld stall=%d", limit_ns, stall);
  h->wait_ns = limit_ns ? (unsigned long long)limit_ns : kDefaultWaitNs;
  h->stall = stall;
  return MOE_OK;
}

}  // extern "C"

namespace {
// The records' unset values: ~0 for the fields stamped with a minimum, 0 for the others.
moe_status_t trace_reset(moe_offload* h) {
  static_assert(MOE_TRACE_FIELDS == kTraceFields, "trace record size");
  std::vector<unsigned long long> v((size_t)h->cfg.num_layers * kTraceFields, 0ull);
  for (size_t i = 0; i < v.size(); ++i)
    if (kTraceMinFields & (1u << (i % kTraceFields))) v[i] = ~0ull;
  CK(h, cudaMemcpy(h->trace, v.data(), v.size() * sizeof(v[0]), cudaMemcpyHostToDevice));
  return MOE_OK;
}
}  // namespace

extern "C" {

moe_status_t moe_offload_trace_enable(moe_offload_t h, int on) {
  if (!h) return MOE_ERR_INVALID;
  if (on != 0 && on != 1) return fail(h, MOE_ERR_INVALID, "trace_enable: on=%d", on);
  moe_status_t st = set_device(h);
  if (st != MOE_OK) return st;
  if (on) {
    if (!h->trace &&
        (st = dev_alloc(h, &h->trace, sizeof(unsigned long long) * (size_t)h->cfg.num_layers * kTraceFields)) !=
            MOE_OK)
      return st;
    if ((st = trace_reset(h)) != MOE_OK) return st;
  }
  h->trace_on = on;
  return MOE_OK;
}

moe_status_t moe_offload_trace_read(moe_offload_t h, uint64_t* out, int reset) {
  if (!h || !out) return MOE_ERR_INVALID;
  if (!h->trace) return fail(h, MOE_ERR_INVALID, "trace_read: the trace was never enabled");
  moe_status_t st = set_device(h);
  if (st != MOE_OK) return st;
  CK(h, cudaDeviceSynchronize());
  CK(h, cudaMemcpy(out, h->trace, sizeof(uint64_t) * (size_t)h->cfg.num_layers * kTraceFields,
                   cudaMemcpyDeviceToHost));
  return reset ? trace_reset(h) : MOE_OK;
}

const char* moe_offload_last_error(moe_offload_t h) {
  return h ? h->err.c_str() : g_create_error.c_str();
}

moe_status_t moe_offload_profile_read(moe_offload_t h, int layer, long long* calls, double* head_ms,
                                      double* gate_up_ms, double* down_ms, int clear) {
  if (!h) return MOE_ERR_INVALID;
  if (layer >= h->cfg.num_layers) return fail(h, MOE_ERR_INVALID, "layer %d out of range", layer);
  moe_status_t st = set_device(h);
  if (st != MOE_OK) return st;
  if ((st = profile_fold(h)) != MOE_OK) return st;
  std::array<double, 4> acc{0.0, 0.0, 0.0, 0.0};
  for (int l = 0; l < h->cfg.num_layers; ++l) {
    if (layer >= 0 && l != layer) continue;
    for (int i = 0; i < 4; ++i) acc[i] += h->prof_sum[l][i];
    if (clear) h->prof_sum[l] = {0.0, 0.0, 0.0, 0.0};
  }
  if (calls) *calls = (long long)acc[0];
  if (head_ms) *head_ms = acc[1];
  if (gate_up_ms) *gate_up_ms = acc[2];
  if (down_ms) *down_ms = acc[3];
  return MOE_OK;
}

void moe_offload_destroy(moe_offload_t h) {
  if (!h) return;
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  if (h->profile) {
    (void)profile_fold(h);
    for (size_t l = 0; l < h->prof_sum.size(); ++l) {
      const auto& acc = h->prof_sum[l];
      if (acc[0] > 0.0)
        fprintf(stderr, "moe_offload profile: layer %zu: %.0f calls, mean head %.2f us, gate/up %.2f us, down %.2f us\n",
                l, acc[0], 1e3 * acc[1] / acc[0], 1e3 * acc[2] / acc[0], 1e3 * acc[3] / acc[0]);
    }
  }
  for (cudaEvent_t e : h->prof_pool) cudaEventDestroy(e);
  prefill_destroy(&h->prefill);
  for (cudaEvent_t e : h->pf_ready)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : h->pf_done)
    if (e) cudaEventDestroy(e);
  if (h->pf_stream) cudaStreamDestroy(h->pf_stream);
  for (void* p : h->allocations) cudaFree(p);
  for (void* p : h->registered) cudaHostUnregister(p);
  (void)cudaGetLastError();
  delete h;
}

}  // extern "C"

// ---- decode step as one CUDA graph ---------------------------------------
struct moe_offload_graph {
  moe_offload* h = nullptr;
  int T = 0;
  const uint16_t* x = nullptr;
  uint16_t* out = nullptr;
  int timing = 0;
  int kernels = 0;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  std::vector<cudaEvent_t> ev;  // 4 per layer: before the head, gate/up, down; after down
};

namespace {

void graph_free(moe_offload_graph* g) {
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  for (cudaEvent_t e : g->ev)
    if (e) cudaEventDestroy(e);
  delete g;
}

// Records the whole decode step on stream cs, which is capturing.
moe_status_t capture_step(moe_offload* h, moe_offload_graph* g, cudaStream_t cs) {
  const int L = h->cfg.num_layers, T = g->T, H = h->cfg.hidden;
  auto mark = [&](int i) -> cudaError_t {
    return g->timing ? cudaEventRecordWithFlags(g->ev[i], cs, cudaEventRecordExternal) : cudaSuccess;
  };
  moe_status_t st;
  for (int l = 0; l < L; ++l) {
    const uint16_t* x = g->x + (size_t)l * T * H;
    uint16_t* out = g->out + (size_t)l * T * H;
    CK(h, mark(4 * l + 0));
    if ((st = do_decode_head(h, l, x, T, cs, !g->timing)) != MOE_OK) return st;
    CK(h, mark(4 * l + 1));
    if ((st = pf_join(h, l, cs)) != MOE_OK) return st;
    FfnArgs a = ffn_args(h, l, x, h->slot_buf, h->w_buf, T, out);
    a.copy_through = 1;
    a.pdl = g->timing ? 0 : h->pdl;  // event nodes sit between the launches of a timing graph
    a.sync = early_down_sync(h, a.pdl);
    CK(h, launch_grouped_ffn_phase(a, 0, cs));
    if (lookahead_on(h, l) && (st = pf_fork(h, l + 1, cs)) != MOE_OK) return st;
    CK(h, mark(4 * l + 2));
    CK(h, launch_grouped_ffn_phase(a, 1, cs));
    CK(h, mark(4 * l + 3));
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_offload_graph_create(moe_offload_t h, int T, const void* x, void* out, int timing,
                                      moe_offload_graph_t* gout) {
  if (!h || !gout) return MOE_ERR_INVALID;
  *gout = nullptr;
  if (T < 1 || T > h->cfg.max_tokens_graph)
    return fail(h, MOE_ERR_INVALID, "graph batch T=%d outside [1, %d]", T, h->cfg.max_tokens_graph);
  if (!x || !out || !aligned16(x) || !aligned16(out))
    return fail(h, MOE_ERR_INVALID, "NULL or unaligned graph buffer");
  moe_status_t st = check_shared(h, 0, h->cfg.num_layers);
  if (st != MOE_OK) return st;
  if ((st = set_device(h)) != MOE_OK) return st;
  moe_offload_graph* g = new (std::nothrow) moe_offload_graph();
  if (!g) return fail(h, MOE_ERR_OOM, "out of host memory");
  g->h = h;
  g->T = T;
  g->x = static_cast<const uint16_t*>(x);
  g->out = static_cast<uint16_t*>(out);
  g->timing = timing ? 1 : 0;
  g->kernels = 0;
  for (int l = 0; l < h->cfg.num_layers; ++l) g->kernels += launches_per_layer(h, l);
  if (g->timing) {
    g->ev.resize((size_t)4 * h->cfg.num_layers, nullptr);
    for (auto& e : g->ev) {
      cudaError_t ce = cudaEventCreate(&e);
      if (ce != cudaSuccess) {
        graph_free(g);
        return cuda_fail(h, ce, "cudaEventCreate");
      }
    }
  }
  cudaStream_t cs = nullptr;
  cudaError_t ce = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (ce != cudaSuccess) {
    graph_free(g);
    return cuda_fail(h, ce, "cudaStreamCreate");
  }
  ce = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (ce != cudaSuccess) {
    cudaStreamDestroy(cs);
    graph_free(g);
    return cuda_fail(h, ce, "cudaStreamBeginCapture");
  }
  st = capture_step(h, g, cs);
  cudaGraph_t graph = nullptr;
  ce = cudaStreamEndCapture(cs, &graph);
  for (int& p : h->pf_pending)
    if (p == 2) p = 0;  // a failed capture leaves no copy behind
  g->graph = graph;
  cudaStreamDestroy(cs);
  if (st != MOE_OK) {
    graph_free(g);
    return st;
  }
  if (ce != cudaSuccess) {
    graph_free(g);
    return cuda_fail(h, ce, "cudaStreamEndCapture");
  }
  ce = cudaGraphInstantiate(&g->exec, g->graph, cudaGraphInstantiateFlagUseNodePriority);
  if (ce != cudaSuccess) {
    graph_free(g);
    return cuda_fail(h, ce, "cudaGraphInstantiate");
  }
  *gout = g;
  return MOE_OK;
}

moe_status_t moe_offload_graph_launch(moe_offload_graph_t g, moe_stream_t stream) {
  if (!g) return MOE_ERR_INVALID;
  moe_offload* h = g->h;
  moe_status_t st = set_device(h);
  if (st != MOE_OK) return st;
  CK(h, cudaGraphLaunch(g->exec, reinterpret_cast<cudaStream_t>(stream)));
  h->last_tk = g->T * h->cfg.top_k;
  return MOE_OK;
}

moe_status_t moe_offload_graph_launch_host(moe_offload_graph_t g, const void* x_host, void* out_host,
                                           moe_stream_t stream) {
  if (!g || !x_host || !out_host) return MOE_ERR_INVALID;
  moe_offload* h = g->h;
  moe_status_t st = set_device(h);
  if (st != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)h->cfg.num_layers * g->T * h->cfg.hidden * 2;
  CK(h, cudaMemcpyAsync(const_cast<uint16_t*>(g->x), x_host, bytes, cudaMemcpyHostToDevice, s));
  CK(h, cudaGraphLaunch(g->exec, s));
  h->last_tk = g->T * h->cfg.top_k;
  CK(h, cudaMemcpyAsync(out_host, g->out, bytes, cudaMemcpyDeviceToHost, s));
  CK(h, cudaStreamSynchronize(s));
  return MOE_OK;
}

moe_status_t moe_offload_graph_times(moe_offload_graph_t g, float* head_ms, float* gate_up_ms,
                                     float* down_ms) {
  if (!g) return MOE_ERR_INVALID;
  moe_offload* h = g->h;
  if (!g->timing) return fail(h, MOE_ERR_INVALID, "graph was created without timing");
  moe_status_t st = set_device(h);
  if (st != MOE_OK) return st;
  CK(h, cudaEventSynchronize(g->ev.back()));
  float* dst[3] = {head_ms, gate_up_ms, down_ms};
  for (int l = 0; l < h->cfg.num_layers; ++l) {
    for (int p = 0; p < 3; ++p) {
      if (!dst[p]) continue;
      float ms = 0.0f;
      CK(h, cudaEventElapsedTime(&ms, g->ev[4 * l + p], g->ev[4 * l + p + 1]));
      dst[p][l] = ms;
    }
  }
  return MOE_OK;
}

int moe_offload_graph_kernel_count(moe_offload_graph_t g) { return g ? g->kernels : 0; }

void moe_offload_graph_destroy(moe_offload_graph_t g) {
  if (!g) return;
  cudaSetDevice(g->h->device);
  cudaDeviceSynchronize();
  graph_free(g);
}

}  // extern "C"
