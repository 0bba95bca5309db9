/*
 * moe_offload.h — C ABI of the offloaded Mixture-of-Experts layer for GB300 (sm_103a).
 *
 * Routed expert weights stay in host RAM, pinned and mapped into the GPU's
 * address space; every MoE layer keeps a fixed number of GPU expert slots.
 * A decode step of one layer is:
 *
 *   moe_offload_route_topk   router logits, softmax, top-k
 *   moe_offload_slot_ensure  LRU lookup in the layer's GPU slot table, victim
 *                            choice for misses, expert id -> slot id rewrite,
 *                            miss list and miss count written to device memory
 *   moe_offload_miss_copy    missing experts copied from mapped host memory into
 *                            their slots by SM loads; the count is read on the GPU
 *   moe_offload_grouped_ffn  gate+up+SiLU, down projection and weighted combine
 *                            over the [num_slots, N, K] slot tensors
 *
 * ("MoE expert offload" page of xinfer-ai 0.14.6, section "How it works"; the
 * fused gate+up+SiLU expert FFN follows the "MoE-Infinity" page's feature list.)
 * moe_offload_decode_layer chains the four on one stream with no host
 * synchronisation, so a whole decode step can be captured in a CUDA graph.
 *
 * Conventions for every call:
 *   - Device pointers are plain CUDA device addresses (cudaMalloc or any
 *     allocator on the handle's device); the caller owns them.
 *   - bf16 tensors are raw 16-bit patterns; every tensor is dense row-major
 *     with the last dimension contiguous; device pointers must be 16-byte aligned.
 *   - Streams are CUDA stream handles (cudaStream_t); NULL means the legacy
 *     default stream. All work is enqueued on the stream given, asynchronously,
 *     unless the comment says the call synchronises.
 *   - A call returns MOE_OK or an error code and never aborts the process;
 *     moe_offload_last_error() gives a one-line reason. Errors the GPU detects
 *     while running (a routed id outside [0, E), a slot id out of range, a
 *     failed audit) never trap: they set bits of the handle's device status
 *     word, which moe_offload_get_stats() returns as MOE_ERR_DEVICE_STATUS.
 *   - One handle serves one stream at a time; calls on one handle that overlap
 *     on the GPU race on its slot tables and scratch buffers.
 */
#ifndef MOE_OFFLOAD_H
#define MOE_OFFLOAD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_offload* moe_offload_t;
typedef struct CUstream_st* moe_stream_t; /* the same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = 1,       /* bad argument, size or configuration */
  MOE_ERR_CUDA = 2,          /* a CUDA runtime call failed (reason in last_error) */
  MOE_ERR_OOM = 3,           /* device or pinned allocation failed */
  MOE_ERR_CAPTURE = 4,       /* a host-synchronising path was asked for under stream capture */
  MOE_ERR_DEVICE_STATUS = 5  /* the GPU flagged an error; see moe_offload_stats_t.device_status */
} moe_status_t;

/* Expert weight formats.
 * MOE_DTYPE_FP8_E4M3_B128: block FP8 experts ("MoE expert offload" page,
 * "Supported" section: block-FP8 experts keep their weight and scale tensors in
 * host RAM like every other format). Codes are e4m3 (1 sign, 4 exponent bits
 * with bias 7, 3 mantissa bits, subnormals, 0x7F/0xFF NaN, largest 448); each
 * 128 x 128 block of a weight matrix has one fp32 scale; a weight is
 * f32(code) * scale. Weight-only: activations stay bf16, accumulation fp32. */
enum { MOE_DTYPE_BF16 = 0, MOE_DTYPE_FP8_E4M3_B128 = 1 };

/* Bits of the device status word. */
enum {
  MOE_DEV_BAD_EXPERT_ID = 1u << 0, /* slot_ensure saw a routed id outside [0, E); that id is skipped */
  MOE_DEV_BAD_SLOT_ID = 1u << 1,   /* grouped_ffn saw a slot id that is neither a slot nor a live spill marker */
  MOE_DEV_AUDIT_FAILED = 1u << 2,  /* moe_offload_audit found the slot table inconsistent */
  MOE_DEV_BAD_COUNT = 1u << 3,     /* a device-resident count exceeded its buffer */
  MOE_DEV_TIMEOUT = 1u << 4        /* a bounded wait inside a kernel ran out; that kernel's output is invalid */
};

typedef struct {
  int num_layers;       /* L >= 1 */
  int num_experts;      /* E, 1..1024 */
  int top_k;            /* k, 1..16 and <= E */
  int hidden;           /* H, multiple of 256, <= 8192 */
  int inter;            /* I (expert intermediate size), multiple of 64 */
  int num_slots;        /* S per layer, top_k <= S <= E (else MOE_ERR_INVALID); 0 = auto:
                           after its other allocations create reads the device's free memory
                           and takes S = moe_offload_slots_auto(free, auto_reserve_bytes, L, E,
                           top_k, bytes of one slot) (MOE_ERR_OOM when fewer than top_k fit);
                           moe_offload_get_config returns the S chosen */
  int dtype;            /* MOE_DTYPE_BF16, or MOE_DTYPE_FP8_E4M3_B128 (H and I multiples of 128) */
  int renormalize;      /* 1: weights = softmax over the k chosen logits;
                           0: weights = softmax over all E, taken at the k chosen */
  int max_tokens_graph; /* T bound of the graph-safe decode path, 1..64;
                           max_tokens_graph * (top_k + shared_expert) <= 1024 */
  int shared_expert;    /* 0, or 1: every layer has one always-resident shared expert of the
                           routed experts' shape and format, added to every token with weight 1
                           after the k routed ranks; set it with moe_offload_set_shared_expert */
  int prefetch_n;       /* router lookahead: 0 = off, else 1..num_slots experts per layer
                           predicted from the previous layer's input and prefetched
                           (see moe_offload_prefetch) */
  unsigned long long auto_reserve_bytes; /* num_slots = 0 only: device memory left free after the
                           slots ("MoE expert offload" page, Options table:
                           XINFER_MOE_OFFLOAD_RESERVE_GB, 2.5 by default); 0 = 2.5 GiB */
} moe_offload_config_t;

typedef struct {
  uint64_t calls;        /* slot_ensure calls */
  uint64_t hits;         /* distinct experts found resident, summed over calls */
  uint64_t misses;       /* distinct experts not resident (installed + spilled) */
  uint64_t spills;       /* misses that found no free slot and were read from host */
  uint64_t bytes_copied; /* bytes moved host -> slots by miss_copy */
  uint64_t staged_calls; /* prefill calls that staged the whole layer */
  uint64_t staged_bytes; /* bytes moved host -> staging */
  uint64_t prefetch_installs; /* experts installed by the router lookahead (not misses) */
  uint64_t prefetch_hits;     /* demand hits on a prefetched slot before its first use */
  uint64_t prefetch_bytes;    /* bytes those installs copied host -> slots */
  uint32_t device_status;/* OR of MOE_DEV_* bits */
} moe_offload_stats_t;

/* Slot count from a fraction of a layer's experts: max(k, floor(f * E)).
 * ("MoE expert offload" page, Options table: a fraction of each layer's experts
 * stays on the GPU, at least num_experts_per_tok.) Returns -1 when f is not in (0, 1]. */
int moe_offload_slots_for_fraction(double fraction, int num_experts, int top_k);

/* Slot count for `auto` sizing ("MoE expert offload" page, Options table: after
 * loading, every layer's slots grow evenly into the free VRAM, leaving a
 * reserve — 2.5 GB by default — for the KV cache and workspaces):
 *   S = min(E, floor((free_bytes - reserve_bytes) / (L * expert_bytes)))
 * where expert_bytes is what one slot holds (weights and scales of one
 * expert). Returns -1 when fewer than top_k slots per layer fit (offload cannot
 * run in that memory) or an argument is out of range. Host only. */
int moe_offload_slots_auto(size_t free_bytes, size_t reserve_bytes, int num_layers, int num_experts,
                           int top_k, size_t expert_bytes);

/* Create a handle on `device`.
 *   host_w13[l]: host array [E, 2I, H] of layer l (rows 0..I-1 gate, I..2I-1 up),
 *                bf16, or e4m3 bytes for MOE_DTYPE_FP8_E4M3_B128
 *   host_w2[l] : host array [E, H, I] of layer l, same element type
 *   host_scales13[l] / host_scales2[l]: FP8 only (NULL for bf16): host fp32
 *                arrays [E, 2I/128, H/128] and [E, H/128, I/128], 4-byte aligned,
 *                pinned and mapped like the weights; a slot holds its expert's
 *                scales beside its weights and they move together
 *   dev_router[l]: device array [E, H] bf16, the router of layer l
 * Host arrays must be 16-byte aligned. The caller owns them and keeps them
 * alive and unchanged until destroy; create registers any that are not yet
 * pinned as pinned, mapped memory (cudaHostRegister) and unregisters those at
 * destroy; it never copies them. The library allocates and owns the slot
 * tensors [S,2I,H] and [S,H,I] per layer, the slot tables, the miss lists, two
 * whole-layer staging buffers for prefill and its scratch. The slot tables start
 * empty. Before returning, create reads the whole host store once from the GPU
 * (on GB300 the first GPU pass over host pages the CPU had just written ran
 * well below the link rate; this moves that cost to load time). Errors: MOE_ERR_INVALID (config), MOE_ERR_OOM, MOE_ERR_CUDA; *out is
 * NULL on error, and everything create had allocated or registered is released.
 * Environment read at create: MOE_OFFLOAD_AUDIT=1 (see moe_offload_audit),
 * MOE_OFFLOAD_PDL=0 (no programmatic dependent launch in the decode chain),
 * MOE_OFFLOAD_EARLY_DOWN=0 (a decode step's down launch waits for the whole
 * gate/up launch instead of per expert, and a prefill call's down GEMM for the
 * whole gate/up GEMM instead of per row tile; outputs are identical either way),
 * MOE_OFFLOAD_PROFILE=1 (see moe_offload_profile_read), and
 * MOE_OFFLOAD_FAIL_ALLOC=n, host-side fault injection: the n-th device
 * allocation or host registration of create (from 0) fails with MOE_ERR_OOM
 * without being attempted. The prefill staging buffers are not counted.
 * Placement of the host arrays matters on GB300: GPU reads over NVLink-C2C of
 * pinned memory from moe_offload_host_alloc ran at 211 GB/s everywhere, while
 * registered pageable memory had address ranges read at 18-160 GB/s, and
 * memory on 512 MB transparent huge pages ran at 60-120 GB/s. Prefer
 * moe_offload_host_alloc for the store. */
moe_status_t moe_offload_create(const moe_offload_config_t* cfg, int device,
                                void* const* host_w13, void* const* host_w2,
                                const float* const* host_scales13,
                                const float* const* host_scales2,
                                const void* const* dev_router, moe_offload_t* out);

/* Router of layer `layer`: logits = x . W_r^T (fp32 accumulation), top-k on the
 * logits in descending order (equal logits: lower expert id first), softmax
 * weights per cfg->renormalize. ("MoE expert offload" page, "How it works":
 * the routed experts of each MoE call.)
 *   x  : device [T, H] bf16           ids: device [T, k] int32 (output)
 *   w  : device [T, k] fp32 (output)  T >= 0 (T = 0 enqueues nothing)
 * Graph-safe for T <= max_tokens_graph. */
moe_status_t moe_offload_route_topk(moe_offload_t h, int layer, const void* x, int T,
                                    int32_t* ids, float* w, moe_stream_t stream);

/* LRU slot table of layer `layer` ("MoE expert offload" page, "How it works":
 * look the routed experts up in a per-layer LRU table kept on the GPU, assign
 * least-recently-used slots to misses, rewrite expert ids to slot ids).
 * One launch of fixed shape; the table, the miss list and the miss count stay
 * in device memory. Per call: the clock advances by one; the call's distinct
 * ids are taken in ascending order; hits refresh their slot's stamp; each miss
 * takes, among slots not used by this call, the one with the smallest key
 * (occupied, stamp, slot index), so empty slots first, then the oldest. When
 * the call's distinct experts outnumber the slots, misses left without a slot
 * are not installed: their slot id is the spill marker S + spill index and
 * grouped_ffn reads them from host memory.
 *   ids     : device [T, k] int32 expert ids, T <= max_tokens_graph
 *   slot_ids: device [T, k] int32 (output) slot ids or spill markers
 * Ids outside [0, E) set MOE_DEV_BAD_EXPERT_ID and get slot id -1. */
moe_status_t moe_offload_slot_ensure(moe_offload_t h, int layer, const int32_t* ids, int T,
                                     int32_t* slot_ids, moe_stream_t stream);

/* Copy the experts installed by the last slot_ensure of `layer` from mapped
 * host memory into their slots ("MoE expert offload" page, "How it works":
 * a second kernel copies the missing experts straight from device-mapped
 * pinned host memory; it reads the miss count from device memory). Fixed grid
 * of 16-byte loads; with no misses it exits at once. */
moe_status_t moe_offload_miss_copy(moe_offload_t h, int layer, moe_stream_t stream);

/* Grouped expert FFN over the slot tensors of `layer` ("MoE expert offload"
 * page, "How it works": the GEMMs read [num_slots, N, K] slot tensors):
 * for every (t, j): g, u = W13[slot] x_t (fp32), h = silu(g) * u, y = W2[slot] h;
 * out_t = bf16( sum_{j=0..k-1} w[t,j] * y_{t,j} ), summed in rank order.
 * Spill markers read that expert's weights from host memory with the same
 * arithmetic, so the result never depends on where an expert lives.
 *   x: device [T,H] bf16; slot_ids: device [T,k] int32 from slot_ensure of the
 *   same call; w: device [T,k] fp32; out: device [T,H] bf16 (output).
 *   T <= max_tokens_graph. */
moe_status_t moe_offload_grouped_ffn(moe_offload_t h, int layer, const void* x,
                                     const int32_t* slot_ids, const float* w, int T,
                                     void* out, moe_stream_t stream);

/* One MoE layer: route_topk -> slot_ensure -> miss_copy -> grouped_ffn on
 * `stream`, using the handle's own id/weight buffers. For T <= max_tokens_graph
 * it never synchronises with the host and may be captured in a CUDA graph; it
 * then runs as three launches: router + top-k + slot ensure in one (the last
 * CTA of the router grid updates the table), the gate/up FFN, whose CTAs read
 * the experts installed by this call from host memory and write them into
 * their slots while the resident experts stream from HBM, and the down
 * projection + combine. Slot contents, tables and outputs are those of the
 * four separate entry points.
 * For larger T (prefill) it learns the call's distinct expert count on the host
 * (a synchronisation); when that count exceeds the slots it copies the whole
 * layer into a staging buffer and runs the grouped GEMM there, leaving the slot
 * table untouched ("MoE expert offload" page, "How it works", Prefill);
 * otherwise it runs the slot path. A staged call also starts staging layer + 1
 * into a second buffer, which the next call uses if it is that layer's and
 * stages too.
 * The prefill path under stream capture returns MOE_ERR_CAPTURE.
 *   x: device [T,H] bf16; out: device [T,H] bf16 (output). */
moe_status_t moe_offload_decode_layer(moe_offload_t h, int layer, const void* x, int T,
                                      void* out, moe_stream_t stream);

/* Check the slot table of `layer` on the GPU: slot_expert and expert_slot are
 * inverse maps, no stamp is newer than the clock, the miss list's slots hold
 * their experts; the grouped FFN's hand-off counters (the down launch of a
 * decode step waits on them per expert, not on the whole gate/up launch) are
 * zero between calls. A failure sets MOE_DEV_AUDIT_FAILED; nothing traps. With the
 * environment variable MOE_OFFLOAD_AUDIT=1 at create, every table update of the
 * handle (slot_ensure, prefetch, decode_layer, the decode graph) is followed by
 * this audit on the same stream (graph_kernel_count includes those launches).
 * (Slot-map audit mode, FreeToken issue 677.) */
moe_status_t moe_offload_audit(moe_offload_t h, int layer, moe_stream_t stream);

/* Counters of `layer`, or summed over all layers when layer < 0. Synchronises
 * the device. Returns MOE_ERR_DEVICE_STATUS when the device status word is
 * non-zero (the stats are filled in all the same). */
moe_status_t moe_offload_get_stats(moe_offload_t h, int layer, moe_offload_stats_t* stats);

/* Host-side fault injection for the audit: overwrite one word of the slot table
 * of `layer` (synchronises the device first, then copies the word).
 *   table MOE_TABLE_SLOT_EXPERT: index < S, value in [-1, E);
 *   table MOE_TABLE_EXPERT_SLOT: index < E, value in [-1, S);
 *   table MOE_TABLE_STAMP:       index < S, value in [0, 2^32);
 *   table MOE_TABLE_CLOCK:       index 0,   value in [0, 2^32).
 * Anything else returns MOE_ERR_INVALID and writes nothing, so a table written
 * this way may be inconsistent (moe_offload_audit reports it) but never sends a
 * kernel out of bounds. Outputs computed from an inconsistent table are
 * unspecified until moe_offload_reset. (Test support for the slot-map audit of
 * FreeToken issue 677; no counterpart on the pages.) */
enum { MOE_TABLE_SLOT_EXPERT = 0, MOE_TABLE_EXPERT_SLOT = 1, MOE_TABLE_STAMP = 2, MOE_TABLE_CLOCK = 3 };
moe_status_t moe_offload_debug_write_table(moe_offload_t h, int layer, int table, int index, int64_t value);

/* Eager decode profile. With MOE_OFFLOAD_PROFILE=1 at create, every
 * decode_layer call on the decode path (T <= max_tokens_graph) outside stream
 * capture records CUDA events before its head launch, after it, after the
 * gate/up launch and after the down launch. The events sit between the launches,
 * so the profiled step runs without launch overlap; graphs captured from the
 * handle are not profiled (moe_offload_graph_create's timing mode is their
 * split). This call waits for the recorded events and returns, for `layer` or
 * summed over all layers when layer < 0, the profiled calls and the summed
 * milliseconds of the three phases since create or the last read with
 * clear != 0. destroy prints the per-layer means to stderr. Any output pointer
 * may be NULL. Without the variable, calls is 0. (The per-call time split of
 * the "MoE expert offload" page, "Options" table, XINFER_MOE_OFFLOAD_PROFILE:
 * a diagnostic mode that gives up graphs and launch overlap.) */
moe_status_t moe_offload_profile_read(moe_offload_t h, int layer, long long* calls, double* head_ms,
                                      double* gate_up_ms, double* down_ms, int clear);

/* Copy the slot table of `layer` to host arrays (synchronises the device):
 * slot_expert[S] (-1 = empty), expert_slot[E] (-1 = not resident), stamp[S],
 * *clock. Any pointer may be NULL. */
moe_status_t moe_offload_read_table(moe_offload_t h, int layer, int32_t* slot_expert,
                                    int32_t* expert_slot, uint32_t* stamp, uint32_t* clock);

/* Copy the miss list of the last slot_ensure of `layer` (synchronises):
 * entries i < *miss_count are (miss_expert[i], miss_slot[i]), installs first in
 * ascending expert id, then spills with slot = S + spill index. At most `cap`
 * entries are written. */
moe_status_t moe_offload_read_misses(moe_offload_t h, int layer, int32_t* miss_expert,
                                     int32_t* miss_slot, int cap, int* miss_count,
                                     int* spill_count);

/* Router lookahead and prefetch install into `layer` (FreeToken issue #677,
 * "Proposal": the next layer's router run on the current layer's input predicts
 * the next layer's experts, which are copied while the current layer computes).
 * x [T, H] bf16 (device, 16-byte aligned) is the input of layer - 1; layer >= 1,
 * 1 <= T <= max_tokens_graph; needs a handle with prefetch_n > 0.
 *   1. logits = x . W_r(layer)^T, per-token top-k (the routing rule of route_topk);
 *   2. candidates: the distinct predicted experts in descending order of their
 *      largest predicted logit over the tokens (equal: lower expert id first);
 *   3. on `stream`: the first prefetch_n candidates not resident in `layer` are
 *      installed in its table at stamp 0 (held, unused, first to be evicted;
 *      the clock does not move; no miss is counted). Slots of resident
 *      candidates and slots filled by this install are never victims; each
 *      install takes the free slot with the smallest (occupied, stamp, index);
 *   4. their weights (and FP8 scales) are copied from host into the slots on the
 *      library's high-priority copy stream, after the work enqueued on `stream`.
 * The next call that reads or writes `layer`'s slots (grouped_ffn, miss_copy,
 * decode_layer, prefetch) makes its stream wait for that copy; under stream
 * capture the copy and that call must be in the same capture (else
 * MOE_ERR_CAPTURE). decode_layer(l) and the decode graph do all of this for
 * layer l + 1 inside their fused first kernel when prefetch_n > 0: every table
 * write stays on the compute stream. */
moe_status_t moe_offload_prefetch(moe_offload_t h, int layer, const void* x, int T, moe_stream_t stream);

/* Static expert placement (the "PolyStrata" page, workflow steps 1-3: profile which
 * experts each layer routes to, derive the slots that fit, place the most frequently used
 * experts in them): an alternative to LRU eviction for a layer.
 *
 * moe_offload_read_route_counts: counts[0..E) of routed (token, rank) pairs per expert of
 * `layer`, summed over every slot_ensure / decode call since create or reset (the profile).
 * Synchronises the device.
 *
 * moe_offload_plan_static: host only. The `top` policy: experts_out[0..n) = the num_slots
 * experts with the largest counts (equal counts: lower expert id first), n = min(num_slots,
 * num_experts); returns n, or -1 on a bad argument.
 *
 * moe_offload_set_placement: slot i of `layer` receives experts[i] (0 <= i < n <= S, distinct
 * ids), copied from host memory; the other slots are emptied; then the layer is frozen: every
 * later call hits a placed expert or spills the others (slot id S + spill index, read from
 * host memory by the FFN, counted as misses and spills), installs nothing and takes no
 * prefetch, and its prefill calls always stage. Outputs are those of LRU (placement never
 * changes the arithmetic). Synchronises the device; not under capture. reset() returns every
 * layer to an empty LRU table. */
moe_status_t moe_offload_read_route_counts(moe_offload_t h, int layer, uint64_t* counts);
int moe_offload_plan_static(const uint64_t* counts, int num_experts, int num_slots, int32_t* experts_out);
moe_status_t moe_offload_set_placement(moe_offload_t h, int layer, const int32_t* experts, int n,
                                       moe_stream_t stream);

/* The last prefetch install into `layer`: its candidates (cand[0..*n_cand)) and
 * its installs (experts[i] into slots[i], i < *n_installed), each array holding
 * up to `cap` entries (any may be NULL). Synchronises the device. For tests. */
moe_status_t moe_offload_read_prefetch(moe_offload_t h, int layer, int32_t* cand, int* n_cand, int32_t* experts,
                                       int32_t* slots, int* n_installed, int cap);

/* Copy the contents of slot `slot` of `layer` to host buffers (synchronises):
 * w13_out receives 2*I*H weights, w2_out H*I (bf16, or e4m3 bytes for FP8
 * handles). Either may be NULL. For tests. */
moe_status_t moe_offload_read_slot(moe_offload_t h, int layer, int slot, void* w13_out, void* w2_out);

/* Copies the fp32 block scales slot `slot` of `layer` holds into s13_out
 * [2I/128, H/128] and s2_out [H/128, I/128] (either may be NULL). FP8 handles
 * only (else MOE_ERR_INVALID). Synchronises the device. For tests. */
moe_status_t moe_offload_read_slot_scales(moe_offload_t h, int layer, int slot, float* s13_out, float* s2_out);

/* Installs the shared expert of `layer` (handles created with shared_expert = 1):
 * device arrays w13 [2I, H] and w2 [H, I] in the handle's weight format (16-byte
 * aligned) and, for FP8, fp32 scales s13 [2I/128, H/128] and s2 [H/128, I/128]
 * (NULL for bf16). The caller owns them and keeps them alive and unchanged
 * until destroy; the shared expert is never in the slot table and never copied.
 * Every token of every later FFN call of the layer adds its output with weight 1
 * after the k routed ranks. Decode calls, grouped_ffn and graph_create return
 * MOE_ERR_INVALID while a layer of a shared-expert handle has none installed.
 * The prefill path (T > max_tokens_graph) of an FP8 or shared-expert handle always
 * stages the layer: FP8 weights are dequantised to bf16 (bf16(code x scale)) for
 * the bf16 tensor-core GEMMs, and the shared expert is one more group with one
 * pair per token, added after the k ranks. With a shared expert, at most 1023
 * routed experts. */
moe_status_t moe_offload_set_shared_expert(moe_offload_t h, int layer, const void* w13, const float* s13,
                                           const void* w2, const float* s2);

/* Empty every slot table, zero the counters and the device status word
 * (synchronises). Slot contents are left as they are and are never read again
 * before being overwritten. */
moe_status_t moe_offload_reset(moe_offload_t h);

/* Allocate `bytes` of pinned host memory, mapped into every GPU's address space
 * (cudaHostAlloc, mapped + portable), to hold a host expert store: create
 * uses it as it is, without registering. *ptr is 4096-byte aligned; NULL on
 * failure (MOE_ERR_OOM, reason in moe_offload_last_error(NULL)). Free it with
 * moe_offload_host_free after the handles that use it are destroyed. */
moe_status_t moe_offload_host_alloc(size_t bytes, void** ptr);
void moe_offload_host_free(void* ptr);

/* Phase times of the handle's last prefill call (decode_layer with T above
 * max_tokens_graph), in milliseconds, from CUDA events on its stream:
 * route = router + top-k + distinct count; copy = whole-layer staging copy
 * (staged) or slot ensure + miss copy (slot path); gemm = bucketing + the two
 * grouped GEMMs; combine = rank-order combine. *staged is 1 when the layer was
 * staged. Synchronises on that call. MOE_ERR_INVALID before any prefill call. */
moe_status_t moe_offload_prefill_times(moe_offload_t h, float* route_ms, float* copy_ms, float* gemm_ms,
                                       float* combine_ms, int* staged);

/* Time of the two tensor-core grouped GEMM launches (gate/up + SiLU, then the
 * down projection) of the handle's last prefill call, in milliseconds: from a
 * CUDA event recorded before the gate/up launch to one recorded after the down
 * launch, so bucketing and the row gather are not in it ("MoE expert offload"
 * page, "How it works", Prefill: the GEMMs on the staged layer or the slot
 * tensors). Synchronises on that call. MOE_ERR_INVALID before any prefill call,
 * or when the last one ran the CUDA-core GEMMs (shapes the 128 x 256 tensor-core
 * tiles do not cover: H not a multiple of 256 or I not a multiple of 128). */
moe_status_t moe_offload_prefill_gemm_ms(moe_offload_t h, float* gemm_kernels_ms);

/* Bytes of device memory the handle holds. */
size_t moe_offload_device_bytes(moe_offload_t h);

/* The handle's configuration as create fixed it (num_slots holds the S an
 * `auto` create chose) and, for num_slots = 0 at create, the free device bytes
 * the sizing read (else 0). Either pointer may be NULL. Host only. */
moe_status_t moe_offload_get_config(moe_offload_t h, moe_offload_config_t* cfg, size_t* auto_free_bytes);

/* Routing of the last decode-path call (decode_layer with T <= max_tokens_graph,
 * or a decode-graph replay, whose last layer it is): routed expert ids [T,k],
 * their weights [T,k] and the slot ids (or spill markers) the slot update wrote,
 * in the handle's own buffers ("MoE expert offload" page, "How it works": ids
 * rewritten to slot ids). *n_pairs = T*k of that call (0 before any); at most
 * `cap` entries of each array are written; any pointer may be NULL.
 * Synchronises the device. For tests that replay the GPU's own routed ids
 * through the LRU simulator. */
moe_status_t moe_offload_read_routing(moe_offload_t h, int32_t* ids, float* w, int32_t* slot_ids, int cap,
                                      int* n_pairs);

/* Zero-copy read ceiling of the host link (no counterpart on the pages; the
 * miss copy's SM loads are measured against it): reads `bytes` (a multiple of
 * 16) of pinned, mapped host memory at host_ptr (16-byte aligned) from `device`
 * with 16-byte SM loads over a grid of two CTAs per SM, once to warm up and then
 * `reps` times, and returns the best rate in GB/s (1e9 bytes per second).
 * Synchronises; allocates 4 device bytes and frees them. Errors:
 * MOE_ERR_INVALID (arguments, or memory that is not pinned and mapped; reason in
 * moe_offload_last_error(NULL)), MOE_ERR_CUDA. */
moe_status_t moe_offload_host_read_gbs(int device, const void* host_ptr, size_t bytes, int reps, double* best_gbs);

/* Bounded waits, for tests that make one run out (no counterpart on the pages).
 * In a decode step the down launch waits per expert group, on counters the
 * gate/up CTAs raise, and in a prefill call the down GEMM's CTAs wait per row
 * tile on counts the gate/up GEMM's CTAs raise, for at most limit_ns (0 = the
 * default, 2 s) per wait; when a wait runs out the kernel sets MOE_DEV_TIMEOUT,
 * computes on (a prefill down CTA whose wait ran out still loads and consumes
 * every stage of its ring, so no copy is left in flight, and writes no output),
 * and every later wait of the handle returns at once until moe_offload_reset, so
 * outputs are invalid while the bit is set. stall = 1 makes the first group's
 * wait of every decode down warp, and every prefill tile wait, target one
 * gate/up CTA more than there is: it runs out after limit_ns on each later
 * call; stall = 0 removes that. Host only; applies to launches enqueued after
 * the call (decode graphs keep the values they were captured with). */
moe_status_t moe_offload_debug_wait(moe_offload_t h, long long limit_ns, int stall);

/* ---- Decode trace (observability; no counterpart on the pages) ---------
 * With the trace on, decode-path launches enqueued afterwards (eager
 * moe_offload_decode_layer, and decode graphs created afterwards) stamp
 * %globaltimer (nanoseconds) into a per-layer record of MOE_TRACE_FIELDS
 * uint64 words: the earliest (fields marked min) or latest time a kernel of that
 * layer passed a point of the step. Layer records accumulate over calls until
 * read with reset, so read (and reset) after every step to see one call.
 * Field order (values of the TraceField enumeration of the kernels):
 *   0 head CTA 0 past its dependency wait      1 head logits complete
 *   2 head top-k and weights written           3 head slot table updated
 *   4 gate/up first CTA past its wait (min)    5 first W13 chunk of an installed expert used (min)
 *   6 last gate/up CTA of an installed expert  7 last W2-copy CTA done
 *   8 last gate/up CTA done                    9 down first CTA started (min)
 *  10 down last CTA past its waits             11 down last CTA done (counter resets included)
 *  12 down, latest CTA past writing its rows   13-15 unused.
 * Fields 4, 5 and 9 read ~0 and the others 0 when nothing stamped.
 * Only one-token calls (T = 1) are traced, through traced variants of the three
 * decode kernels (the plain ones carry no stamp code; the traced FFN variants
 * spill a few more registers, so a traced step is not the timed one). */
#define MOE_TRACE_FIELDS 16

/* on = 1: allocate the layer records (L * MOE_TRACE_FIELDS uint64 on the
 * device, once per handle), reset them and stamp from now on; on = 0: stop
 * (the records stay). Host only, no synchronisation beyond the reset.
 * Errors: MOE_ERR_INVALID, MOE_ERR_OOM, MOE_ERR_CUDA. */
moe_status_t moe_offload_trace_enable(moe_offload_t h, int on);

/* Copy the layer records into out[L * MOE_TRACE_FIELDS] (host), after
 * synchronising the device; reset = 1 then sets them back to their unset
 * values. MOE_ERR_INVALID when the trace was never enabled. */
moe_status_t moe_offload_trace_read(moe_offload_t h, uint64_t* out, int reset);

/* ---- Decode step as one CUDA graph -------------------------------------
 * A decode step of the whole stack (moe_offload_decode_layer for layers
 * 0..L-1 at batch T, layer l reading x + l*T*H and writing out + l*T*H) is
 * captured once into a CUDA graph and replayed per token with no host
 * synchronisation ("MoE expert offload" page, "How it works": fixed launch
 * shapes and device-resident miss counts keep decode inside CUDA graphs). */
typedef struct moe_offload_graph* moe_offload_graph_t;

/* Capture the step for batch T (1 <= T <= max_tokens_graph) over the fixed
 * device buffers x [L,T,H] bf16 (input) and out [L,T,H] bf16 (output), which
 * the caller owns and keeps alive. With timing != 0 the graph also records
 * CUDA events around each layer's route, ensure, miss copy and FFN launches
 * (read with moe_offload_graph_times). Capture runs on a private stream and
 * enqueues no work. The graph shares the handle's scratch: replays of two
 * graphs of one handle must not overlap on the GPU. */
moe_status_t moe_offload_graph_create(moe_offload_t h, int T, const void* x, void* out, int timing,
                                      moe_offload_graph_t* g);

/* Enqueue one replay of the step on `stream` (asynchronous, no host sync). */
moe_status_t moe_offload_graph_launch(moe_offload_graph_t g, moe_stream_t stream);

/* One step from host buffers: copy x_host [L,T,H] bf16 into the graph's input
 * buffer, replay, copy the output buffer to out_host [L,T,H] bf16, and wait
 * for that copy to finish. Host buffers should be pinned for full speed. */
moe_status_t moe_offload_graph_launch_host(moe_offload_graph_t g, const void* x_host, void* out_host,
                                           moe_stream_t stream);

/* Kernel times of the last launch of a timing graph, in milliseconds, one
 * entry per layer for each of the step's three launches (any array may be
 * NULL): head = router + top-k + slot ensure; gate_up = gate/up FFN, which also
 * copies the experts this call installed from host memory into their slots;
 * down = down projection + rank-order combine. Waits for that launch. */
moe_status_t moe_offload_graph_times(moe_offload_graph_t g, float* head_ms, float* gate_up_ms,
                                     float* down_ms);

/* Kernel launches one replay performs. */
int moe_offload_graph_kernel_count(moe_offload_graph_t g);

/* Free the graph (synchronises the device). NULL is ignored. */
void moe_offload_graph_destroy(moe_offload_graph_t g);

/* ---- Grouped FFN that allocates nothing ----------------------------------
 * The pages have no counterpart to this call; it exists for callers that
 * cannot call cudaMalloc: code running inside another runtime's memory arena
 * (a serving engine whose allocator owns all device memory and forbids side
 * allocations), plug-ins whose host process must account for every byte, and
 * paths that may not allocate after start-up. It computes what
 * moe_offload_grouped_ffn computes, with the same kernels, but takes the
 * expert tensors directly and keeps its intermediate rows in one fixed
 * library-owned device array instead of a handle's buffers.
 *
 *   w13: [E, 2I, H] bf16, w2: [E, H, I] bf16 — device memory (or host memory
 *        the GPU can read); ids [T, k] int32 index these arrays directly
 *   x: [T, H] bf16 device; w: [T, k] fp32 device; out: [T, H] bf16 device (output)
 *   status: optional device uint32 word; device-detected errors (an id outside
 *        [0, E)) are OR-ed into it (MOE_DEV_BAD_SLOT_ID); NULL = not reported
 * Limits: T*k <= 64 and T*k*I <= 1,048,576 (4 MiB of fp32 scratch);
 * H a multiple of 256 up to 8192, I a multiple of 64; weights, x and out
 * 16-byte aligned. Larger sizes return MOE_ERR_INVALID with the reason in
 * moe_offload_last_error(NULL); nothing is launched then.
 * It runs on the calling thread's current device and context. The scratch is
 * a file-scope __device__ array of about 4 MiB that every GPU loading the
 * library holds until the process exits. Each call looks up the array's
 * address in the current context (cudaGetSymbolAddress), so a context that was
 * reset or replaced gets the address that is valid in it. With lazy module
 * loading (the CUDA default) the first call in a context loads the library's
 * device code there and places the array: make that first call at start-up,
 * before any stream capture, so that later calls allocate nothing. No call
 * allocates: no cudaMalloc, no cudaFree, no allocating library routine. Every
 * call on a device shares the array and it keeps the last call's contents
 * (nothing read from it needs to start at zero: each call writes every
 * intermediate row it reads); calls that overlap on the GPU race on it. */
moe_status_t moe_offload_grouped_ffn_noalloc(const void* w13, const void* w2, int num_experts,
                                             int hidden, int inter, const void* x, const int32_t* ids,
                                             const float* w, int T, int top_k, void* out,
                                             uint32_t* status, moe_stream_t stream);

/* One-line reason of the last failed call on this handle ("" when none). With
 * h == NULL: the reason of the last failed call that takes no handle
 * (moe_offload_create, moe_offload_host_read_gbs, moe_offload_grouped_ffn_noalloc) on this thread. */
const char* moe_offload_last_error(moe_offload_t h);

/* Free everything the handle owns and unregister host memory it registered.
 * Synchronises the device. NULL is ignored. */
void moe_offload_destroy(moe_offload_t h);

#ifdef __cplusplus
}
#endif

#endif /* MOE_OFFLOAD_H */
