// Grouped expert FFN that allocates nothing.
//
// Some callers cannot call cudaMalloc: code that runs inside another runtime's
// memory arena (an inference server that owns all device memory through its own
// allocator and forbids side allocations), plug-ins loaded into a process whose
// allocator must see every byte, or code paths that must not allocate after
// start-up. This entry point serves them: the caller passes inputs and outputs,
// and the FFN's intermediate rows (SiLU(g)*u of every token and rank) and its
// small count block live in one file-scope device array of fixed size that the
// library owns for the life of the process.
//
// The array is a module-scope __device__ variable: every GPU that loads the
// library holds it until the process exits. In host code its name is only a
// host-side stand-in, so each call looks the device address up with
// cudaGetSymbolAddress in the calling thread's current context and passes that
// address to the kernels. A symbol's address belongs to a context, not to a
// device: a runtime that calls this under its own context, or after a device
// reset, gets the address valid there (the lookup is cheap once the module is
// loaded in that context; with lazy loading the first call loads it and places
// the array, which is why callers make that first call at start-up). All calls
// on a device share the array, which keeps the last call's contents; calls that
// overlap on the GPU (two streams, or two threads without ordering) race on it.
#include <cuda_runtime.h>

#include <string>

#include "../../include/moe_offload.h"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kNoAllocMaxPairs = 64;                  // T * top_k
constexpr size_t kNoAllocFloats = (size_t)1 << 20;    // h rows: T*k*I floats (4 MiB)
// layout: [h floats | counts | status], each part 256-byte aligned. With no
// copy-through and no host sources (pair_src = nullptr) the FFN kernels never
// read the count area; it only gives counts/miss_expert a valid address. The
// status word collects device-detected errors when the caller passes none.
constexpr size_t kOffCounts = kNoAllocFloats * sizeof(float);
constexpr size_t kOffStatus = kOffCounts + 256;
constexpr size_t kNoAllocBytes = kOffStatus + 256;
static_assert(kNumCounts * sizeof(int32_t) <= 256, "count area");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

moe_status_t noalloc_fail(moe_status_t st, const std::string& msg) {
  set_handleless_error(msg.c_str());  // read back with moe_offload_last_error(NULL)
  return st;
}

// Device address of the scratch array in the current context.
cudaError_t scratch_in_current_context(unsigned char** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = static_cast<unsigned char*>(p);
  return cudaSuccess;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_offload_grouped_ffn_noalloc(const void* w13, const void* w2, int num_experts,
                                                        int hidden, int inter, const void* x,
                                                        const int32_t* ids, const float* w, int T,
                                                        int top_k, void* out, uint32_t* status,
                                                        moe_stream_t stream) {
  const int E = num_experts, H = hidden, I = inter, k = top_k;
  if (T == 0) return MOE_OK;
  if (!w13 || !w2 || !x || !ids || !w || !out)
    return noalloc_fail(MOE_ERR_INVALID, "grouped_ffn_noalloc: NULL pointer");
  if (!al16(w13) || !al16(w2) || !al16(x) || !al16(out))
    return noalloc_fail(MOE_ERR_INVALID, "grouped_ffn_noalloc: weights, x and out must be 16-byte aligned");
  if (E < 1 || k < 1 || k > 16 || k > E || H < 256 || H % 256 != 0 || H > 8192 || I < 64 || I % 64 != 0 ||
      T < 0)
    return noalloc_fail(MOE_ERR_INVALID, "grouped_ffn_noalloc: invalid shape (E=" + std::to_string(E) +
                                             " k=" + std::to_string(k) + " H=" + std::to_string(H) +
                                             " I=" + std::to_string(I) + " T=" + std::to_string(T) + ")");
  const size_t pairs = (size_t)T * k;
  if (pairs > (size_t)kNoAllocMaxPairs)
    return noalloc_fail(MOE_ERR_INVALID, "grouped_ffn_noalloc: T*top_k=" + std::to_string(pairs) +
                                             " exceeds the fixed maximum of " +
                                             std::to_string(kNoAllocMaxPairs));
  if (pairs * (size_t)I > kNoAllocFloats)
    return noalloc_fail(MOE_ERR_INVALID, "grouped_ffn_noalloc: T*top_k*I=" +
                                             std::to_string(pairs * (size_t)I) +
                                             " floats exceed the fixed scratch of " +
                                             std::to_string(kNoAllocFloats) + " floats (4 MiB)");
  unsigned char* base = nullptr;
  cudaError_t e = scratch_in_current_context(&base);
  if (e != cudaSuccess)
    return noalloc_fail(MOE_ERR_CUDA, std::string("grouped_ffn_noalloc: cudaGetSymbolAddress: ") +
                                          cudaGetErrorString(e));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  float* fl = reinterpret_cast<float*>(base);
  FfnArgs a{};
  a.lw.host_w13 = nullptr;
  a.lw.host_w2 = nullptr;
  a.lw.slot_w13 = const_cast<uint8_t*>(static_cast<const uint8_t*>(w13));
  a.lw.slot_w2 = const_cast<uint8_t*>(static_cast<const uint8_t*>(w2));
  a.x = static_cast<const uint16_t*>(x);
  a.slot_ids = ids;
  a.w = w;
  a.T = T;
  a.k = k;
  a.H = H;
  a.I = I;
  a.E = E;
  a.S = E;  // ids index the expert arrays directly
  a.counts = reinterpret_cast<const int32_t*>(base + kOffCounts);
  a.miss_expert = reinterpret_cast<const int32_t*>(base + kOffCounts);
  a.hbuf = fl;
  a.out = static_cast<uint16_t*>(out);
  a.status = status ? status : reinterpret_cast<uint32_t*>(base + kOffStatus);
  e = launch_grouped_ffn(a, st);
  if (e != cudaSuccess)
    return noalloc_fail(MOE_ERR_CUDA, std::string("grouped_ffn_noalloc: launch: ") + cudaGetErrorString(e));
  return MOE_OK;
}
