// Prefill grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// The (token, rank) pairs of a prefill call are bucketed by expert; the x rows
// of the pairs are gathered in bucket order into Xp [Tk, H]. One CTA computes a
// 128-row tile of one bucket against one column block of that bucket's expert:
//   gate/up:  Xp[128 x H] . [W1 rows n..n+128 ; W3 rows n..n+128]^T -> TMEM
//             [128 x 256] fp32, epilogue h = silu(g) * u -> Hp (bf16, bucket order)
//   down:     Hp[128 x I] . W2[rows n..n+256]^T -> TMEM [128 x 256] fp32,
//             epilogue writes y of each pair (fp32) for the rank-order combine
// ("MoE expert offload" page, "How it works", Prefill: the unmodified GEMM runs
// on the staged [E, N, K] layer, or on the slot tensors.) Rows of a tile past
// the end of its bucket are computed and discarded; every output row depends
// only on its own input row, so the bucket order never changes a result.
//
// Two CTAs per SM (256 TMEM columns and a 96 KB ring each), so that one CTA's
// epilogue, which leaves the tensor core and the copies idle, overlaps the other
// CTA's main loop. The ring holds two stages of K = 64 (128-byte swizzle): at
// prefill sizes of the Qwen3-30B-A3B shape (about 128 rows per expert) the kernels
// are bound by the bytes they stream and the stage size does not matter; at the
// Mixtral-8x7B shape (I = 14336, tensor-bound) the larger stages halve the
// per-stage barrier and commit work of the MMA thread.
//
// Early down: the down launch follows the gate/up launch under programmatic
// dependent launch. Each gate/up CTA triggers it at its start and, once its h
// rows are written, counts itself into its tile's counter; a down CTA issues the
// weight (W2) loads of its first stages at once and the h-tile loads only when
// its tile's count is complete (a bounded wait), so down CTAs take the SMs that
// the gate/up launch's last, partial wave leaves idle. The down grid starts only
// after every gate/up CTA has started, so a waiting down CTA never keeps a
// producer off the GPU.
//
// Warp roles (8 warps): warp 0 allocates TMEM and, one lane, issues the TMA
// loads of a 2-stage shared-memory ring (K = 64 each); warp 1, one lane, issues
// tcgen05.mma (M=128, N=256, K=16, bf16 in, fp32 accumulate) and commits each
// stage back to the producer; all 8 warps read the accumulator with tcgen05.ld
// for the epilogue (warp w reads TMEM lanes 32(w%4)..32(w%4)+31 = tile rows and
// the w/4-th half of the columns) and move their rows through a transpose tile
// in the idle ring, so that stores write whole row segments. Every wait is bounded:
// a wait that runs out sets a status bit and the CTA drains its own copies
// (again bounded), frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "kernels.h"
#include "prefill_tc.h"

namespace moe {
namespace {

constexpr int BM = 128;        // tile rows (pairs)
constexpr int BN = 256;        // accumulator columns
constexpr int BK = 64;         // K per stage: one 128-byte swizzle row of bf16
constexpr int A_BYTES = BM * BK * 2;     // 8 KB
constexpr int B_BYTES = BN * BK * 2;     // 16 KB
constexpr int kStages = 2;
constexpr int kStageBytes = A_BYTES + B_BYTES;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 256;  // ring, 1 KB alignment slack, barriers
constexpr uint32_t kTmemCols = BN;
constexpr int kGemmThreads = 256;                // 8 warps
constexpr int kColParts = kGemmThreads / 128;    // epilogue warps per TMEM lane quadrant
constexpr int kCtasPerSm = 2;
static_assert(kCtasPerSm * (kSmemBytes + 1024) <= 228 * 1024 && kCtasPerSm * kTmemCols <= 512, "two CTAs per SM");
constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

__device__ __forceinline__ void tma_load_2d(const CUtensorMap* tm, uint64_t* bar, void* dst, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(smem_u32(dst)), "l"(tm), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart (the layout a SWIZZLE_128B TMA box of 64 bf16 columns writes).
// The k-th K=16 step of a stage starts 32 bytes further into the swizzled rows.
__device__ __forceinline__ uint64_t sdesc(const void* p) {
  const uint64_t a = smem_u32(p);
  uint64_t d = (a >> 4) & 0x3FFFull;        // start address
  d |= 1ull << 16;                          // leading byte offset (unused with this swizzle)
  d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: 8 rows x 128 B
  d |= 1ull << 46;                          // descriptor version
  d |= 2ull << 61;                          // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(tmem_d), "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Epilogue transpose tile: 32 rows of up to 32 words per warp, row stride 33 words
// (writes by row and reads by column are both free of bank conflicts).
constexpr int kTileStride = 33;
static_assert(kGemmThreads / 32 * 32 * kTileStride * 4 <= kStages * kStageBytes, "epilogue tiles fit the ring");

// Stores a warp's transpose tile (32 rows x W words, W = 16 or 32) row segment by row
// segment: W/4 lanes per row, 16 bytes each, 128/W rows per instruction. dst(rr) gives
// the first word of row rr's segment in global memory, or nullptr for a row past the tile.
// Every lane calls dst for every iteration (it may hold a warp shuffle).
template <int W, typename Dst>
__device__ __forceinline__ void store_rows(const uint32_t* tile, int lane, Dst dst) {
  constexpr int kLanesPerRow = W / 4, kRowsPerStep = 32 / kLanesPerRow;
#pragma unroll
  for (int it = 0; it < 32 / kRowsPerStep; ++it) {
    const int rr = it * kRowsPerStep + lane / kLanesPerRow;
    const int w0 = (lane % kLanesPerRow) * 4;
    const uint32_t* src = tile + rr * kTileStride + w0;
    const uint4 v = make_uint4(src[0], src[1], src[2], src[3]);
    uint32_t* d = dst(rr);
    if (d) *reinterpret_cast<uint4*>(d + w0) = v;
  }
}

// The CTA's work: bucket g, row tile (global index), column block, first row in bucket
// order and valid rows. CTAs run in launch order (linear id L), and bucket g owns the
// cb x R_g consecutive ids from cb * tiles[g]; within them the R_g row tiles of one
// column block are adjacent, so the CTAs that stream the same weight block run
// together (it is read from DRAM once however many rows the bucket has), and a row
// tile's x (or h) tile is read by CTAs at most R_g ids apart, also running together.
__device__ bool cta_work(const int32_t* counts, const int32_t* offsets, const int32_t* tiles, int G, int cb,
                         int* g_out, int* tile, int* col, int* row0, int* rows) {
  const int L = blockIdx.x + gridDim.x * blockIdx.y;
  const int t = L / cb;  // cb * tiles[g] <= L exactly when tiles[g] <= t
  if (t >= tiles[G]) return false;
  int lo = 0, hi = G - 1;
  while (lo < hi) {  // largest g with tiles[g] <= t (never an empty bucket: it shares the next one's offset)
    const int mid = (lo + hi + 1) >> 1;
    if (tiles[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  const int R = tiles[lo + 1] - tiles[lo];
  const int j = L - cb * tiles[lo];
  const int c = j / R, r = j - c * R;
  const int m0 = r * BM;
  *g_out = lo;
  *tile = tiles[lo] + r;
  *col = c;
  *row0 = offsets[lo] + m0;
  *rows = min(BM, counts[lo] - m0);
  return *rows > 0;
}

// MODE 1: gate/up + SiLU epilogue into Hp; column block j: gate rows j*128.. and the
// matching up rows I + j*128.. in one accumulator (h columns j*128..). MODE 2: down
// projection into Y by pair, output columns j*256...
template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, kCtasPerSm)
tc_grouped_gemm(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, TcGemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* done = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  __shared__ int s_fail;
  __shared__ int s_stale;  // early down: the tile's h rows did not arrive in time (no output written)

  if (MODE == 1) pdl_trigger();  // the down launch may start once every gate/up CTA has started
  int g, tile, col, row0, rows;
  if (!cta_work(p.counts, p.offsets, p.tiles, p.G, p.cb, &g, &tile, &col, &row0, &rows)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = p.K / BK;

  if (threadIdx.x == 0) {
    s_fail = 0;
    s_stale = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int issued = 0;  // stages the producer loaded (for the drain on failure)
  if (warp == 0 && lane == 0) {
    // TMA producer. Stage kb: the A tile (x or h rows) and the weight tile.
    const CUtensorMap* tmb = &tm_b;
    auto load_b = [&](int kb, uint8_t* a_dst, uint64_t* bar) {
      uint8_t* b_dst = a_dst + A_BYTES;
      if (MODE == 1) {
        const int gate_row = g * 2 * p.I + col * (BN / 2);
        tma_load_2d(tmb, bar, b_dst, kb * BK, gate_row);
        tma_load_2d(tmb, bar, b_dst + B_BYTES / 2, kb * BK, gate_row + p.I);
      } else {
        tma_load_2d(tmb, bar, b_dst, kb * BK, g * p.H + col * BN);
      }
    };
    // Early down: the weight tiles of the first stages do not depend on the gate/up
    // launch and go out at once; the h tiles follow once the tile's count is complete.
    const int pre = (MODE == 2 && p.tile_done) ? min(nk, kStages) : 0;
    for (int kb = 0; kb < pre; ++kb) {
      mbar_expect_tx(&full[kb], kStageBytes);
      load_b(kb, smem + kb * kStageBytes, &full[kb]);
    }
    if (pre) {
      // On a timeout (status bit set) every stage is still loaded and consumed, so no
      // copy is left in flight, and the epilogue writes nothing.
      if (!wait_at_least(p.tile_done + tile, p.tile_need, p.status, p.wait_ns ? p.wait_ns : kDefaultWaitNs))
        s_stale = 1;
      asm volatile("fence.proxy.async.global;" ::: "memory");  // h rows were written by generic stores
    }
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kStages;
      if (kb >= kStages && !mbar_wait(&empty[s], ((kb / kStages) - 1) & 1)) {
        atomicOr(p.status, kDevTimeout);
        s_fail = 1;
        break;
      }
      uint8_t* a_dst = smem + s * kStageBytes;
      if (kb >= pre) {
        mbar_expect_tx(&full[s], kStageBytes);
        load_b(kb, a_dst, &full[s]);
      }
      tma_load_2d(&tm_a, &full[s], a_dst, kb * BK, row0);
      issued = kb + 1;
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    constexpr uint32_t idesc = idesc_bf16(BM, BN);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kStages;
      if (!mbar_wait(&full[s], (kb / kStages) & 1)) {
        atomicOr(p.status, kDevTimeout);
        s_fail = 1;
        break;
      }
      tc_fence_after();
      const uint8_t* a = smem + s * kStageBytes;
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk)
        mma_bf16(tmem, sdesc(a + kk * 32), sdesc(a + A_BYTES + kk * 32), idesc, (kb > 0 || kk > 0) ? 1u : 0u);
      mma_commit(&empty[s]);
    }
    mma_commit(done);
  }
  __syncwarp();
  const bool ok = mbar_wait(done, 0);
  if (!ok && threadIdx.x == 0) {
    atomicOr(p.status, kDevTimeout);
    s_fail = 1;
  }
  tc_fence_after();
  __syncthreads();
  if (!s_fail && !s_stale) {
    // Epilogue. Each warp moves its 32 rows through a transpose tile in shared memory
    // (the idle ring: every load it received was consumed by the MMAs), so that each
    // store instruction writes four row segments of 128 bytes instead of 32 segments
    // of 16 bytes.
    const int quad = warp & 3, part = warp >> 2;  // TMEM lane quadrant, half of the columns
    const int r = quad * 32 + lane;                // tile row = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    uint32_t* tile = reinterpret_cast<uint32_t*>(smem) + warp * (32 * kTileStride);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (MODE == 1) {
      constexpr int kPart = BN / 2 / kColParts;  // this warp's h columns (gate in 0..127, up in 128..255)
      static_assert(kPart == 64, "epilogue column split");
      const int col0 = col * (BN / 2) + part * kPart;
#pragma unroll 1
      for (int c = 0; c < kPart; c += 32) {
        uint32_t gv[32], uv[32];
        tmem_ld32(lane_base + part * kPart + c, gv);
        tmem_ld32(lane_base + BN / 2 + part * kPart + c, uv);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          float h2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float gs = __uint_as_float(gv[2 * q + e]), us = __uint_as_float(uv[2 * q + e]);
            h2[e] = __fdividef(gs, 1.0f + __expf(-gs)) * us;  // silu(g) * u; h is rounded to bf16 next
          }
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(h2[0], h2[1]);
          tile[lane * kTileStride + c / 2 + q] = *reinterpret_cast<const uint32_t*>(&b2);
        }
      }
      __syncwarp();
      store_rows<kPart / 2>(tile, lane, [&](int rr) -> uint32_t* {
        const int row = quad * 32 + rr;
        return row < rows ? reinterpret_cast<uint32_t*>(p.hp + (size_t)(row0 + row) * p.I + col0) : nullptr;
      });
    } else {
      const int col0 = col * BN;
      const int pair = r < rows ? p.perm[row0 + r] : 0;
      constexpr int kPart = BN / kColParts;
      static_assert(kPart % 32 == 0, "epilogue column split");
#pragma unroll 1
      for (int c = part * kPart; c < (part + 1) * kPart; c += 32) {
        uint32_t v[32];
        tmem_ld32(lane_base + c, v);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 32; ++q) tile[lane * kTileStride + q] = v[q];
        __syncwarp();
        store_rows<32>(tile, lane, [&](int rr) -> uint32_t* {
          const int pr = __shfl_sync(0xffffffffu, pair, rr);
          return quad * 32 + rr < rows ? reinterpret_cast<uint32_t*>(p.y + (size_t)pr * p.H + col0 + c) : nullptr;
        });
        __syncwarp();
      }
    }
  } else if (s_fail && warp == 0 && lane == 0) {
    // Drain: wait (bounded) for every load this CTA issued before its memory goes away.
    for (int kb = 0; kb < issued; ++kb) mbar_wait(&full[kb % kStages], (kb / kStages) & 1);
  }
  if (MODE == 1 && p.tile_done) asm volatile("fence.proxy.async.global;" ::: "memory");  // h rows: read by TMA
  tc_fence_before();
  __syncthreads();
  if (MODE == 1 && p.tile_done && threadIdx.x == 0) {  // early down: this CTA's h rows are written
    __threadfence();
    atomicAdd(p.tile_done + tile, 1u);
  }
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

__global__ void gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm, int Tk, int k,
                                   int Tr, int H, uint16_t* __restrict__ xp) {
  const int h8 = H / 8;
  const size_t total = (size_t)Tk * h8;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int pos = (int)(i / h8), c = (int)(i - (size_t)pos * h8);
    const int pair = perm[pos];
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (pair >= 0 && pair < Tk)
      v = reinterpret_cast<const uint4*>(x + (size_t)(pair < Tr ? pair / k : pair - Tr) * H)[c];
    reinterpret_cast<uint4*>(xp + (size_t)pos * H)[c] = v;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t encoder() {
  if (g_encode) return cudaSuccess;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess) return e;
  if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return cudaSuccess;
}

// 2-D bf16 tensor map [rows, cols] (cols contiguous), box rows x 64 columns, 128-byte swizzle.
cudaError_t make_map(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

bool tc_gemm_supported(int H, int I) { return H % BN == 0 && I % (BN / 2) == 0 && I % BK == 0 && H % BK == 0; }

int tc_gemm_tile_rows() { return BM; }

cudaError_t tc_gemm_init_attributes() {
  cudaError_t e = cudaFuncSetAttribute(tc_grouped_gemm<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_grouped_gemm<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  return e;
}

cudaError_t launch_tc_prefill(const TcPrefillArgs& a, cudaStream_t st) {
  cudaError_t e = encoder();
  if (e != cudaSuccess) return e;
  const int Tk = a.Tk;
  gather_rows_kernel<<<1024, 256, 0, st>>>(a.x, a.perm, Tk, a.k, a.Tr, a.H, a.xp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  CUtensorMap ta1, tb1, ta2, tb2;
  if ((e = make_map(&ta1, a.xp, (uint64_t)Tk, (uint64_t)a.H, BM)) != cudaSuccess) return e;
  // gate/up weight boxes: 128 gate rows and the matching 128 up rows
  if ((e = make_map(&tb1, a.w13, (uint64_t)a.G * 2 * a.I, (uint64_t)a.H, BN / 2)) != cudaSuccess) return e;
  if ((e = make_map(&ta2, a.hp, (uint64_t)Tk, (uint64_t)a.I, BM)) != cudaSuccess) return e;
  if ((e = make_map(&tb2, a.w2, (uint64_t)a.G * a.H, (uint64_t)a.I, BN)) != cudaSuccess) return e;
  TcGemmArgs p{};
  p.counts = a.counts;
  p.offsets = a.offsets;
  p.tiles = a.tiles;
  p.G = a.G;
  p.I = a.I;
  p.H = a.H;
  p.perm = a.perm;
  p.hp = a.hp;
  p.y = a.y;
  p.status = a.status;
  const int max_tiles = (Tk + BM - 1) / BM + a.G;
  const int cb1 = a.I / (BN / 2), cb2 = a.H / BN;  // column blocks of the two GEMMs
  p.tile_done = a.tile_done;
  p.tile_need = (uint32_t)cb1 + (a.stall ? 1u : 0u);  // (stall: a target no tile reaches, so the wait runs out)
  p.wait_ns = a.wait_ns;
  if (a.tile_done &&
      (e = cudaMemsetAsync(a.tile_done, 0, sizeof(uint32_t) * (size_t)max_tiles, st)) != cudaSuccess)
    return e;
  p.K = a.H;
  p.cb = cb1;
  if (a.ev_gemm_begin && (e = cudaEventRecord(a.ev_gemm_begin, st)) != cudaSuccess) return e;
  tc_grouped_gemm<1><<<dim3(cb1, max_tiles), kGemmThreads, kSmemBytes, st>>>(ta1, tb1, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  p.K = a.I;
  p.cb = cb2;
  if ((e = launch_k(tc_grouped_gemm<2>, dim3(cb2, max_tiles), dim3(kGemmThreads), kSmemBytes, st,
                    a.tile_done != nullptr, ta2, tb2, p)) != cudaSuccess)
    return e;
  return a.ev_gemm_end ? cudaEventRecord(a.ev_gemm_end, st) : cudaSuccess;
}

}  // namespace moe
