// pkv_prefill_common.cuh - what the two tcgen05 prefill kernels share: tile
// sizes, the shared-memory layout, the MMA instruction descriptors, the
// bounded wait that honours a grid-wide abort flag, and the host-side
// cuTensorMapEncodeTiled lookup.
#pragma once

#include "pkv_launch.h"

namespace pkv {
namespace prefill_detail {

constexpr int kBM = 128;                 // query rows per tile
constexpr int kBN = 128;                 // keys per KV tile
constexpr int kHalf = 128 * 128;         // one [128 rows x 64 elems] bf16 block, bytes
constexpr int kTileBytes = 2 * kHalf;    // 128 x 128 bf16 (32 KB)
constexpr int kRing = 3;                 // K/V half-stage slots
constexpr int kThreads = 10 * 32;
constexpr int kGroupThreads = 128;       // one softmax warpgroup
constexpr uint32_t kTmemCols = 512;      // S0 S1 O0 O1, 128 columns each
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// shared memory layout (offsets from a 1024-aligned base)
constexpr int kOffQ = 0;                              // Q0, Q1
constexpr int kOffP = kOffQ + 2 * kTileBytes;         // P0, P1
constexpr int kOffRing = kOffP + 2 * kTileBytes;      // 3 slots
constexpr int kOffBar = kOffRing + kRing * kTileBytes;
// q_full, q_empty, ring_full[3], ring_empty[3], s_full[2], p_full[2],
// pv_done[2], o_free[2], s_free[2], grp_sync[2]
constexpr int kNumBars = 20;
constexpr int kOffMisc = kOffBar + kNumBars * 8;      // tmem slot, abort flag
constexpr int kSmemBytes = kOffMisc + 16 + 1024;      // + slack for 1024 alignment

constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, /*b_mn_major=*/false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kHeadDim, /*b_mn_major=*/true);

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

}  // namespace prefill_detail

namespace prefill_host {

inline bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// {D, heads, tokens} view; box = 64 head dims x 1 head x 128 tokens, 128-byte
// swizzled (the tcgen05 operand layout).
inline bool encode_packed_map(CUtensorMap* map, const void* base, int heads, int n_tokens) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(n_tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                                 static_cast<cuuint64_t>(heads) * kHeadDim * 2};
  const cuuint32_t box[3] = {64u, 1u, 128u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace prefill_host
}  // namespace pkv
