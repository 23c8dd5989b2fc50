// pkv_mixed.cu - the routing kernel of pkv_mixed_attention.
//
// A step that interleaves prefill chunks with decode tokens ("flex_vs_vllm.md",
// "What's left on the table": prefill and decode in one pass) is served by
// two kernels in one call: the chunked prefill (pkv_prefill_paged.cu) for the
// runs of tokens of one slot, and the split-KV decode (pkv_decode.cu) for the
// tokens that are a run of one. Through the chunked prefill such a token
// costs a full 128-row tensor product per key tile of its prefix; the decode
// kernel streams its keys once. This kernel picks those tokens: token i is
// routed iff its slot is live (> 0) and differs from the slots of tokens i - 1
// and i + 1 of the packing. The first `cap` of them, in token order, are
// listed for the decode kernel and flagged for the prefill kernel to leave
// out; any beyond the cap stay with the prefill kernel.
// It also cuts the other tokens into the prefill kernel's query tiles: every
// run of equal slots (a run starts where the slot changes) is cut into pieces
// of at most 128 tokens, and a tile covers one piece. Fixed 128-token tiles
// of the packing would straddle runs (decode tokens between chunks shift
// every later chunk off the 128-token grid) and pay both runs' key ranges.
// One CTA walks the packing, 8 192 tokens a pass (eight consecutive tokens
// per thread, block-wide scans for the list positions and the run starts),
// so both lists are in token order, fixed by the input.
#include <climits>

#include "pkv.h"
#include "pkv_launch.h"

namespace pkv {
namespace {

constexpr int kRouteThreads = 1024;
constexpr int kPer = 8;  // consecutive tokens per thread

// Block-wide exclusive sum of `v` (and the block total) over kRouteThreads
// threads; `scratch` holds kRouteThreads / 32 ints. Contains __syncthreads.
__device__ __forceinline__ int block_excl_sum(int v, int* scratch, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = scratch[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    scratch[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  total = scratch[31];
  const int before = warp > 0 ? scratch[warp - 1] : 0;
  __syncthreads();  // scratch is reused by the caller's next scan
  return before + x - v;
}

// Block-wide exclusive maximum of `v` (identity -1) and the block maximum.
__device__ __forceinline__ int block_excl_max(int v, int* scratch, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = max(x, y);
  }
  const int up = __shfl_up_sync(0xffffffffu, x, 1);
  const int in_warp = lane > 0 ? up : -1;
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = scratch[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w = max(w, y);
    }
    scratch[lane] = w;
  }
  __syncthreads();
  total = scratch[31];
  const int before = warp > 0 ? scratch[warp - 1] : -1;
  __syncthreads();
  return max(before, in_warp);
}

// Each thread takes kPer consecutive tokens, so a pass over 8 192 tokens
// costs one round of loads and four block scans.
__global__ void __launch_bounds__(kRouteThreads) route_lone_kernel(
    const int32_t* __restrict__ batch_idx, int n_tokens, int cap, int32_t* __restrict__ list,
    int32_t* __restrict__ count, uint8_t* __restrict__ skip, int32_t* __restrict__ seg_start,
    int32_t* __restrict__ seg_count) {
  __shared__ int scratch[kRouteThreads / 32];
  int base = 0, seg_base = 0, run_carry = -1;  // identical in every thread
  for (int c0 = 0; c0 < n_tokens; c0 += kRouteThreads * kPer) {
    const int i0 = c0 + threadIdx.x * kPer;
    // slots of tokens i0 - 1 .. i0 + kPer; outside the packing they differ
    // from every slot (run starts and ends there)
    int b[kPer + 2];
#pragma unroll
    for (int k = 0; k < kPer + 2; ++k) {
      const int i = i0 - 1 + k;
      b[k] = (i >= 0 && i < n_tokens) ? __ldg(batch_idx + i) : (i < 0 ? INT_MIN : INT_MIN + 1);
    }
    uint32_t lone = 0, start = 0;
    int last_start = -1;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = i0 + k;
      if (i >= n_tokens) break;
      const bool st = b[k] != b[k + 1];
      if (st) {
        start |= 1u << k;
        last_start = i;
      }
      if (b[k + 1] > 0 && st && b[k + 2] != b[k + 1]) lone |= 1u << k;
    }
    int lone_total, max_total;
    const int lone_before = block_excl_sum(__popc(lone), scratch, lone_total);
    // the run in force at each token: the last run start at or before it,
    // earlier threads' and earlier passes' starts included
    const int prev = max(run_carry, block_excl_max(last_start, scratch, max_total));
    int rs_tok[kPer];
    {
      int cur = prev;
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        if ((start >> k) & 1u) cur = i0 + k;
        rs_tok[k] = cur;
      }
    }
    uint32_t seg = 0;
    int pos = base + lone_before;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = i0 + k;
      if (i >= n_tokens) break;
      bool routed = false;
      if ((lone >> k) & 1u) {
        routed = pos < cap;
        if (routed) list[pos] = i;
        ++pos;
      }
      skip[i] = routed ? 1 : 0;
      if (!routed && ((i - rs_tok[k]) & 127) == 0) seg |= 1u << k;
    }
    int seg_total;
    int spos = seg_base + block_excl_sum(__popc(seg), scratch, seg_total);
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if ((seg >> k) & 1u) seg_start[spos++] = i0 + k;
    base += lone_total;
    seg_base += seg_total;
    run_carry = max(run_carry, max_total);
  }
  if (threadIdx.x == 0) {
    *count = min(base, cap);
    *seg_count = seg_base;
  }
}

}  // namespace

cudaError_t launch_route_lone(const int32_t* batch_idx, int n_tokens, int cap, int32_t* list,
                              int32_t* count, uint8_t* skip, int32_t* seg_start,
                              int32_t* seg_count, cudaStream_t stream) {
  route_lone_kernel<<<1, kRouteThreads, 0, stream>>>(batch_idx, n_tokens, cap, list, count, skip,
                                                     seg_start, seg_count);
  return cudaGetLastError();
}

}  // namespace pkv
