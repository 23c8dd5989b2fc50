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
// One CTA walks the packing in chunks of 1024 tokens, so both lists are in
// token order, fixed by the input.
#include "pkv.h"
#include "pkv_launch.h"

namespace pkv {
namespace {

constexpr int kRouteThreads = 1024;

__global__ void __launch_bounds__(kRouteThreads) route_lone_kernel(
    const int32_t* __restrict__ batch_idx, int n_tokens, int cap, int32_t* __restrict__ list,
    int32_t* __restrict__ count, uint8_t* __restrict__ skip, int32_t* __restrict__ seg_start,
    int32_t* __restrict__ seg_count) {
  __shared__ int s_warp[kRouteThreads / 32];
  __shared__ int s_wseg[kRouteThreads / 32];
  __shared__ int s_wmax[kRouteThreads / 32];
  __shared__ int s_base, s_segbase, s_runstart;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  constexpr int kWarps = kRouteThreads / 32;
  if (tid == 0) {
    s_base = 0;
    s_segbase = 0;
    s_runstart = 0;
  }
  __syncthreads();
  for (int c0 = 0; c0 < n_tokens; c0 += kRouteThreads) {
    const int i = c0 + tid;
    const bool valid = i < n_tokens;
    bool run_start = false, lone = false;
    if (valid) {
      const int b = batch_idx[i];
      run_start = i == 0 || batch_idx[i - 1] != b;
      const bool next_differs = i + 1 == n_tokens || batch_idx[i + 1] != b;
      lone = b > 0 && run_start && next_differs;
    }
    // routed tokens: position among the lone tokens so far
    const uint32_t bal = __ballot_sync(0xffffffffu, lone);
    // the latest run start at or before i (prefix max over token indices)
    int rs = run_start ? i : -1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, rs, o);
      if (lane >= o) rs = max(rs, v);
    }
    if (lane == 0) s_warp[warp] = __popc(bal);
    if (lane == 31) s_wmax[warp] = rs;
    __syncthreads();
    int pos = s_base + __popc(bal & ((1u << lane) - 1u));
    int rs_in = s_runstart;
    for (int w = 0; w < warp; ++w) {
      pos += s_warp[w];
      rs_in = max(rs_in, s_wmax[w]);
    }
    rs = max(rs, rs_in);
    const bool routed = lone && pos < cap;
    if (valid) skip[i] = routed ? 1 : 0;
    if (routed) list[pos] = i;
    // query tiles of the prefill kernel: run pieces of at most 128 tokens
    const bool seg = valid && !routed && ((i - rs) & 127) == 0;
    const uint32_t sbal = __ballot_sync(0xffffffffu, seg);
    if (lane == 0) s_wseg[warp] = __popc(sbal);
    __syncthreads();
    int spos = s_segbase + __popc(sbal & ((1u << lane) - 1u));
    for (int w = 0; w < warp; ++w) spos += s_wseg[w];
    if (seg) seg_start[spos] = i;
    __syncthreads();  // every thread has read the shared counters
    if (tid == 0) {
      int tot = 0, stot = 0, mx = s_runstart;
      for (int w = 0; w < kWarps; ++w) {
        tot += s_warp[w];
        stot += s_wseg[w];
        mx = max(mx, s_wmax[w]);
      }
      s_base += tot;
      s_segbase += stot;
      s_runstart = mx;
    }
    __syncthreads();
  }
  if (tid == 0) {
    *count = min(s_base, cap);
    *seg_count = s_segbase;
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
