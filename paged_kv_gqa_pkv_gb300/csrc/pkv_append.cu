// pkv_append.cu - K1: KV append through the page table.
//
// Source: "qwen3_flex_inference.py", attention forward ("Write to paged KV
// cache") and capture_decode_cudagraph (the k_cache[addr] = k_val write, which
// crashed with an illegal address through an unreserved entry;
// "flex_paged_attention.py" commit log, "Files").
//
// In the token-major pool [P*ps, H_kv, D] one token's K (or V) row for all kv
// heads is H_kv*D*2 contiguous bytes (2 KB for 8 heads), and so is its source
// row in k_new [N, H_kv, D]. One warp moves one token: 16-byte vector loads
// and stores, fully coalesced, a bit-exact byte copy. Every index is checked
// before the store; a bad one skips the token and sets a dev_err bit.
#include "pkv_launch.h"

namespace pkv {

constexpr int kAppendWarps = 8;

__global__ void __launch_bounds__(kAppendWarps * 32)
append_kernel(AppendParams p) {
  // Launched as a programmatic dependent: wait for the previous kernel (it may
  // still read the pools), then let the next launch start its prologue.
  pdl_wait_primary();
  pdl_launch_dependents();

  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  if (i >= p.n_tokens) return;

  const int b = p.batch_idx[i];
  const int pos = p.input_pos[i];
  if (b == 0) return;  // padding slot: no-op
  int err = 0;
  if (b < 0 || b >= p.max_batch) err |= PKV_DEV_ERR_BAD_SLOT;
  const int block = pos / p.page_size;
  if (pos < 0 || block >= p.max_blocks) err |= PKV_DEV_ERR_BAD_POS;
  int page = -1;
  if (!err) {
    page = p.page_table[static_cast<int64_t>(b) * p.max_blocks + block];
    if (page < 0 || page >= p.num_pages) err |= PKV_DEV_ERR_BAD_PAGE;
  }
  if (err) {
    if (lane == 0) set_dev_err(p.dev_err, err);
    return;
  }
  const int64_t row = static_cast<int64_t>(page) * p.page_size + pos % p.page_size;
  const int vecs = p.row_vecs;  // 16-byte vectors per token row (H_kv * D * 2 / 16)
  const uint4* ks = reinterpret_cast<const uint4*>(p.k_new) + static_cast<int64_t>(i) * vecs;
  const uint4* vs = reinterpret_cast<const uint4*>(p.v_new) + static_cast<int64_t>(i) * vecs;
  uint4* kd = reinterpret_cast<uint4*>(p.k_pool) + row * vecs;
  uint4* vd = reinterpret_cast<uint4*>(p.v_pool) + row * vecs;
  for (int e = lane; e < vecs; e += 32) {
    const uint4 kv = __ldg(ks + e);
    const uint4 vv = __ldg(vs + e);
    kd[e] = kv;
    vd[e] = vv;
  }
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const int grid = (p.n_tokens + kAppendWarps - 1) / kAppendWarps;
  return launch_kernel(append_kernel, dim3(grid), dim3(kAppendWarps * 32), 0, stream,
                       /*programmatic=*/true, p);
}

}  // namespace pkv
