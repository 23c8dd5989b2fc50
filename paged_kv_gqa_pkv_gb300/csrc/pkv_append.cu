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

// The same append with the rotary embedding fused in front of the K write
// ("qwen3_flex_inference.py", _apply_rotary, applied to k right before the
// cache update): for each head, dims d and d + D/2 form a pair rotated by the
// angle of (position, d): out_d = k_d c - k_{d+D/2} s, out_{d+D/2} =
// k_{d+D/2} c + k_d s, computed in fp32 and rounded to bf16 (nearest even).
// A lane takes one 16-byte chunk of the first half of a head and its partner
// chunk of the second half; the tables' eight cos and sin values of that
// chunk are two float4 loads each. V rows are copied unchanged.
// With a k_norm weight, K is first normalised per head (the model's k_norm,
// applied to k just before _apply_rotary): x_d * w_d / sqrt(mean x^2 + eps).
// The 8 lanes of a head (an aligned group of 8) add their sums of squares
// with three shuffles, so the loop steps all lanes together.
// a*c - b*s and a*c + b*s accurate to about one fp32 ulp of the result even
// when the two products nearly cancel: the rounding error of b*s is kept
// exactly (an FMA) and folded back in after the fused multiply-add.
__device__ __forceinline__ float rot_diff(float a, float c, float b, float s) {
  const float p = b * s;
  const float e = fmaf(b, s, -p);
  return fmaf(a, c, -p) - e;
}
__device__ __forceinline__ float rot_sum(float a, float c, float b, float s) {
  const float p = b * s;
  const float e = fmaf(b, s, -p);
  return fmaf(a, c, p) + e;
}

__global__ void __launch_bounds__(kAppendWarps * 32)
append_rope_kernel(AppendRopeParams rp) {
  pdl_wait_primary();
  pdl_launch_dependents();
  const AppendParams& p = rp.a;
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  if (i >= p.n_tokens) return;

  const int b = p.batch_idx[i];
  const int pos = p.input_pos[i];
  if (b == 0) return;  // padding slot: no-op
  int err = 0;
  if (b < 0 || b >= p.max_batch) err |= PKV_DEV_ERR_BAD_SLOT;
  const int block = pos / p.page_size;
  if (pos < 0 || block >= p.max_blocks || pos >= rp.rope_len) err |= PKV_DEV_ERR_BAD_POS;
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
  const int vecs = p.row_vecs;
  const uint4* ks = reinterpret_cast<const uint4*>(p.k_new) + static_cast<int64_t>(i) * vecs;
  const uint4* vs = reinterpret_cast<const uint4*>(p.v_new) + static_cast<int64_t>(i) * vecs;
  uint4* kd = reinterpret_cast<uint4*>(p.k_pool) + row * vecs;
  uint4* vd = reinterpret_cast<uint4*>(p.v_pool) + row * vecs;
  for (int e = lane; e < vecs; e += 32) vd[e] = __ldg(vs + e);

  const float4* cs = reinterpret_cast<const float4*>(rp.rope_cos + static_cast<int64_t>(pos) * (kHeadDim / 2));
  const float4* sn = reinterpret_cast<const float4*>(rp.rope_sin + static_cast<int64_t>(pos) * (kHeadDim / 2));
  const int pairs = rp.num_kv_heads * 8;  // eight 16-byte chunk pairs per head
  const float* wn = rp.k_norm_weight;
  for (int e0 = 0; e0 < pairs; e0 += 32) {
    const int e = e0 + lane;
    const bool act = e < pairs;  // whole groups of 8: pairs is a multiple of 8
    const int h = e >> 3;
    const int c = e & 7;
    uint4 a = make_uint4(0u, 0u, 0u, 0u), bb = a;
    if (act) {
      a = __ldg(ks + h * 16 + c);
      bb = __ldg(ks + h * 16 + 8 + c);
    }
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
    float x1[8], x2[8];  // dims 8c..8c+7 and D/2 + 8c..
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      x1[2 * u] = bf16lo(aw[u]);
      x1[2 * u + 1] = bf16hi(aw[u]);
      x2[2 * u] = bf16lo(bw[u]);
      x2[2 * u + 1] = bf16hi(bw[u]);
    }
    if (wn != nullptr) {
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(x1[j], x1[j], fmaf(x2[j], x2[j], ss));
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      ss += __shfl_xor_sync(0xffffffffu, ss, 4);
      const float inv = rsqrtf(ss * (1.f / kHeadDim) + rp.k_norm_eps);
      if (act) {
        const float4* w1 = reinterpret_cast<const float4*>(wn + 8 * c);
        const float4* w2 = reinterpret_cast<const float4*>(wn + kHeadDim / 2 + 8 * c);
        const float4 wa = __ldg(w1), wb = __ldg(w1 + 1), wc = __ldg(w2), wd = __ldg(w2 + 1);
        const float wv1[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
        const float wv2[8] = {wc.x, wc.y, wc.z, wc.w, wd.x, wd.y, wd.z, wd.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          x1[j] = (x1[j] * inv) * wv1[j];
          x2[j] = (x2[j] * inv) * wv2[j];
        }
      }
    }
    if (!act) continue;
    const float4 c0 = __ldg(cs + 2 * c), c1 = __ldg(cs + 2 * c + 1);
    const float4 s0 = __ldg(sn + 2 * c), s1 = __ldg(sn + 2 * c + 1);
    const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    uint32_t o1[4], o2[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int l = 2 * u, hh = 2 * u + 1;
      o1[u] = pack_bf16x2(rot_diff(x1[l], cv[l], x2[l], sv[l]),
                          rot_diff(x1[hh], cv[hh], x2[hh], sv[hh]));
      o2[u] = pack_bf16x2(rot_sum(x2[l], cv[l], x1[l], sv[l]),
                          rot_sum(x2[hh], cv[hh], x1[hh], sv[hh]));
    }
    kd[h * 16 + c] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
    kd[h * 16 + 8 + c] = make_uint4(o2[0], o2[1], o2[2], o2[3]);
  }
}

cudaError_t launch_append_rope(const AppendRopeParams& p, cudaStream_t stream) {
  const int grid = (p.a.n_tokens + kAppendWarps - 1) / kAppendWarps;
  return launch_kernel(append_rope_kernel, dim3(grid), dim3(kAppendWarps * 32), 0, stream,
                       /*programmatic=*/true, p);
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const int grid = (p.n_tokens + kAppendWarps - 1) / kAppendWarps;
  return launch_kernel(append_kernel, dim3(grid), dim3(kAppendWarps * 32), 0, stream,
                       /*programmatic=*/true, p);
}

}  // namespace pkv
