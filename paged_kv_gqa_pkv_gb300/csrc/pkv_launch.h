// pkv_launch.h - parameter blocks and launch entry points of the libpkv
// kernels (internal; the public ABI is include/pkv.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "pkv_device.cuh"

namespace pkv {

struct AppendParams;
struct AppendRopeParams;

struct AppendParams {
  void* k_pool;
  void* v_pool;
  const int32_t* page_table;
  const void* k_new;
  const void* v_new;
  const int32_t* batch_idx;
  const int32_t* input_pos;
  int32_t* dev_err;
  int n_tokens;
  int row_vecs;     // 16-byte vectors per token row = H_kv * D * 2 / 16
  int page_size;
  int num_pages;
  int max_batch;
  int max_blocks;
};

// Append with the rotary embedding applied to K (tables fp32 [rope_len, D/2]).
struct AppendRopeParams {
  AppendParams a;
  const float* rope_cos;
  const float* rope_sin;
  int rope_len;
  int num_kv_heads;
  const float* k_norm_weight;  // [D] or null: no k_norm
  float k_norm_eps;
};

// Split-KV decode. The work of a call is the sequence of 16-token tiles of all
// (row, kv head) items, rows in order, kv heads within a row; it is cut into
// num_workers equal contiguous ranges, one per warp of a persistent grid.
struct DecodeParams {
  const void* q;              // bf16 [B, Hq, D]
  const int32_t* page_table;  // [max_batch, max_blocks]
  const int32_t* batch_idx;   // [B]
  const int32_t* seq_lens;    // [B]
  void* out;                  // bf16 [B, Hq, D]
  float* lse;                 // [B, Hq]
  float* partials;            // workspace: (num_workers + B*Hkv) slots
  // Fused append (all null for attention alone): the new token of row b,
  // k_new/v_new bf16 [B, Hkv, D], goes to position seq_lens[b] - 1 of its slot.
  const void* k_new;
  const void* v_new;
  void* k_pool;               // the pools as written (the tensor maps read them)
  void* v_pool;
  // Token list (all null for the usual rows): row r serves packed token
  // t = row_token[r] of a prefill-style call. Its slot is batch_idx[t], it
  // attends input_pos[t] + 1 keys, and q, out and lse are indexed by t. The
  // number of rows is min(*row_count, batch), read on the device.
  const int32_t* row_token;
  const int32_t* row_count;
  const int32_t* input_pos;
  int32_t* dev_err;
  int q_host;                 // q is mapped host memory: its rows arrive by cp.async
  int batch;
  int num_q_heads;
  int num_kv_heads;
  int page_size;
  int num_pages;
  int max_batch;
  int max_blocks;
  int num_workers;
  float qscale;               // scale * log2(e): scores kept in log2 units
};

constexpr int kDecodeTile = 16;       // tokens per pipeline stage
constexpr int kDecodeWarps = 8;       // workers (warps) per CTA
// Stages per worker. Sweeping warps x stages on the Qwen3-4B decode shape
// put the optimum at 8 x 2 (16 tiles, 128 KB in flight per SM): 8 x 3 was
// 6.6 % slower, 10 x 2 and 12 x 2 slower too, 6 x 2 and 8 x 1 slower. Past
// what covers the memory latency, more tiles in flight only add queueing.
constexpr int kDecodeStages = 2;
constexpr int kDecodeMaxBatch = 512;  // rows per call (row tables live in smem)

// Floats per partial slot: unnormalised o[G][D], then m[G], l[G] (padded).
__host__ __device__ constexpr int decode_slot_floats(int g) {
  return g * kHeadDim + ((2 * g + 3) / 4) * 4;
}

size_t decode_workspace_bytes(int batch, int num_kv_heads, int group, int num_workers);
int decode_workers_for_device(int sm_count);

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_append_rope(const AppendRopeParams& p, cudaStream_t stream);

// PKV_OK for cudaSuccess; otherwise remembers `e` for
// pkv_last_cuda_error_string() and returns PKV_ERR_CUDA.
pkv_status record_cuda_status(cudaError_t e);

// Validation and launch of pkv_prefill_attention (pkv_prefill.cu).
pkv_status prefill_entry(const void* q, const void* k, const void* v, int num_q_heads,
                         int num_kv_heads, int head_dim, const int32_t* batch_idx,
                         const int32_t* input_pos, int n_tokens, float scale, void* out,
                         float* lse, int32_t* dev_err, cudaStream_t stream);

// Validation and launch of pkv_prefill_paged_attention (pkv_prefill_paged.cu).
// skip (nullable, one byte per token): tokens with a nonzero byte are left
// out entirely (no keys, nothing written); another kernel serves them.
// seg_start/seg_count (nullable, device): query tiles start at these tokens
// and cover the run of equal slots from there (at most 128 tokens) instead of
// fixed 128-token windows of the packing.
pkv_status prefill_paged_entry(const pkv_cache_desc* cache, const void* k_pool,
                               const void* v_pool, const int32_t* page_table, const void* q,
                               int num_q_heads, const int32_t* batch_idx,
                               const int32_t* input_pos, int n_tokens, float scale, void* out,
                               float* lse, int32_t* dev_err, cudaStream_t stream,
                               const uint8_t* skip = nullptr, const int32_t* seg_start = nullptr,
                               const int32_t* seg_count = nullptr);
cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          int sm_count, cudaStream_t stream);

// pkv_mixed.cu: lists the first `cap` tokens that are a run of one in the
// packing (ascending) in list[0, *count) and sets skip[i] = 1 for each of them
// (0 for every other token); lists the first tokens of the prefill kernel's
// query tiles (pieces of at most 128 tokens of each run of equal slots, the
// listed tokens left out) in seg_start[0, *seg_count).
cudaError_t launch_route_lone(const int32_t* batch_idx, int n_tokens, int cap, int32_t* list,
                              int32_t* count, uint8_t* skip, int32_t* seg_start,
                              int32_t* seg_count, cudaStream_t stream);

// cudaLaunchKernelEx with an optional programmatic-stream-serialisation
// attribute (programmatic dependent launch).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool programmatic, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace pkv
