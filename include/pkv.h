/*
 * pkv.h - C ABI of libpkv: attention over a paged KV cache on GB300 (sm_103a).
 *
 * The KV cache of one attention layer is one contiguous physical pool per
 * tensor, K and V, each bf16 [num_pages * page_size, H_kv, D] (token-major,
 * row-major, contiguous). A page table, int32 [max_batch, max_blocks]
 * row-major, maps (batch slot, logical block) to a physical page. Batch slot 0
 * and page 0 are reserved as no-op padding; an entry of -1 means "no page
 * reserved". Source: "flex_paged_attention.py" commit log, section "Why this
 * works", items 1 and 3.
 *
 * Three stream-ordered calls replace the pages' PagedKVCache.update followed
 * by flex_attention(q, k, v, scale, block_mask, enable_gqa=True)
 * ("qwen3_flex_inference.py", attention forward, _decode_step_eager,
 * _prefill):
 *   pkv_append            - write new tokens' K/V rows through the page table
 *   pkv_append_rope       - the same with k_norm and the rotary embedding
 *                           applied to K
 *   pkv_prefill_paged_attention - chunked prefill / mixed prefill + decode
 *                           tokens attending their slots' keys through pages
 *   pkv_decode_attention  - one query token per row, GQA, over the pages
 *   pkv_prefill_attention - packed document-causal attention over fresh k/v
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller. The library
 *    keeps no pointer after the call returns and allocates no device memory;
 *    scratch space, where needed, is a caller-provided workspace.
 *  - Arguments are validated on the host, synchronously, before anything is
 *    launched; a failed check returns its status and launches nothing.
 *  - Problems only visible on the device (a page entry outside [0, num_pages),
 *    a slot outside [0, max_batch), a position past the table) never trap:
 *    the affected work is skipped and a PKV_DEV_ERR_* bit is OR-ed into the
 *    optional int32 word dev_err (device memory, may be NULL). The caller
 *    reads it after synchronising the stream. Results of affected rows are
 *    unspecified; everything else is still computed.
 *  - Calls only enqueue work on `stream` (NULL = the legacy default stream),
 *    never synchronise it, and keep no state between calls, so they may be
 *    captured into a CUDA graph.
 *  - head_dim must be 128; num_q_heads / num_kv_heads (the GQA group) must be
 *    1, 2, 4 or 8; page_size must be a positive multiple of 16; bf16 tensors
 *    must be 16-byte aligned; int32/fp32 arrays 4-byte aligned.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_ARG = 1,        /* bad size, null pointer or unsupported shape   */
  PKV_ERR_ALIGN = 2,      /* a pointer misses its required alignment       */
  PKV_ERR_BAD_PAGE = 3,   /* pkv_status_from_device_error: bad page entry  */
  PKV_ERR_WORKSPACE = 4,  /* workspace missing or smaller than required    */
  PKV_ERR_CUDA = 5,       /* a CUDA runtime call failed (launch, query)    */
  PKV_ERR_DEVICE = 6,     /* current device is not a supported sm_103 GPU  */
  PKV_ERR_BAD_INPUT = 7   /* pkv_status_from_device_error: other device err */
} pkv_status;

/* Bits OR-ed into *dev_err by the kernels. */
#define PKV_DEV_ERR_BAD_PAGE   0x1  /* page entry not in [0, num_pages)          */
#define PKV_DEV_ERR_BAD_SLOT   0x2  /* batch_idx not in [0, max_batch)           */
#define PKV_DEV_ERR_BAD_POS    0x4  /* position/seq_len < 0 or past max_blocks   */
#define PKV_DEV_ERR_LAYOUT     0x8  /* prefill packing precondition violated     */
#define PKV_DEV_ERR_TIMEOUT    0x10 /* a bounded wait inside a kernel gave up    */

/* Geometry of one layer's paged cache. */
typedef struct {
  int num_pages;     /* P: physical pages per pool (page 0 reserved)          */
  int page_size;     /* ps: token slots per page, multiple of 16               */
  int num_kv_heads;  /* H_kv                                                   */
  int head_dim;      /* D, must be 128                                         */
  int max_batch;     /* rows of page_table (slot 0 reserved)                   */
  int max_blocks;    /* columns of page_table: logical blocks per sequence     */
} pkv_cache_desc;

/*
 * pkv_append - KV append through the page table.
 * Source: "qwen3_flex_inference.py", attention forward ("Write to paged KV
 * cache"), capture_decode_cudagraph (the k_cache[addr] = k_val write); the
 * crash on an unreserved entry: "flex_paged_attention.py" commit log, "Files".
 *
 * For each token i in [0, n_tokens) with slot b = batch_idx[i] and position
 * p = input_pos[i], copies the bytes of k_new[i] and v_new[i] (each bf16
 * [H_kv, D], contiguous rows of a [n_tokens, H_kv, D] tensor) to pool row
 *     page_table[b, p / ps] * ps + p % ps
 * of k_pool and v_pool. Bit-exact byte copy. Tokens with b == 0 (padding
 * slot) are skipped without error. A token whose slot, block or page entry is
 * out of range is skipped and sets PKV_DEV_ERR_BAD_SLOT / _BAD_POS / _BAD_PAGE.
 * Two tokens that address the same row race (the last writer is unspecified).
 * Decode passes n_tokens = B (one new token per row), prefill passes the
 * packed tokens.
 */
pkv_status pkv_append(const pkv_cache_desc* cache, void* k_pool, void* v_pool,
                      const int32_t* page_table, const void* k_new,
                      const void* v_new, const int32_t* batch_idx,
                      const int32_t* input_pos, int n_tokens, int32_t* dev_err,
                      cudaStream_t stream);

/*
 * pkv_append_rope - pkv_append with the model's per-head k_norm (optional)
 * and the rotary position embedding applied to each new K row on the way
 * into the pool (V rows are copied unchanged).
 * Source: "qwen3_flex_inference.py", attention forward (k = k_norm(k_proj(..)
 * per head), then _apply_rotary: x * cos + rotate_half(x) * sin with
 * rotate_half(x) = cat(-x2, x1), right before the cache write).
 *
 * rope_cos, rope_sin: fp32 [rope_len, D/2] row-major, 16-byte aligned; row p
 * holds the cos/sin of the angles of position p (the full-width tables repeat
 * them for the second half of D). For each kv head of token i at position
 * p = input_pos[i], with x1 = k_new[i][h][0:D/2], x2 = k_new[i][h][D/2:D],
 * c = rope_cos[p], s = rope_sin[p]:
 *     K row = bf16_rne(concat(x1*c - x2*s, x2*c + x1*s))   (computed in fp32)
 * k_norm_weight: null (no normalisation) or fp32 [D], 16-byte aligned. When
 * given, each head x of k_new[i] is first replaced by
 *     x_d * k_norm_weight[d] / sqrt(mean_d(x_d^2) + k_norm_eps)
 * (the pages name the k_norm module; this is the Qwen3 family's RMSNorm over
 * the head dims), kept in fp32 and rotated, with one rounding to bf16 at the
 * end. k_norm_eps must be finite and >= 0 (else PKV_ERR_ARG); it is ignored
 * without a weight.
 * A position outside [0, rope_len) sets PKV_DEV_ERR_BAD_POS and skips the
 * token; everything else (slots, pages, errors, races) is as pkv_append.
 */
pkv_status pkv_append_rope(const pkv_cache_desc* cache, void* k_pool, void* v_pool,
                           const int32_t* page_table, const void* k_new,
                           const void* v_new, const int32_t* batch_idx,
                           const int32_t* input_pos, int n_tokens,
                           const float* rope_cos, const float* rope_sin, int rope_len,
                           const float* k_norm_weight, float k_norm_eps,
                           int32_t* dev_err, cudaStream_t stream);

/*
 * pkv_decode_workspace_size - bytes of workspace pkv_decode_attention needs
 * on the CURRENT device for `batch` rows and `num_q_heads` query heads.
 * max_seq_len is accepted for interface stability; the split-KV schedule
 * balances work over the device's SMs and its scratch does not grow with
 * sequence length. A batch above 512 rows runs as equal launches of at most
 * 512 rows that reuse the workspace, so the size is that of one launch.
 * Returns 0 for invalid arguments.
 */
size_t pkv_decode_workspace_size(const pkv_cache_desc* cache, int batch,
                                 int num_q_heads, int max_seq_len);

/*
 * pkv_decode_attention - split-KV GQA decode over the paged cache.
 * Source: "qwen3_flex_inference.py", _decode_block_mask (causal_offset:
 * keys kv_idx <= input_pos of the row's own slot), attention forward
 * (enable_gqa); zero-safe padded rows: "flex_vs_vllm.md", "What broke
 * correctness and had to be dropped" (ROWS_GUARANTEED_SAFE).
 *
 * batch may be any count >= 0. Above 512 rows (the kernels' row tables in
 * shared memory) the call enqueues equal launches of at most 512 rows each,
 * in row order on `stream`, sharing the workspace.
 * Row b in [0, batch) has one query token q[b] (bf16 [num_q_heads, D] within
 * a contiguous [batch, num_q_heads, D] tensor) and attends the first
 * n = seq_lens[b] logical keys of slot c = batch_idx[b] (for a decode step
 * seq_lens[b] = input_pos[b] + 1, the new token included). Query head h reads
 * kv head h / (num_q_heads / num_kv_heads). Writes
 *   lse[b, h] = ln sum_{t<n} exp(scale * q[b,h] . K[c,t,kvh])       (fp32)
 *   out[b, h] = sum_{t<n} exp(scale * q[b,h] . K[c,t,kvh] - lse) V[c,t,kvh]
 * out: bf16 [batch, num_q_heads, D] (rounded to nearest even); lse: fp32
 * [batch, num_q_heads], natural log. Rows with c == 0 or n == 0 give out = 0
 * and lse = -inf (never NaN). A row with c outside [0, max_batch) or
 * n > max_blocks * page_size (or n < 0) sets a PKV_DEV_ERR bit and gives
 * 0 / -inf; a page entry out of range within the first n keys sets
 * PKV_DEV_ERR_BAD_PAGE and leaves that row unspecified.
 * out and lse are only written, with plain stores (no bulk copies): besides
 * device memory they may be pinned host memory mapped into the device's
 * address space (unified addressing), so that the results land on the host
 * without a separate copy; the caller synchronises the stream before reading.
 *
 * q, batch_idx and seq_lens (and k_new, v_new of the fused call) may
 * likewise be pinned host memory mapped into the device's address space:
 * the kernels then read them over the host link (q's rows by ordinary
 * asynchronous copies, the rest by plain loads), so a step needs no input
 * copy; the host must not rewrite them before the call has completed. q in
 * pageable host memory, which the GPU cannot read, returns PKV_ERR_ARG. The
 * pools, the page table, the workspace and dev_err stay in device memory.
 *
 * workspace: device scratch of at least pkv_decode_workspace_size() bytes,
 * 256-byte aligned, owned by the caller; its contents need no initialisation
 * and are overwritten; calls that share a workspace must be stream-ordered.
 * Each launch runs two kernels: the split-KV pass and the LSE merge.
 */
pkv_status pkv_decode_attention(const pkv_cache_desc* cache, const void* k_pool,
                                const void* v_pool, const int32_t* page_table,
                                const void* q, int num_q_heads,
                                const int32_t* batch_idx,
                                const int32_t* seq_lens, int batch, float scale,
                                void* out, float* lse, void* workspace,
                                size_t workspace_bytes, int32_t* dev_err,
                                cudaStream_t stream);

/*
 * pkv_decode_append_attention - one decode step's KV append fused into the
 * decode attention (one launch fewer than pkv_append + pkv_decode_attention).
 * Source: the pages' decode step writes the new token's K/V into the paged
 * cache, then attends over the cache including it ("qwen3_flex_inference.py",
 * forward "Write to paged KV cache" then flex_attention with
 * _decode_block_mask); fused, a step is one call and one launch fewer.
 *
 * Same arguments and results as pkv_decode_attention, plus k_new, v_new:
 * bf16 [batch, num_kv_heads, D], 16-byte aligned. Row b's new token is
 * written to position seq_lens[b] - 1 of slot batch_idx[b] (a decode step has
 * seq_lens[b] = input_pos[b] + 1), exactly as pkv_append would write it
 * (bit-exact byte copy), and the attention of row b includes it. Rows that
 * attend nothing (batch_idx 0, seq_lens 0, or rejected entries) write
 * nothing. A page entry for the new position outside [0, num_pages) skips
 * that write and sets PKV_DEV_ERR_BAD_PAGE. The pools are written, so they
 * are non-const here; k_pool/v_pool must not alias k_new/v_new.
 */
pkv_status pkv_decode_append_attention(const pkv_cache_desc* cache, void* k_pool,
                                       void* v_pool, const int32_t* page_table,
                                       const void* q, int num_q_heads,
                                       const void* k_new, const void* v_new,
                                       const int32_t* batch_idx,
                                       const int32_t* seq_lens, int batch,
                                       float scale, void* out, float* lse,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t* dev_err, cudaStream_t stream);

/*
 * pkv_decode_attention_static_scratch - pkv_decode_attention for callers that
 * cannot allocate device memory. The source pages have no counterpart: this
 * is a deployment convenience of this library.
 *
 * Some callers cannot hand pkv_decode_attention a workspace, because they may
 * not call cudaMalloc at all: code that runs inside a custom allocator's own
 * hooks, processes whose device memory is reserved entirely at start-up, or
 * plug-in hosts that forbid allocations once running. This entry point takes
 * the same arguments minus the workspace and uses a scratch array compiled
 * into the library instead: a file-scope __device__ array of 8 MiB, held on
 * every GPU that loads the library until the process exits. It allocates
 * nothing and calls no allocating routine.
 *  - A call whose pkv_decode_workspace_size() exceeds 8 MiB returns
 *    PKV_ERR_WORKSPACE without launching (one launch of more than about 350
 *    rows at 8 KV heads and a GQA group of 4 on a 152-SM GB300; a batch above
 *    512 rows runs as equal launches, so whether it fits depends on their
 *    size, which pkv_decode_workspace_size() reflects; use
 *    pkv_decode_attention where it does not fit).
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current and caches it; make that
 *    first call before any stream capture. A failed lookup returns
 *    PKV_ERR_CUDA (its text in pkv_last_cuda_error_string()). The cached
 *    address does not survive cudaDeviceReset: after a reset, do not use
 *    this entry point on that device again in the same process.
 *  - Other argument errors give the status pkv_decode_attention gives for
 *    them (an empty batch is validated the same way and returns PKV_OK).
 *  - All calls share the one array. Its contents from the previous call are
 *    never read before being overwritten, so nothing needs clearing, but two
 *    calls whose kernels overlap on the GPU (different streams, or different
 *    host threads without ordering) race on it: keep them stream-ordered.
 * Results are those of pkv_decode_attention on the same inputs.
 */
pkv_status pkv_decode_attention_static_scratch(
    const pkv_cache_desc* cache, const void* k_pool, const void* v_pool,
    const int32_t* page_table, const void* q, int num_q_heads,
    const int32_t* batch_idx, const int32_t* seq_lens, int batch, float scale,
    void* out, float* lse, int32_t* dev_err, cudaStream_t stream);

/*
 * pkv_prefill_paged_attention - chunked prefill over the paged cache, on
 * tcgen05 tensor cores. Source: the step the pages leave on the table
 * ("flex_vs_vllm.md", "What's left on the table": chunked prefill, prefill
 * and decode interleaved in one pass, reading earlier context from the
 * pages); the per-token rule is the decode rule ("qwen3_flex_inference.py",
 * _decode_block_mask, causal_offset: keys kv_idx <= input_pos).
 *
 * q: bf16 [n_tokens, num_q_heads, D], 16-byte aligned; batch_idx, input_pos:
 * int32 [n_tokens]. Token i attends the logical keys 0..input_pos[i] of slot
 * batch_idx[i], read through page_table from k_pool/v_pool:
 *   lse[i, h] = ln sum_{t<=p} exp(scale * q[i,h] . K[slot,t,kvh])       (fp32)
 *   out[i, h] = sum_{t<=p} exp(scale * q[i,h] . K[slot,t,kvh] - lse) V[slot,t,kvh]
 * with kvh = h / (num_q_heads / num_kv_heads). The keys of the token's own
 * chunk must be in the pools already (pkv_append first). Tokens need no order
 * or packing: a chunk of a prompt is its tokens with consecutive positions, a
 * decode token is a chunk of one, and both can share a call. Tokens of slot 0
 * give out 0, lse -inf. A slot outside [0, max_batch) or a position outside
 * [0, max_blocks * page_size) sets PKV_DEV_ERR_BAD_SLOT / _BAD_POS and gives
 * 0 / -inf; an unreserved page entry among a token's keys sets
 * PKV_DEV_ERR_BAD_PAGE and leaves that token's result unspecified.
 * page_size must be 16, 32, 64 or a multiple of 128 (PKV_ERR_ARG otherwise);
 * scale must be finite and > 0. out: bf16 [n_tokens, num_q_heads, D] and
 * lse: fp32 [n_tokens, num_q_heads], 16- and 4-byte aligned. The pools are
 * only read. A decode token costs a full 128-row product per key tile of its
 * prefix here: in a step that mixes chunks and decode tokens, the decode
 * tokens are cheaper through pkv_decode_append_attention.
 */
pkv_status pkv_prefill_paged_attention(const pkv_cache_desc* cache, const void* k_pool,
                                       const void* v_pool, const int32_t* page_table,
                                       const void* q, int num_q_heads,
                                       const int32_t* batch_idx,
                                       const int32_t* input_pos, int n_tokens,
                                       float scale, void* out, float* lse,
                                       int32_t* dev_err, cudaStream_t stream);

/*
 * pkv_prefill_attention - packed document-causal prefill on tcgen05 tensor
 * cores. Source: "qwen3_flex_inference.py", _prefill (prompts concatenated
 * into one sequence with a document-causal mask; the mask built without
 * paging, so attention reads the packed fresh k/v).
 *
 * q: bf16 [n_tokens, num_q_heads, D]; k, v: bf16 [n_tokens, num_kv_heads, D];
 * batch_idx, input_pos: int32 [n_tokens]. Token i may attend token j iff
 * batch_idx[j] == batch_idx[i] != 0 and input_pos[j] <= input_pos[i].
 * Precondition (the pages' packing): each document's tokens are contiguous
 * and numbered input_pos = 0, 1, 2, ...; padding tokens carry batch_idx 0.
 * A token that breaks it sets PKV_DEV_ERR_LAYOUT (its row is unspecified).
 * Writes out bf16 [n_tokens, num_q_heads, D] and lse fp32
 * [n_tokens, num_q_heads] with the same formulas as decode; padding tokens
 * give 0 / -inf. scale must be finite and > 0. q, k, v and out are
 * 16-byte aligned device memory (out is written with bulk tensor stores).
 * Writing the k/v into the pages is a separate pkv_append.
 */
pkv_status pkv_prefill_attention(const void* q, const void* k, const void* v,
                                 int num_q_heads, int num_kv_heads,
                                 int head_dim, const int32_t* batch_idx,
                                 const int32_t* input_pos, int n_tokens,
                                 float scale, void* out, float* lse,
                                 int32_t* dev_err, cudaStream_t stream);

/*
 * pkv_mixed_workspace_size - bytes of device scratch pkv_mixed_attention
 * needs for n_tokens tokens (0 for invalid arguments).
 */
size_t pkv_mixed_workspace_size(const pkv_cache_desc* cache, int n_tokens,
                                int num_q_heads);

/*
 * pkv_mixed_attention - one call for a step that interleaves prefill chunks
 * and decode tokens, each token attending its slot's keys 0..input_pos
 * through the page table. Source: the step the pages leave on the table,
 * prefill and decode served in one pass ("flex_vs_vllm.md", "What's left on
 * the table"); the rule per token is the decode rule
 * ("qwen3_flex_inference.py", _decode_block_mask, causal_offset).
 *
 * Arguments, results and error behaviour are those of
 * pkv_prefill_paged_attention (the same out and lse, within rounding), plus
 * a workspace: device scratch of at least pkv_mixed_workspace_size() bytes,
 * 256-byte aligned, owned by the caller, no initialisation needed; calls
 * sharing one must be stream-ordered. Inside, tokens that are a run of one
 * in the packing (a live slot different from both neighbours' slots: decode
 * tokens) are routed to the split-KV decode kernels, up to 512 of them in
 * token order; every other token goes through the chunked prefill, where a
 * lone token would cost a full 128-row product per key tile of its prefix.
 * Four kernels run on `stream`: the routing, the chunked prefill, the
 * split-KV decode and its merge. The chunks' and decode tokens' own K/V must
 * be in the pools already (pkv_append first). page_size must be 16, 32, 64
 * or a multiple of 128.
 */
pkv_status pkv_mixed_attention(const pkv_cache_desc* cache, const void* k_pool,
                               const void* v_pool, const int32_t* page_table,
                               const void* q, int num_q_heads,
                               const int32_t* batch_idx, const int32_t* input_pos,
                               int n_tokens, float scale, void* out, float* lse,
                               void* workspace, size_t workspace_bytes,
                               int32_t* dev_err, cudaStream_t stream);

/*
 * pkv_stage_from_host - copies a step's inputs from pinned host memory into
 * device memory with the GPU's own loads. Source: the pages' decode step
 * copies each step's inputs into the static buffers its captured graph reads,
 * then replays the graph ("qwen3_flex_inference.py", _decode_step and
 * capture_decode_cudagraph). On GB300 a copy-engine transfer of such a step's
 * inputs (under 1 MB) costs ~14 us of mostly fixed latency; read by the SMs
 * over the coherent host link it takes a few microseconds.
 *
 * dst: device (or managed) memory; src: pinned host memory (cudaHostAlloc,
 * cudaMallocHost or cudaHostRegister; device memory also works); bytes a
 * multiple of 16, both pointers 16-byte aligned (PKV_ERR_ARG /
 * PKV_ERR_ALIGN otherwise, nothing launched). Memory the GPU cannot reach
 * (pageable host memory) is rejected with PKV_ERR_ARG before any launch.
 * The copy is one kernel on `stream`; a kernel that starts after it on the
 * stream (a programmatic dependent such as the decode kernels included)
 * sees the copied bytes. src must not change until the copy has run.
 */
pkv_status pkv_stage_from_host(void* dst, const void* src, size_t bytes,
                               cudaStream_t stream);

/* Static, human-readable name of a status. */
const char* pkv_status_string(pkv_status status);

/* Text of the CUDA runtime error behind the calling thread's most recent
 * PKV_ERR_CUDA (static storage; "no error" if there was none). */
const char* pkv_last_cuda_error_string(void);

/* Maps a dev_err word read back by the caller to a status: PKV_OK when 0,
 * PKV_ERR_BAD_PAGE when the bad-page bit is set, PKV_ERR_BAD_INPUT else. */
pkv_status pkv_status_from_device_error(int32_t dev_err_value);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
