// pkv_api.cu - the extern "C" entry points of libpkv (declared in pkv.h):
// synchronous host validation, TMA descriptor encoding and kernel launches.
// Nothing here allocates device memory or synchronises a stream.
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <utility>

#include "pkv.h"
#include "pkv_launch.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, found through the runtime so the
// library does not link against libcuda.
EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

struct DeviceInfo {
  bool known = false;
  bool supported = false;
  int sm_count = 0;
};

constexpr int kMaxDevices = 64;

// SM count and architecture of `dev`, queried once per device.
pkv_status device_info(int* sm_count) {
  static DeviceInfo cache[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pkv::record_cuda_status(e);
  if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& d = cache[dev];
  if (!d.known) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return pkv::record_cuda_status(e);
    d.supported = (major == 10 && minor == 3);  // built for sm_103a only
    d.sm_count = sms;
    d.known = true;
  }
  if (!d.supported) return PKV_ERR_DEVICE;
  *sm_count = d.sm_count;
  return PKV_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

pkv_status cuda_status(cudaError_t e) { return pkv::record_cuda_status(e); }

pkv_status check_cache(const pkv_cache_desc* c) {
  if (c == nullptr) return PKV_ERR_ARG;
  if (c->num_pages <= 0 || c->page_size <= 0 || c->page_size % 16 != 0) return PKV_ERR_ARG;
  if (c->num_kv_heads <= 0 || c->head_dim != pkv::kHeadDim) return PKV_ERR_ARG;
  if (c->max_batch <= 0 || c->max_blocks <= 0) return PKV_ERR_ARG;
  if (static_cast<long long>(c->num_pages) * c->page_size > INT_MAX) return PKV_ERR_ARG;
  if (static_cast<long long>(c->max_blocks) * c->page_size > INT_MAX) return PKV_ERR_ARG;
  if (static_cast<long long>(c->max_batch) * c->max_blocks > INT_MAX) return PKV_ERR_ARG;
  return PKV_OK;
}

bool group_ok(int num_q_heads, int num_kv_heads) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return false;
  const int g = num_q_heads / num_kv_heads;
  return g == 1 || g == 2 || g == 4 || g == 8;
}

pkv_status encode_pool_map(CUtensorMap* map, const void* pool, const pkv_cache_desc* c) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return PKV_ERR_CUDA;
  // 4-D view {64 dims, rows, 2 halves of the head dims, H_kv}: the halves get
  // their own axis (stride 128 B) so that one box {64, 16 tokens, 2, 1} is a
  // whole 16-token tile of one head, landing as two 128-byte-swizzled
  // [16 rows x 128 B] halves, the layout ldmatrix reads.
  const cuuint64_t dims[4] = {64u, static_cast<cuuint64_t>(c->num_pages) * c->page_size, 2u,
                              static_cast<cuuint64_t>(c->num_kv_heads)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(c->num_kv_heads) * c->head_dim * 2,
                                 128u, static_cast<cuuint64_t>(c->head_dim) * 2};
  const cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(pkv::kDecodeTile), 2u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  std::memset(map, 0, sizeof(*map));
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_ARG;
}

}  // namespace

namespace pkv {
pkv_status record_cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return PKV_OK;
  t_last_cuda_error = e;
  return PKV_ERR_CUDA;
}
}  // namespace pkv

namespace {

// Shared by the attention-only and the append-fused entry points: k_new and
// v_new null means attention alone (the pools are then only read).
pkv_status decode_entry(const pkv_cache_desc* cache, const void* k_pool, const void* v_pool,
                        const int32_t* page_table, const void* q, int num_q_heads,
                        const void* k_new, const void* v_new, const int32_t* batch_idx,
                        const int32_t* seq_lens, int batch, float scale, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, int32_t* dev_err,
                        cudaStream_t stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (batch < 0) return PKV_ERR_ARG;
  if (!group_ok(num_q_heads, cache->num_kv_heads)) return PKV_ERR_ARG;
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return PKV_ERR_ARG;
  if (batch == 0) return PKV_OK;
  if (!k_pool || !v_pool || !page_table || !q || !batch_idx || !seq_lens || !out || !lse)
    return PKV_ERR_ARG;
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(q, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(page_table, 4) || !aligned(batch_idx, 4) ||
      !aligned(seq_lens, 4) || !aligned(dev_err, 4))
    return PKV_ERR_ALIGN;
  int sms = 0;
  st = device_info(&sms);
  if (st != PKV_OK) return st;
  const int group = num_q_heads / cache->num_kv_heads;
  const int workers = pkv::decode_workers_for_device(sms);
  // A batch past the kernels' row tables runs as consecutive launches of at
  // most kDecodeMaxBatch rows each, equal in size, on the caller's stream;
  // they reuse one workspace in stream order.
  const int64_t launches =
      (static_cast<int64_t>(batch) + pkv::kDecodeMaxBatch - 1) / pkv::kDecodeMaxBatch;
  const int rows_per_launch = static_cast<int>((batch + launches - 1) / launches);
  const size_t need =
      pkv::decode_workspace_bytes(rows_per_launch, cache->num_kv_heads, group, workers);
  if (workspace == nullptr || workspace_bytes < need) return PKV_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PKV_ERR_ALIGN;
  // q may sit in mapped pinned host memory (its rows then arrive by cp.async,
  // read over the host link); pageable host memory the GPU cannot reach
  cudaPointerAttributes qa;
  const cudaError_t qe = cudaPointerGetAttributes(&qa, q);
  if (qe != cudaSuccess) return pkv::record_cuda_status(qe);
  if (qa.type == cudaMemoryTypeUnregistered || qa.devicePointer == nullptr) return PKV_ERR_ARG;
  const bool q_host = qa.type == cudaMemoryTypeHost;

  CUtensorMap kmap, vmap;
  st = encode_pool_map(&kmap, k_pool, cache);
  if (st != PKV_OK) return st;
  st = encode_pool_map(&vmap, v_pool, cache);
  if (st != PKV_OK) return st;

  pkv::DecodeParams p;
  p.q = q_host ? qa.devicePointer : q;
  p.q_host = q_host ? 1 : 0;
  p.page_table = page_table;
  p.batch_idx = batch_idx;
  p.seq_lens = seq_lens;
  p.out = out;
  p.lse = lse;
  p.partials = static_cast<float*>(workspace);
  p.k_new = k_new;
  p.v_new = v_new;
  p.k_pool = const_cast<void*>(k_pool);
  p.v_pool = const_cast<void*>(v_pool);
  p.row_token = nullptr;
  p.row_count = nullptr;
  p.input_pos = nullptr;
  p.dev_err = dev_err;
  p.batch = batch;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = cache->num_kv_heads;
  p.page_size = cache->page_size;
  p.num_pages = cache->num_pages;
  p.max_batch = cache->max_batch;
  p.max_blocks = cache->max_blocks;
  p.num_workers = workers;
  p.qscale = scale * 1.4426950408889634f;
  if (launches == 1) return cuda_status(pkv::launch_decode(p, kmap, vmap, sms, stream));
  const size_t q_row = static_cast<size_t>(num_q_heads) * cache->head_dim * 2;
  const size_t kv_row = static_cast<size_t>(cache->num_kv_heads) * cache->head_dim * 2;
  for (int64_t r0 = 0; r0 < batch; r0 += rows_per_launch) {
    pkv::DecodeParams pr = p;
    pr.batch = static_cast<int>(batch - r0 < rows_per_launch ? batch - r0 : rows_per_launch);
    pr.q = static_cast<const uint8_t*>(p.q) + r0 * q_row;
    pr.batch_idx = batch_idx + r0;
    pr.seq_lens = seq_lens + r0;
    pr.out = static_cast<uint8_t*>(out) + r0 * q_row;
    pr.lse = lse + static_cast<size_t>(r0) * num_q_heads;
    if (k_new != nullptr) {
      pr.k_new = static_cast<const uint8_t*>(k_new) + r0 * kv_row;
      pr.v_new = static_cast<const uint8_t*>(v_new) + r0 * kv_row;
    }
    const pkv_status s = cuda_status(pkv::launch_decode(pr, kmap, vmap, sms, stream));
    if (s != PKV_OK) return s;
  }
  return PKV_OK;
}

// Workspace of pkv_mixed_attention: the routed-token and query-tile counts,
// the routed tokens (up to `cap`), one skip byte per token, the first token
// of each prefill query tile, then the decode partials; each part 256-byte
// aligned.
struct MixedLayout {
  int cap;
  size_t off_list, off_skip, off_seg, off_part, total;
};

MixedLayout mixed_layout(int n_tokens, int num_kv_heads, int group, int workers) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  MixedLayout m;
  m.cap = n_tokens < pkv::kDecodeMaxBatch ? n_tokens : pkv::kDecodeMaxBatch;
  m.off_list = 256;  // [0]: routed count, [1]: query-tile count
  m.off_skip = m.off_list + up(static_cast<size_t>(m.cap) * 4);
  m.off_seg = m.off_skip + up(static_cast<size_t>(n_tokens));
  m.off_part = m.off_seg + up(static_cast<size_t>(n_tokens) * 4);
  m.total = m.off_part + pkv::decode_workspace_bytes(m.cap, num_kv_heads, group, workers);
  return m;
}

bool paged_page_size_ok(int ps) { return ps == 16 || ps == 32 || ps == 64 || ps % 128 == 0; }

}  // namespace

extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_ARG: return "invalid argument";
    case PKV_ERR_ALIGN: return "misaligned pointer";
    case PKV_ERR_BAD_PAGE: return "page table entry out of range";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_CUDA: return "CUDA runtime error";
    case PKV_ERR_DEVICE: return "current device is not a supported sm_103 GPU";
    case PKV_ERR_BAD_INPUT: return "invalid slot, position or packing found on the device";
  }
  return "unknown status";
}

const char* pkv_last_cuda_error_string(void) {
  return t_last_cuda_error == cudaSuccess ? "no error" : cudaGetErrorString(t_last_cuda_error);
}

pkv_status pkv_status_from_device_error(int32_t v) {
  if (v == 0) return PKV_OK;
  if (v & PKV_DEV_ERR_BAD_PAGE) return PKV_ERR_BAD_PAGE;
  return PKV_ERR_BAD_INPUT;
}

pkv_status pkv_append(const pkv_cache_desc* cache, void* k_pool, void* v_pool,
                      const int32_t* page_table, const void* k_new, const void* v_new,
                      const int32_t* batch_idx, const int32_t* input_pos, int n_tokens,
                      int32_t* dev_err, cudaStream_t stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (n_tokens < 0) return PKV_ERR_ARG;
  if (n_tokens == 0) return PKV_OK;
  if (!k_pool || !v_pool || !page_table || !k_new || !v_new || !batch_idx || !input_pos)
    return PKV_ERR_ARG;
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) ||
      !aligned(page_table, 4) || !aligned(batch_idx, 4) || !aligned(input_pos, 4) ||
      !aligned(dev_err, 4))
    return PKV_ERR_ALIGN;
  int sms = 0;
  st = device_info(&sms);
  if (st != PKV_OK) return st;
  pkv::AppendParams p;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.page_table = page_table;
  p.k_new = k_new;
  p.v_new = v_new;
  p.batch_idx = batch_idx;
  p.input_pos = input_pos;
  p.dev_err = dev_err;
  p.n_tokens = n_tokens;
  p.row_vecs = cache->num_kv_heads * cache->head_dim * 2 / 16;
  p.page_size = cache->page_size;
  p.num_pages = cache->num_pages;
  p.max_batch = cache->max_batch;
  p.max_blocks = cache->max_blocks;
  return cuda_status(pkv::launch_append(p, stream));
}

pkv_status pkv_append_rope(const pkv_cache_desc* cache, void* k_pool, void* v_pool,
                           const int32_t* page_table, const void* k_new, const void* v_new,
                           const int32_t* batch_idx, const int32_t* input_pos, int n_tokens,
                           const float* rope_cos, const float* rope_sin, int rope_len,
                           const float* k_norm_weight, float k_norm_eps, int32_t* dev_err,
                           cudaStream_t stream) {
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (n_tokens < 0 || rope_len <= 0) return PKV_ERR_ARG;
  if (k_norm_weight != nullptr && !(k_norm_eps >= 0.f && k_norm_eps < INFINITY))
    return PKV_ERR_ARG;
  if (n_tokens == 0) return PKV_OK;
  if (!k_pool || !v_pool || !page_table || !k_new || !v_new || !batch_idx || !input_pos ||
      !rope_cos || !rope_sin)
    return PKV_ERR_ARG;
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) ||
      !aligned(rope_cos, 16) || !aligned(rope_sin, 16) || !aligned(page_table, 4) ||
      !aligned(batch_idx, 4) || !aligned(input_pos, 4) || !aligned(dev_err, 4) ||
      !aligned(k_norm_weight, 16))
    return PKV_ERR_ALIGN;
  int sms = 0;
  st = device_info(&sms);
  if (st != PKV_OK) return st;
  pkv::AppendRopeParams p;
  p.a.k_pool = k_pool;
  p.a.v_pool = v_pool;
  p.a.page_table = page_table;
  p.a.k_new = k_new;
  p.a.v_new = v_new;
  p.a.batch_idx = batch_idx;
  p.a.input_pos = input_pos;
  p.a.dev_err = dev_err;
  p.a.n_tokens = n_tokens;
  p.a.row_vecs = cache->num_kv_heads * cache->head_dim * 2 / 16;
  p.a.page_size = cache->page_size;
  p.a.num_pages = cache->num_pages;
  p.a.max_batch = cache->max_batch;
  p.a.max_blocks = cache->max_blocks;
  p.rope_cos = rope_cos;
  p.rope_sin = rope_sin;
  p.rope_len = rope_len;
  p.num_kv_heads = cache->num_kv_heads;
  p.k_norm_weight = k_norm_weight;
  p.k_norm_eps = k_norm_eps;
  return cuda_status(pkv::launch_append_rope(p, stream));
}

size_t pkv_decode_workspace_size(const pkv_cache_desc* cache, int batch, int num_q_heads,
                                 int max_seq_len) {
  (void)max_seq_len;
  if (check_cache(cache) != PKV_OK || batch < 0) return 0;
  if (!group_ok(num_q_heads, cache->num_kv_heads)) return 0;
  int sms = 0;
  if (device_info(&sms) != PKV_OK) return 0;
  // rows of one launch: larger batches run as equal launches of at most
  // kDecodeMaxBatch rows that reuse the workspace
  const int64_t launches =
      (static_cast<int64_t>(batch) + pkv::kDecodeMaxBatch - 1) / pkv::kDecodeMaxBatch;
  const int rows = launches > 1 ? static_cast<int>((batch + launches - 1) / launches) : batch;
  return pkv::decode_workspace_bytes(rows, cache->num_kv_heads,
                                     num_q_heads / cache->num_kv_heads,
                                     pkv::decode_workers_for_device(sms));
}


pkv_status pkv_decode_attention(const pkv_cache_desc* cache, const void* k_pool,
                                const void* v_pool, const int32_t* page_table, const void* q,
                                int num_q_heads, const int32_t* batch_idx,
                                const int32_t* seq_lens, int batch, float scale, void* out,
                                float* lse, void* workspace, size_t workspace_bytes,
                                int32_t* dev_err, cudaStream_t stream) {
  return decode_entry(cache, k_pool, v_pool, page_table, q, num_q_heads, nullptr, nullptr,
                      batch_idx, seq_lens, batch, scale, out, lse, workspace, workspace_bytes,
                      dev_err, stream);
}

pkv_status pkv_decode_append_attention(const pkv_cache_desc* cache, void* k_pool, void* v_pool,
                                       const int32_t* page_table, const void* q,
                                       int num_q_heads, const void* k_new, const void* v_new,
                                       const int32_t* batch_idx, const int32_t* seq_lens,
                                       int batch, float scale, void* out, float* lse,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t* dev_err, cudaStream_t stream) {
  if (batch > 0 && (k_new == nullptr || v_new == nullptr)) return PKV_ERR_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16)) return PKV_ERR_ALIGN;
  return decode_entry(cache, k_pool, v_pool, page_table, q, num_q_heads, k_new, v_new,
                      batch_idx, seq_lens, batch, scale, out, lse, workspace, workspace_bytes,
                      dev_err, stream);
}

pkv_status pkv_prefill_paged_attention(const pkv_cache_desc* cache, const void* k_pool,
                                      const void* v_pool, const int32_t* page_table,
                                      const void* q, int num_q_heads, const int32_t* batch_idx,
                                      const int32_t* input_pos, int n_tokens, float scale,
                                      void* out, float* lse, int32_t* dev_err,
                                      cudaStream_t stream) {
  const pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  return pkv::prefill_paged_entry(cache, k_pool, v_pool, page_table, q, num_q_heads, batch_idx,
                                  input_pos, n_tokens, scale, out, lse, dev_err, stream);
}

size_t pkv_mixed_workspace_size(const pkv_cache_desc* cache, int n_tokens, int num_q_heads) {
  if (check_cache(cache) != PKV_OK || n_tokens < 0) return 0;
  if (!group_ok(num_q_heads, cache->num_kv_heads)) return 0;
  int sms = 0;
  if (device_info(&sms) != PKV_OK) return 0;
  return mixed_layout(n_tokens, cache->num_kv_heads, num_q_heads / cache->num_kv_heads,
                      pkv::decode_workers_for_device(sms))
      .total;
}

pkv_status pkv_mixed_attention(const pkv_cache_desc* cache, const void* k_pool,
                               const void* v_pool, const int32_t* page_table, const void* q,
                               int num_q_heads, const int32_t* batch_idx,
                               const int32_t* input_pos, int n_tokens, float scale, void* out,
                               float* lse, void* workspace, size_t workspace_bytes,
                               int32_t* dev_err, cudaStream_t stream) {
  // every check of both kernels runs here, before anything is launched
  pkv_status st = check_cache(cache);
  if (st != PKV_OK) return st;
  if (!paged_page_size_ok(cache->page_size)) return PKV_ERR_ARG;
  if (!group_ok(num_q_heads, cache->num_kv_heads)) return PKV_ERR_ARG;
  if (n_tokens < 0 || !std::isfinite(scale) || !(scale > 0.f)) return PKV_ERR_ARG;
  if (n_tokens == 0) return PKV_OK;
  if (!k_pool || !v_pool || !page_table || !q || !batch_idx || !input_pos || !out || !lse)
    return PKV_ERR_ARG;
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(q, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(page_table, 4) || !aligned(batch_idx, 4) ||
      !aligned(input_pos, 4) || !aligned(dev_err, 4))
    return PKV_ERR_ALIGN;
  if (static_cast<long long>(((n_tokens + 127) / 128)) * num_q_heads > INT_MAX)
    return PKV_ERR_ARG;
  int sms = 0;
  st = device_info(&sms);
  if (st != PKV_OK) return st;
  const int group = num_q_heads / cache->num_kv_heads;
  const int workers = pkv::decode_workers_for_device(sms);
  const MixedLayout lay = mixed_layout(n_tokens, cache->num_kv_heads, group, workers);
  if (workspace == nullptr || workspace_bytes < lay.total) return PKV_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PKV_ERR_ALIGN;
  CUtensorMap kmap, vmap;
  st = encode_pool_map(&kmap, k_pool, cache);
  if (st != PKV_OK) return st;
  st = encode_pool_map(&vmap, v_pool, cache);
  if (st != PKV_OK) return st;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* count = reinterpret_cast<int32_t*>(ws);
  int32_t* seg_count = count + 1;
  int32_t* list = reinterpret_cast<int32_t*>(ws + lay.off_list);
  uint8_t* skip = ws + lay.off_skip;
  int32_t* seg_start = reinterpret_cast<int32_t*>(ws + lay.off_seg);
  // 1. the tokens that are a run of one, listed and flagged, and the query
  //    tiles of the others
  cudaError_t e = pkv::launch_route_lone(batch_idx, n_tokens, lay.cap, list, count, skip,
                                         seg_start, seg_count, stream);
  if (e != cudaSuccess) return cuda_status(e);
  // 2. every other token through the chunked prefill, tiled by run pieces
  st = pkv::prefill_paged_entry(cache, k_pool, v_pool, page_table, q, num_q_heads, batch_idx,
                                input_pos, n_tokens, scale, out, lse, dev_err, stream, skip,
                                seg_start, seg_count);
  if (st != PKV_OK) return st;
  // 3. the listed tokens through the split-KV decode and its merge
  pkv::DecodeParams p;
  p.q = q;
  p.q_host = 0;
  p.page_table = page_table;
  p.batch_idx = batch_idx;
  p.seq_lens = nullptr;
  p.out = out;
  p.lse = lse;
  p.partials = reinterpret_cast<float*>(ws + lay.off_part);
  p.k_new = nullptr;
  p.v_new = nullptr;
  p.k_pool = const_cast<void*>(k_pool);
  p.v_pool = const_cast<void*>(v_pool);
  p.row_token = list;
  p.row_count = count;
  p.input_pos = input_pos;
  p.dev_err = dev_err;
  p.batch = lay.cap;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = cache->num_kv_heads;
  p.page_size = cache->page_size;
  p.num_pages = cache->num_pages;
  p.max_batch = cache->max_batch;
  p.max_blocks = cache->max_blocks;
  p.num_workers = workers;
  p.qscale = scale * 1.4426950408889634f;
  return cuda_status(pkv::launch_decode(p, kmap, vmap, sms, stream));
}

pkv_status pkv_prefill_attention(const void* q, const void* k, const void* v, int num_q_heads,
                                 int num_kv_heads, int head_dim, const int32_t* batch_idx,
                                 const int32_t* input_pos, int n_tokens, float scale, void* out,
                                 float* lse, int32_t* dev_err, cudaStream_t stream) {
  return pkv::prefill_entry(q, k, v, num_q_heads, num_kv_heads, head_dim, batch_idx, input_pos,
                            n_tokens, scale, out, lse, dev_err, stream);
}

}  // extern "C"
