// pkv_decode_static.cu - decode attention for callers that cannot allocate.
//
// pkv_decode_attention needs a scratch workspace from its caller. Some callers
// cannot provide one: code running where cudaMalloc is off limits (inside a
// custom allocator's own callbacks, in a process whose memory pool is fully
// reserved up front, or in plug-in hosts that forbid device allocations after
// start-up). For them, pkv_decode_attention_static_scratch uses a scratch
// array compiled into this library instead. The array is a file-scope
// __device__ variable of kStaticScratchBytes (8 MiB), so every GPU that loads
// the library holds those 8 MiB until the process exits. Nothing here calls
// cudaMalloc, cudaFree or any allocating routine.
//
// The array's name in host code is only a host-side handle for the symbol, not
// a device address: the device address is looked up with cudaGetSymbolAddress
// the first time the entry point runs on a device (with that device current),
// and cached per device. The cache is not told about cudaDeviceReset: a
// process that resets a device and keeps using this library on it holds a
// stale address (the header says so).
#include <mutex>

#include "pkv.h"
#include "pkv_launch.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t{8} << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// Device address of g_decode_scratch on the current device, looked up once
// per device. Returns nullptr (and sets *err) when the lookup fails.
void* scratch_address(cudaError_t* err) {
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* ptr = nullptr;
    *err = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = ptr;
  }
  return addr[dev];
}

}  // namespace

extern "C" pkv_status pkv_decode_attention_static_scratch(
    const pkv_cache_desc* cache, const void* k_pool, const void* v_pool,
    const int32_t* page_table, const void* q, int num_q_heads, const int32_t* batch_idx,
    const int32_t* seq_lens, int batch, float scale, void* out, float* lse, int32_t* dev_err,
    cudaStream_t stream) {
  const size_t need =
      batch > 0 ? pkv_decode_workspace_size(cache, batch, num_q_heads, 0) : size_t{0};
  // An empty batch, or arguments the workspace entry point rejects (invalid
  // descriptor, GQA group or batch, unsupported device): that entry point,
  // given no workspace, runs the same checks and returns the same status.
  if (need == 0)
    return pkv_decode_attention(cache, k_pool, v_pool, page_table, q, num_q_heads, batch_idx,
                                seq_lens, batch, scale, out, lse, nullptr, 0, dev_err, stream);
  if (need > kStaticScratchBytes) return PKV_ERR_WORKSPACE;  // past the fixed maximum
  cudaError_t err = cudaSuccess;
  void* scratch = scratch_address(&err);
  if (scratch == nullptr) return pkv::record_cuda_status(err);
  return pkv_decode_attention(cache, k_pool, v_pool, page_table, q, num_q_heads, batch_idx,
                              seq_lens, batch, scale, out, lse, scratch, kStaticScratchBytes,
                              dev_err, stream);
}
