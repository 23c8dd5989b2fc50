// pkv_stage.cu - pkv_stage_from_host: the GPU's own loads bring a pinned host
// buffer into device memory.
//
// A decode step's inputs (q, the new K/V, slots, lengths, page-table rows)
// are under a megabyte. Moved by a copy engine, such a copy costs ~14 us on
// GB300, almost all of it fixed latency; read by the SMs over the coherent
// host link, the same bytes arrive in a few microseconds. The copy is a plain
// grid-stride loop of 16-byte loads and stores; every CTA fences its writes
// before it exits, so a kernel that starts after this grid completes (a
// programmatic dependent included) reads the staged bytes.
#include "pkv.h"
#include "pkv_launch.h"

namespace pkv {
namespace {

constexpr int kStageThreads = 256;
constexpr int kStageUnroll = 4;

__global__ void __launch_bounds__(kStageThreads) stage_kernel(uint4* __restrict__ dst,
                                                              const uint4* __restrict__ src,
                                                              size_t n16) {
  const size_t stride = static_cast<size_t>(gridDim.x) * kStageThreads;
  size_t i = static_cast<size_t>(blockIdx.x) * kStageThreads + threadIdx.x;
  for (; i + (kStageUnroll - 1) * stride < n16; i += kStageUnroll * stride) {
    uint4 v[kStageUnroll];
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u) v[u] = src[i + u * stride];
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u) dst[i + u * stride] = v[u];
  }
  for (; i < n16; i += stride) dst[i] = src[i];
  __threadfence();
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_stage_from_host(void* dst, const void* src, size_t bytes,
                                          cudaStream_t stream) {
  if (bytes == 0) return PKV_OK;
  if (dst == nullptr || src == nullptr || bytes % 16 != 0) return PKV_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(dst) % 16 != 0 || reinterpret_cast<uintptr_t>(src) % 16 != 0)
    return PKV_ERR_ALIGN;
  // the GPU must be able to reach both buffers: src pinned (or device or
  // managed) memory, dst device (or managed) memory; pageable host memory is
  // rejected here, before anything is launched
  cudaPointerAttributes as, ad;
  cudaError_t e = cudaPointerGetAttributes(&as, src);
  if (e != cudaSuccess) return pkv::record_cuda_status(e);
  e = cudaPointerGetAttributes(&ad, dst);
  if (e != cudaSuccess) return pkv::record_cuda_status(e);
  if (as.type == cudaMemoryTypeUnregistered || as.devicePointer == nullptr) return PKV_ERR_ARG;
  if (ad.type != cudaMemoryTypeDevice && ad.type != cudaMemoryTypeManaged) return PKV_ERR_ARG;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return pkv::record_cuda_status(e);
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return pkv::record_cuda_status(e);
  const size_t n16 = bytes / 16;
  const size_t per_cta = static_cast<size_t>(pkv::kStageThreads) * pkv::kStageUnroll;
  const size_t want = (n16 + per_cta - 1) / per_cta;
  const unsigned grid = static_cast<unsigned>(want < static_cast<size_t>(4 * sms) ? want : 4 * sms);
  pkv::stage_kernel<<<grid, pkv::kStageThreads, 0, stream>>>(
      static_cast<uint4*>(ad.devicePointer ? ad.devicePointer : dst),
      static_cast<const uint4*>(as.devicePointer), n16);
  return pkv::record_cuda_status(cudaGetLastError());
}
