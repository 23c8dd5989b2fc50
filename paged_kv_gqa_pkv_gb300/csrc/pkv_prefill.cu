// pkv_prefill.cu - K4 packed document-causal prefill (host validation; the
// tcgen05 kernel follows).
#include <cmath>

#include "pkv_launch.h"

namespace pkv {

namespace {
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
}  // namespace

pkv_status prefill_entry(const void* q, const void* k, const void* v, int num_q_heads,
                         int num_kv_heads, int head_dim, const int32_t* batch_idx,
                         const int32_t* input_pos, int n_tokens, float scale, void* out,
                         float* lse, int32_t* dev_err, cudaStream_t stream) {
  (void)stream;
  if (head_dim != kHeadDim || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads != 0)
    return PKV_ERR_ARG;
  const int g = num_q_heads / num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return PKV_ERR_ARG;
  if (n_tokens < 0 || !std::isfinite(scale)) return PKV_ERR_ARG;
  if (n_tokens == 0) return PKV_OK;
  if (!q || !k || !v || !batch_idx || !input_pos || !out || !lse) return PKV_ERR_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(batch_idx, 4) || !aligned(input_pos, 4) ||
      !aligned(dev_err, 4))
    return PKV_ERR_ALIGN;
  return PKV_ERR_DEVICE;
}

}  // namespace pkv
