// pkv_prefill.cu - K4 packed document-causal prefill on tcgen05 tensor cores.
//
// Source: "qwen3_flex_inference.py", _prefill: all prompts are concatenated
// into one sequence; token i attends token j iff both belong to the same
// document (batch slot != 0) and input_pos[j] <= input_pos[i]; attention reads
// the packed fresh k/v (the mask is built "no paging"). The pages ran this
// through flex_attention's Triton kernel; FA4 was blocked by its 256-row block
// requirement ("flex_vs_vllm.md", "What I tried that did NOT move the needle").
//
// Packing precondition (the pages' packing): each document is contiguous and
// numbered 0, 1, 2, ...; then the keys of query i are exactly the packed rows
// [i - input_pos[i], i]. A row that breaks it sets PKV_DEV_ERR_LAYOUT.
//
// One CTA computes a 128-row query tile for one query head:
//  * warp 0 issues TMA loads: the Q tile once, then K/V tiles of 128 keys
//    into a two-stage ring, starting at the first key any row of the tile
//    can see (KV tiles outside the tile's documents are never loaded);
//  * warp 1 (one thread) issues the tcgen05 MMAs: S = Q K^T into one of two
//    TMEM buffers (the next S is computed while the current one is in
//    softmax), then O += P V into a TMEM accumulator;
//  * warps 2..5 own one query row per thread (its TMEM lane): masked online
//    softmax in fp32 (exp2 with the scale folded in), P written to shared
//    memory as bf16 in the MMA's K-major 128-byte-swizzled layout, O rescaled
//    in TMEM only when the running max grows by more than 2^8, and the
//    epilogue O / l -> bf16 plus the LSE.
// Shared-memory operands (all 128-byte swizzled, 1024-byte aligned atoms):
// Q, K and P are K-major (64 elements per 128-byte row, two 16 KB halves of
// D or of the key block); V is used MN-major straight from its TMA tile
// (64 head dims per 128-byte row, one row per key).
#include <cmath>

#include "pkv_launch.h"

namespace pkv {

namespace {

constexpr int kBM = 128;                 // query rows per tile
constexpr int kBN = 128;                 // keys per KV tile
constexpr int kHalf = 128 * 128;         // one [128 rows x 64 elems] bf16 block, bytes
constexpr int kTileBytes = 2 * kHalf;    // 128 x 128 bf16
constexpr int kStages = 2;
constexpr int kThreads = 6 * 32;
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kTmemCols = 512;      // S0 [0,128) S1 [128,256) O [256,384)
constexpr uint32_t kColO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// shared memory layout (offsets from a 1024-aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffP = kOffV + kStages * kTileBytes;
constexpr int kOffBar = kOffP + kTileBytes;
// barriers: q_full, kv_full[2], kv_empty[2], s_full[2], p_full, pv_done
constexpr int kNumBars = 9;
constexpr int kOffMisc = kOffBar + kNumBars * 8;   // tmem slot, kv_lo, kv_hi, abort
constexpr int kSmemBytes = kOffMisc + 64 + 1024;   // + slack for 1024 alignment

constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, /*b_mn_major=*/false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kHeadDim, /*b_mn_major=*/true);

struct PrefillParams {
  const int32_t* batch_idx;
  const int32_t* input_pos;
  void* out;
  float* lse;
  int32_t* dev_err;
  int n_tokens;
  int num_q_heads;
  int group;
  float qscale;  // scale * log2(e)
};

__device__ __forceinline__ bool aborted(volatile int* flag) { return *flag != 0; }

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
prefill_tcgen05_kernel(const __grid_constant__ CUtensorMap qmap,
                       const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* p_full = bars + 7;
  uint64_t* pv_done = bars + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  int* s_kv_lo = reinterpret_cast<int*>(smem + kOffMisc + 4);
  int* s_kv_hi = reinterpret_cast<int*>(smem + kOffMisc + 8);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 12);
  int* s_skip = reinterpret_cast<int*>(smem + kOffMisc + 16);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int head = blockIdx.x % p.num_q_heads;
  const int tile = blockIdx.x / p.num_q_heads;
  const int kvh = head / p.group;
  const int r0 = tile * kBM;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
      mbar_init(&s_full[s], 1);
    }
    mbar_init(p_full, kSoftmaxThreads);
    mbar_init(pv_done, 1);
    *s_kv_lo = 0x7fffffff;
    *s_kv_hi = -1;
    *s_abort = 0;
    // After a timeout anywhere in the grid, later CTAs do no work (their
    // results are unspecified then) instead of each waiting out its limit.
    *s_skip = (p.dev_err != nullptr &&
               (*reinterpret_cast<volatile int32_t*>(p.dev_err) & PKV_DEV_ERR_TIMEOUT)) ? 1 : 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);

  // ---- per-row document bounds (softmax threads), CTA-wide key range ----
  const bool is_softmax = warp >= 2;
  const int lane_base = 32 * (warp & 3);  // TMEM lanes this warp may access
  const int row = lane_base + lane;       // query row within the tile
  const int i = r0 + row;                 // packed token index
  bool valid = false;
  int start = 0;
  if (is_softmax && i < p.n_tokens) {
    const int b = p.batch_idx[i];
    const int pos = p.input_pos[i];
    if (b != 0) {
      valid = true;
      bool ok = pos >= 0 && pos <= i;
      if (ok && pos > 0) ok = (p.batch_idx[i - 1] == b) && (p.input_pos[i - 1] == pos - 1);
      if (!ok) set_dev_err(p.dev_err, PKV_DEV_ERR_LAYOUT);
      start = (pos >= 0 && pos <= i) ? i - pos : i;
      atomicMin(s_kv_lo, start);
      atomicMax(s_kv_hi, i + 1);
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int kv_lo = *s_kv_lo;
  const int kv_hi = *s_kv_hi;
  const int n_kv = (kv_hi > kv_lo && *s_skip == 0) ? (kv_hi - kv_lo + kBN - 1) / kBN : 0;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer ----
    if (lane == 0 && n_kv > 0) {
      mbar_arrive_expect_tx(q_full, kTileBytes);
      tma_load_3d(smem + kOffQ, &qmap, q_full, 0, head, r0);
      tma_load_3d(smem + kOffQ + kHalf, &qmap, q_full, 64, head, r0);
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % kStages;
        if (j >= kStages && !mbar_wait_bounded(&kv_empty[s], ((j / kStages) - 1) & 1)) {
          set_dev_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
          *s_abort = 1;
          break;
        }
        const int krow = kv_lo + j * kBN;
        uint8_t* kd = smem + kOffK + s * kTileBytes;
        uint8_t* vd = smem + kOffV + s * kTileBytes;
        mbar_arrive_expect_tx(&kv_full[s], 2 * kTileBytes);
        tma_load_3d(kd, &kmap, &kv_full[s], 0, kvh, krow);
        tma_load_3d(kd + kHalf, &kmap, &kv_full[s], 64, kvh, krow);
        tma_load_3d(vd, &vmap, &kv_full[s], 0, kvh, krow);
        tma_load_3d(vd + kHalf, &vmap, &kv_full[s], 64, kvh, krow);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer ----
    if (lane == 0 && n_kv > 0) {
      const uint32_t sQ = smem_u32(smem + kOffQ);
      const uint32_t sP = smem_u32(smem + kOffP);
      auto issue_qk = [&](int j) {
        const int s = j % kStages;
        const uint32_t sK = smem_u32(smem + kOffK + s * kTileBytes);
        const uint32_t d = tmem + static_cast<uint32_t>((j & 1) * kBN);
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          umma_bf16(d, sw128_desc(sQ + off, 0, 1024), sw128_desc(sK + off, 0, 1024), kIdescQK,
                    kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[j & 1]);
      };
      bool ok = mbar_wait_bounded(q_full, 0) && mbar_wait_bounded(&kv_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_qk(0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv) {
          const int s1 = (j + 1) % kStages;
          if (!mbar_wait_bounded(&kv_full[s1], ((j + 1) / kStages) & 1)) { ok = false; break; }
          tc_fence_after();
          issue_qk(j + 1);
        }
        if (!mbar_wait_bounded(p_full, j & 1)) { ok = false; break; }
        tc_fence_after();
        const int s = j % kStages;
        const uint32_t sV = smem_u32(smem + kOffV + s * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t a_off = (kk >> 2) * kHalf + (kk & 3) * 32;
          umma_bf16(tmem + kColO, sw128_desc(sP + a_off, 0, 1024),
                    sw128_desc(sV + kk * 2048, kHalf, 1024), kIdescPV,
                    (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(pv_done);
        umma_commit(&kv_empty[s]);
      }
      if (!ok) {
        set_dev_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
        *s_abort = 1;
      }
    }
  } else {
    // ------------------------------------------------ softmax rows ----
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(lane_base) << 16);
    float m_run = -INFINITY;  // running max, raw score units
    float l_run = 0.f;
    uint8_t* sP = smem + kOffP;
    bool ok = true;
    for (int j = 0; j < n_kv && ok; ++j) {
      // wait outcomes are made warp-uniform: the TMEM accesses below are
      // warp-collective
      const bool got_s = mbar_wait_bounded(&s_full[j & 1], (j >> 1) & 1) && !aborted(s_abort);
      if (!__all_sync(0xffffffffu, got_s)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
      {
        uint32_t (&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
        uint32_t (&b)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
        uint32_t (&c)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[64]);
        uint32_t (&d)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[96]);
        const uint32_t base = t_lane + static_cast<uint32_t>((j & 1) * kBN);
        tmem_ld32(base + 0, a);
        tmem_ld32(base + 32, b);
        tmem_ld32(base + 64, c);
        tmem_ld32(base + 96, d);
        tmem_wait_ld();
      }
      // mask: key k = kv_lo + j*128 + c is visible iff start <= k <= i
      const int k0 = kv_lo + j * kBN;
      const bool full = valid && k0 >= start && k0 + kBN - 1 <= i;
      float mx = -INFINITY;
      if (full) {
#pragma unroll
        for (int c = 0; c < kBN; ++c) mx = fmaxf(mx, __uint_as_float(sr[c]));
      } else {
#pragma unroll
        for (int c = 0; c < kBN; ++c) {
          const int k = k0 + c;
          const bool vis = valid && k >= start && k <= i;
          const float v = vis ? __uint_as_float(sr[c]) : -INFINITY;
          sr[c] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      }
      // lazy rescale: keep the old max unless it grew by more than 2^8
      const float m_cand = fmaxf(m_run, mx);
      const bool grow = (m_run == -INFINITY) ? (m_cand != -INFINITY)
                                             : ((m_cand - m_run) * p.qscale > kRescaleThreshold);
      const float m_use = grow ? m_cand : m_run;
      const float alpha = grow ? exp2f((m_run - m_use) * p.qscale) : 1.f;  // 0 when m_run=-inf
      const float neg_m = (m_use == -INFINITY) ? 0.f : -m_use * p.qscale;
      float psum = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < kBN; c += 2) {
        const float x0 = __uint_as_float(sr[c]);
        const float x1 = __uint_as_float(sr[c + 1]);
        const float e0 = (x0 == -INFINITY) ? 0.f : exp2f(fmaf(x0, p.qscale, neg_m));
        const float e1 = (x1 == -INFINITY) ? 0.f : exp2f(fmaf(x1, p.qscale, neg_m));
        psum += e0 + e1;
        pk[c >> 1] = pack_bf16x2(e0, e1);
      }
      l_run = l_run * alpha + psum;
      m_run = m_use;
      // P and O are free once the previous PV product has completed
      const bool got_pv = (j == 0) || mbar_wait_bounded(pv_done, (j - 1) & 1);
      if (!__all_sync(0xffffffffu, got_pv)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // P row -> shared memory, K-major SW128: 16-byte chunk q of row r in a
      // 64-key half lives at chunk position q ^ (r % 8)
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int half = q >> 3;
        const int cq = (q & 7) ^ (row & 7);
        uint4* dst = reinterpret_cast<uint4*>(sP + half * kHalf + row * 128 + cq * 16);
        *dst = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
      // O *= alpha when any row of this warp changed its max (warp-collective)
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int c = 0; c < kHeadDim; c += 32) {
          uint32_t o[32];
          tmem_ld32(t_lane + kColO + c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(t_lane + kColO + c, o);
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    // ---- epilogue: O / l, LSE ----
    if (ok && n_kv > 0 && !mbar_wait_bounded(pv_done, (n_kv - 1) & 1)) ok = false;
    if (!ok) {
      set_dev_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
      *s_abort = 1;
    }
    tc_fence_after();
    // Every thread of the warp issues the same TMEM loads (they are
    // warp-collective); only the stores depend on the row.
    const bool in_range = i < p.n_tokens;
    const bool has = in_range && valid && ok && l_run > 0.f;
    const float inv = has ? 1.f / l_run : 0.f;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                          (static_cast<int64_t>(in_range ? i : 0) * p.num_q_heads + head) *
                              kHeadDim;
#pragma unroll
    for (int c = 0; c < kHeadDim; c += 32) {
      uint32_t o[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = 0u;
      if (n_kv > 0) {  // CTA-uniform
        tmem_ld32(t_lane + kColO + c, o);
        tmem_wait_ld();
      }
      if (in_range) {
        uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 w = make_uint4(0u, 0u, 0u, 0u);
          if (has) {
            w.x = pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
          }
          dst[e / 8] = w;
        }
      }
    }
    if (in_range)
      p.lse[static_cast<int64_t>(i) * p.num_q_heads + head] =
          has ? (m_run * p.qscale + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

namespace {
bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// {D, heads, tokens} view; box = 64 head dims x 1 head x 128 tokens, 128-byte
// swizzled (the tcgen05 operand layout).
bool encode_packed_map(CUtensorMap* map, const void* base, int heads, int n_tokens) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(n_tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                                 static_cast<cuuint64_t>(heads) * kHeadDim * 2};
  const cuuint32_t box[3] = {64u, 1u, 128u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

pkv_status prefill_entry(const void* q, const void* k, const void* v, int num_q_heads,
                         int num_kv_heads, int head_dim, const int32_t* batch_idx,
                         const int32_t* input_pos, int n_tokens, float scale, void* out,
                         float* lse, int32_t* dev_err, cudaStream_t stream) {
  if (head_dim != kHeadDim || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads != 0)
    return PKV_ERR_ARG;
  const int g = num_q_heads / num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return PKV_ERR_ARG;
  if (n_tokens < 0 || !std::isfinite(scale) || !(scale > 0.f)) return PKV_ERR_ARG;
  if (n_tokens == 0) return PKV_OK;
  if (!q || !k || !v || !batch_idx || !input_pos || !out || !lse) return PKV_ERR_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(batch_idx, 4) || !aligned(input_pos, 4) ||
      !aligned(dev_err, 4))
    return PKV_ERR_ALIGN;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (major != 10 || minor != 3) return PKV_ERR_DEVICE;
  if (static_cast<long long>(((n_tokens + kBM - 1) / kBM)) * num_q_heads > INT32_MAX)
    return PKV_ERR_ARG;

  CUtensorMap qmap, kmap, vmap;
  if (!encode_packed_map(&qmap, q, num_q_heads, n_tokens) ||
      !encode_packed_map(&kmap, k, num_kv_heads, n_tokens) ||
      !encode_packed_map(&vmap, v, num_kv_heads, n_tokens))
    return PKV_ERR_ARG;

  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return PKV_ERR_DEVICE;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(prefill_tcgen05_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return PKV_ERR_CUDA;
    attr_set[dev] = true;
  }
  PrefillParams prm;
  prm.batch_idx = batch_idx;
  prm.input_pos = input_pos;
  prm.out = out;
  prm.lse = lse;
  prm.dev_err = dev_err;
  prm.n_tokens = n_tokens;
  prm.num_q_heads = num_q_heads;
  prm.group = g;
  prm.qscale = scale * 1.4426950408889634f;
  const int tiles = (n_tokens + kBM - 1) / kBM;
  const cudaError_t e = launch_kernel(prefill_tcgen05_kernel, dim3(tiles * num_q_heads),
                                      dim3(kThreads), kSmemBytes, stream, false, qmap, kmap,
                                      vmap, prm);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
