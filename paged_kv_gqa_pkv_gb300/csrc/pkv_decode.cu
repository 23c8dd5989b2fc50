// pkv_decode.cu - K2 split-KV GQA decode over the paged cache, and K3 the
// LSE merge of its partial results.
//
// Source of the computation: "qwen3_flex_inference.py", _decode_block_mask
// (causal_offset: row b attends keys kv_idx <= input_pos of its own slot) and
// attention forward (enable_gqa); zero-safe padded rows: "flex_vs_vllm.md",
// "What broke correctness and had to be dropped" (ROWS_GUARANTEED_SAFE).
// Design levers the pages found for their own kernel and that carry over:
// prescaled q (PRESCALE_QK), bulk asynchronous staging (USE_TMA), skipping
// per-block indirection for sequential pages (BLOCKS_ARE_CONTIGUOUS) and many
// warps in flight (num_warps) ("FlexKernelOptions sweep"; "flex_vs_vllm.md",
// "What each option did").
//
// Schedule (persistent, balanced): the work of a call is the ordered list of
// 16-token tiles of every (row, kv head) item. Every CTA recomputes the
// per-row tile prefix sum in shared memory; the list is cut into
// num_workers = SMs x 8 equal contiguous ranges, one per warp. A warp streams
// its range through a private ring of TMA stages (K tile, V tile and, at a
// segment start, the item's G query rows), so no barrier is shared between
// warps. Each (worker, item) segment leaves one partial (unnormalised o for
// the G heads, running max m and sum l in log2 units) in slot
// worker + item, unique because both indices grow along the list. The merge
// kernel combines an item's segments by LSE.
//
// Arithmetic per tile (CUDA cores, fp32): all G query heads of a kv head use
// one load of each K and V row.
//  * QK: lane (grp = lane/8, j = lane%8) takes token it*4 + grp and dims
//    {8j..8j+7, 64+8j..64+8j+7} of it, for 4 tokens; the 8 lanes of a group
//    finish the dot products with a reduce-scatter butterfly (xor 4, 2, 1).
//  * softmax: scores go through a per-warp shared buffer; the tile max per
//    head is a warp shuffle reduction; p = exp2(s - m) in place.
//  * PV: lane owns dims 4*lane..4*lane+3 of all G heads and reads p[t][0..G)
//    as a broadcast.
#include "pkv_launch.h"

namespace pkv {

namespace {

constexpr int kKTileBytes = kDecodeTile * kHeadDim * 2;  // one head, 16 tokens

template <int G>
struct DecodeCfg {
  static constexpr int kStages = (G >= 8) ? 2 : kDecodeStages;
  static constexpr int kQBytes = G * kHeadDim * 2;
  static constexpr int kStageStride = ((2 * kKTileBytes + kQBytes) + 127) / 128 * 128;
  static constexpr int kBarOffset = kDecodeWarps * kStages * kStageStride;
  static constexpr int kScoreOffset = kBarOffset + kDecodeWarps * kStages * 8;
  static constexpr int kLenOffset = kScoreOffset + kDecodeWarps * kDecodeTile * G * 4;
  static constexpr int kWarpSumOffset = kLenOffset;  // int[kDecodeWarps]
  static constexpr int kRowsOffset = kWarpSumOffset + kDecodeWarps * 4;
  static constexpr size_t smem_bytes(int batch) {
    // seq_len per row, then the tile prefix over rows ([batch + 1])
    return kRowsOffset + static_cast<size_t>(batch) * 4 + static_cast<size_t>(batch + 1) * 4;
  }
};

// Position of a worker inside the tile list.
struct Cursor {
  int b;      // row
  int kvh;    // kv head
  int tile;   // tile within the item
  int tiles;  // tiles of row b
};

__device__ __forceinline__ Cursor locate(const int32_t* prefix, int batch, int hkv, int64_t u) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(prefix[mid + 1]) * hkv > u) hi = mid;
    else lo = mid + 1;
  }
  Cursor c;
  c.b = lo;
  c.tiles = prefix[lo + 1] - prefix[lo];
  const int64_t r = u - static_cast<int64_t>(prefix[lo]) * hkv;
  c.kvh = static_cast<int>(r / c.tiles);
  c.tile = static_cast<int>(r % c.tiles);
  return c;
}

// Next tile; the caller guarantees one exists.
__device__ __forceinline__ void advance(Cursor& c, const int32_t* prefix, int hkv) {
  if (++c.tile < c.tiles) return;
  c.tile = 0;
  if (++c.kvh < hkv) return;
  c.kvh = 0;
  do {
    ++c.b;
    c.tiles = prefix[c.b + 1] - prefix[c.b];
  } while (c.tiles == 0);
}

// One reduce-scatter step across lanes `lane ^ M`: of 2*H partial sums, a lane
// keeps the lower H (bit M of the lane clear) or the upper H, adding its
// partner's copy of them.
template <int H, int M>
__device__ __forceinline__ void rs_step(float* v, int lane, int& idx0) {
  const bool upper = (lane & M) != 0;
#pragma unroll
  for (int i = 0; i < H; ++i) {
    const float send = upper ? v[i] : v[i + H];
    const float keep = upper ? v[i + H] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
  }
  if (upper) idx0 += H;
}

// Producer-side view of the current row's pages (warp-uniform).
struct RowPages {
  int b;            // row these describe (-1: none yet)
  int slot;         // batch_idx[b]
  int base;         // first page when contiguous
  bool contiguous;  // page_table[slot, j] == base + j for every needed block
};

__device__ __forceinline__ void load_row_pages(RowPages& rp, const DecodeParams& p, int b,
                                               int tiles, int lane) {
  rp.b = b;
  rp.slot = p.batch_idx[b];
  const int32_t* row = p.page_table + static_cast<int64_t>(rp.slot) * p.max_blocks;
  const int nblk = (tiles * kDecodeTile + p.page_size - 1) / p.page_size;
  const int base = row[0];
  bool ok = base >= 0 && base + nblk <= p.num_pages;
  for (int j0 = 0; j0 < nblk && ok; j0 += 32) {
    const int j = j0 + lane;
    const bool mine = (j >= nblk) || (row[j] == base + j);
    ok = __all_sync(0xffffffffu, mine);
  }
  rp.base = base;
  rp.contiguous = ok;
}

}  // namespace

template <int G>
__global__ void __launch_bounds__(kDecodeWarps * 32, 1)
decode_splitkv_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  using C = DecodeCfg<G>;
  constexpr int S = C::kStages;
  extern __shared__ __align__(128) uint8_t smem[];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int B = p.batch;
  const int hkv = p.num_kv_heads;

  uint8_t* stages = smem + warp * S * C::kStageStride;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset) + warp * S;
  float* s_score = reinterpret_cast<float*>(smem + C::kScoreOffset) + warp * kDecodeTile * G;
  int* s_warp_sum = reinterpret_cast<int*>(smem + C::kWarpSumOffset);
  int32_t* s_len = reinterpret_cast<int32_t*>(smem + C::kRowsOffset);
  int32_t* s_prefix = s_len + B;

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  if (tid == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  // Everything read below may be written by the previous kernel on the stream.
  pdl_wait_primary();
  pdl_launch_dependents();

  // ---- tiles per row and their exclusive prefix sum (every CTA, in smem) ----
  const int per_thread = (B + blockDim.x - 1) / blockDim.x;
  const int r0 = min(tid * per_thread, B);
  const int r1 = min(r0 + per_thread, B);
  const int max_len = p.max_blocks * p.page_size;
  int local = 0;
  for (int r = r0; r < r1; ++r) {
    const int c = p.batch_idx[r];
    const int n = p.seq_lens[r];
    int tiles = 0, err = 0;
    if (c < 0 || c >= p.max_batch) err = PKV_DEV_ERR_BAD_SLOT;
    else if (n < 0 || n > max_len) err = PKV_DEV_ERR_BAD_POS;
    else if (c != 0) tiles = (n + kDecodeTile - 1) / kDecodeTile;
    if (err && blockIdx.x == 0) set_dev_err(p.dev_err, err);
    s_len[r] = n;
    s_prefix[r] = tiles;
    local += tiles;
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp_sum[warp] = incl;
  __syncthreads();
  int run = incl - local;
  for (int w = 0; w < warp; ++w) run += s_warp_sum[w];
  for (int r = r0; r < r1; ++r) {
    const int t = s_prefix[r];
    s_prefix[r] = run;
    run += t;
  }
  if (tid == blockDim.x - 1) s_prefix[B] = run;
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int r = tid; r <= B; r += blockDim.x) p.prefix[r] = s_prefix[r];
  }

  // ---- this warp's range of the tile list ----
  const int64_t total = static_cast<int64_t>(s_prefix[B]) * hkv;
  const int worker = blockIdx.x * kDecodeWarps + warp;
  const int64_t per = (total + p.num_workers - 1) / p.num_workers;
  const int64_t u_begin = static_cast<int64_t>(worker) * per;
  const int64_t u_end = min(u_begin + per, total);
  if (u_begin >= u_end) return;
  const int count = static_cast<int>(u_end - u_begin);

  const Cursor start = locate(s_prefix, B, hkv, u_begin);
  Cursor pc = start;  // producer: next tile to stage
  Cursor cc = start;  // consumer: tile being computed
  RowPages rp;
  rp.b = -1;
  bool bail = false;

  const uint8_t* qbase = static_cast<const uint8_t*>(p.q);
  auto issue = [&](const Cursor& c, int k) {
    if (c.b != rp.b) load_row_pages(rp, p, c.b, c.tiles, lane);
    if (lane == 0) {
      const int s = k % S;
      uint8_t* st = stages + s * C::kStageStride;
      const int t0 = c.tile * kDecodeTile;
      const int blk = t0 / p.page_size;
      int page;
      if (rp.contiguous) {
        page = rp.base + blk;
      } else {
        page = p.page_table[static_cast<int64_t>(rp.slot) * p.max_blocks + blk];
        if (page < 0 || page >= p.num_pages) {
          set_dev_err(p.dev_err, PKV_DEV_ERR_BAD_PAGE);
          page = 0;  // stage a valid page; this row's result is unspecified
        }
      }
      const int row = page * p.page_size + t0 % p.page_size;
      const bool seg_start = (k == 0) || (c.tile == 0);
      mbar_arrive_expect_tx(&bars[s], 2 * kKTileBytes + (seg_start ? C::kQBytes : 0));
      tma_load_3d(st, &kmap, &bars[s], 0, c.kvh, row);
      tma_load_3d(st + kKTileBytes, &vmap, &bars[s], 0, c.kvh, row);
      if (seg_start) {
        const size_t qoff =
            (static_cast<size_t>(c.b) * p.num_q_heads + static_cast<size_t>(c.kvh) * G) *
            kHeadDim * 2;
        bulk_load(st + 2 * kKTileBytes, qbase + qoff, C::kQBytes, &bars[s]);
      }
    }
  };

  const int prologue = min(S, count);
  for (int k = 0; k < prologue; ++k) {
    issue(pc, k);
    if (k + 1 < count) advance(pc, s_prefix, hkv);
  }

  const int grp = lane >> 3;
  const int jl = lane & 7;
  const int hg = lane % G;  // head whose softmax statistics this lane keeps
  float q[G][16];
  float acc[G][4];
  float m_run = -INFINITY, l_run = 0.f;
  int n_row = 0;
  int issued = prologue;

  for (int k = 0; k < count; ++k) {
    const int s = k % S;
    if (!mbar_wait_bounded(&bars[s], (k / S) & 1)) {
      if (lane == 0) set_dev_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
      bail = true;
      break;
    }
    const uint8_t* st = stages + s * C::kStageStride;
    const bool seg_start = (k == 0) || (cc.tile == 0);
    if (seg_start) {
      const uint8_t* qs = st + 2 * kKTileBytes;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const uint4 a = *reinterpret_cast<const uint4*>(qs + g * 256 + jl * 16);
        const uint4 c = *reinterpret_cast<const uint4*>(qs + g * 256 + 128 + jl * 16);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          q[g][2 * e] = bf16lo(w[e]) * p.qscale;
          q[g][2 * e + 1] = bf16hi(w[e]) * p.qscale;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[g][e] = 0.f;
      }
      m_run = -INFINITY;
      l_run = 0.f;
      n_row = s_len[cc.b];
    }
    const int n_valid = min(kDecodeTile, n_row - cc.tile * kDecodeTile);

    // ---- QK: partial dot products over this lane's 16 dims ----
    constexpr int N = 4 * G;
    float v[N];
    const uint8_t* ks = st;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int t = it * 4 + grp;
      const uint4 a = *reinterpret_cast<const uint4*>(ks + t * 256 + jl * 16);
      const uint4 c = *reinterpret_cast<const uint4*>(ks + t * 256 + 128 + jl * 16);
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
      float kf[16];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        kf[2 * e] = bf16lo(w[e]);
        kf[2 * e + 1] = bf16hi(w[e]);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float d0 = 0.f, d1 = 0.f;
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          d0 = fmaf(q[g][e], kf[e], d0);
          d1 = fmaf(q[g][e + 1], kf[e + 1], d1);
        }
        v[it * G + g] = d0 + d1;
      }
    }
    // ---- reduce-scatter across the 8 lanes of the group ----
    int idx0 = 0;
    rs_step<N / 2, 4>(v, lane, idx0);
    rs_step<N / 4, 2>(v, lane, idx0);
    if constexpr (N / 4 >= 2) {
      rs_step<N / 8, 1>(v, lane, idx0);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
    }
    constexpr int kHeld = (N >= 8) ? N / 8 : 1;
#pragma unroll
    for (int i = 0; i < kHeld; ++i) {
      const int idx = idx0 + i;
      const int t = (idx / G) * 4 + grp;
      const int g = idx % G;
      s_score[t * G + g] = (t < n_valid) ? v[i] : -INFINITY;
    }
    __syncwarp();

    // ---- online softmax (log2 units) ----
    constexpr int kPer = (kDecodeTile * G + 31) / 32;
    constexpr int kStride = 32 / G;
    float sv[kPer];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int t = lane / G + i * kStride;
      sv[i] = (t < kDecodeTile) ? s_score[t * G + hg] : -INFINITY;
      mx = fmaxf(mx, sv[i]);
    }
#pragma unroll
    for (int m = G; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    const float m_new = fmaxf(m_run, mx);
    const float alpha = exp2f(m_run - m_new);
    float psum = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int t = lane / G + i * kStride;
      if (t < kDecodeTile) {
        const float pv = exp2f(sv[i] - m_new);
        s_score[t * G + hg] = pv;
        psum += pv;
      }
    }
    l_run = l_run * alpha + psum;
    m_run = m_new;
    __syncwarp();
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float a = __shfl_sync(0xffffffffu, alpha, g);
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[g][e] *= a;
    }

    // ---- PV over the valid tokens ----
    const uint8_t* vs = st + kKTileBytes;
#pragma unroll 4
    for (int t = 0; t < n_valid; ++t) {
      const uint2 w = *reinterpret_cast<const uint2*>(vs + t * 256 + lane * 8);
      const float v0 = bf16lo(w.x), v1 = bf16hi(w.x), v2 = bf16lo(w.y), v3 = bf16hi(w.y);
      float pg[G];
      if constexpr (G % 4 == 0) {
#pragma unroll
        for (int g = 0; g < G; g += 4) {
          const float4 p4 = *reinterpret_cast<const float4*>(s_score + t * G + g);
          pg[g] = p4.x; pg[g + 1] = p4.y; pg[g + 2] = p4.z; pg[g + 3] = p4.w;
        }
      } else {
#pragma unroll
        for (int g = 0; g < G; ++g) pg[g] = s_score[t * G + g];
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        acc[g][0] = fmaf(pg[g], v0, acc[g][0]);
        acc[g][1] = fmaf(pg[g], v1, acc[g][1]);
        acc[g][2] = fmaf(pg[g], v2, acc[g][2]);
        acc[g][3] = fmaf(pg[g], v3, acc[g][3]);
      }
    }

    // ---- segment end: leave the partial in slot worker + item ----
    const bool seg_end = (k == count - 1) || (cc.tile == cc.tiles - 1);
    if (seg_end) {
      float lt = l_run;
#pragma unroll
      for (int m = G; m < 32; m <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, m);
      const int64_t slot_id = static_cast<int64_t>(worker) + static_cast<int64_t>(cc.b) * hkv + cc.kvh;
      float* slot = p.partials + slot_id * decode_slot_floats(G);
#pragma unroll
      for (int g = 0; g < G; ++g)
        *reinterpret_cast<float4*>(slot + g * kHeadDim + lane * 4) =
            make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
      if (lane < G) {
        slot[G * kHeadDim + lane] = m_run;
        slot[G * kHeadDim + G + lane] = lt;
      }
    }
    __syncwarp();

    // ---- refill this stage with the tile S ahead ----
    if (k + S < count) {
      issue(pc, k + S);
      ++issued;
      if (k + S + 1 < count) advance(pc, s_prefix, hkv);
    }
    if (k + 1 < count) advance(cc, s_prefix, hkv);
  }

  if (bail && lane == 0) {
    // Drain copies still in flight into this warp's stages before exiting.
    for (int k = 0; k < issued; ++k) {
      const int s = k % S;
      mbar_wait_bounded(&bars[s], (k / S) & 1);
    }
  }
}

// One warp per (row, q head): lanes load the segments' (m, l) in parallel,
// the o loads of the first segments go out in the same round, and the LSE
// combination is a warp reduction.
template <int G>
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeParams p) {
  pdl_wait_primary();
  const int lane = threadIdx.x & 31;
  const int wid = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wid >= p.batch * p.num_q_heads) return;
  const int b = wid / p.num_q_heads;
  const int h = wid % p.num_q_heads;
  const int kvh = h / G;
  const int g = h % G;
  const int hkv = p.num_kv_heads;
  const int pb = p.prefix[b];
  const int tiles = p.prefix[b + 1] - pb;
  const int64_t total = static_cast<int64_t>(p.prefix[p.batch]) * hkv;
  __nv_bfloat16* out =
      static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(wid) * kHeadDim + lane * 4;
  if (tiles == 0) {
    *reinterpret_cast<uint2*>(out) = make_uint2(0u, 0u);
    if (lane == 0) p.lse[wid] = -INFINITY;
    return;
  }
  const int64_t per = (total + p.num_workers - 1) / p.num_workers;
  const int64_t u0 = static_cast<int64_t>(pb) * hkv + static_cast<int64_t>(kvh) * tiles;
  const int w0 = static_cast<int>(u0 / per);
  const int nseg = static_cast<int>((u0 + tiles - 1) / per) - w0 + 1;
  constexpr int SF = decode_slot_floats(G);
  const float* slots = p.partials + (static_cast<int64_t>(w0) + static_cast<int64_t>(b) * hkv + kvh) * SF;

  float M = -INFINITY;
  for (int s0 = 0; s0 < nseg; s0 += 32) {
    const int s = s0 + lane;
    if (s < nseg) M = fmaxf(M, slots[static_cast<int64_t>(s) * SF + G * kHeadDim + g]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < nseg; s0 += 32) {
    const int s = s0 + lane;
    float sc = 0.f;
    if (s < nseg) {
      const float* sl = slots + static_cast<int64_t>(s) * SF;
      sc = exp2f(sl[G * kHeadDim + g] - M);
      L = fmaf(sl[G * kHeadDim + G + g], sc, L);
    }
    const int n = min(32, nseg - s0);
#pragma unroll 4
    for (int j = 0; j < n; ++j) {
      const float scj = __shfl_sync(0xffffffffu, sc, j);
      const float4 ov = *reinterpret_cast<const float4*>(
          slots + static_cast<int64_t>(s0 + j) * SF + g * kHeadDim + lane * 4);
      acc.x = fmaf(ov.x, scj, acc.x);
      acc.y = fmaf(ov.y, scj, acc.y);
      acc.z = fmaf(ov.z, scj, acc.z);
      acc.w = fmaf(ov.w, scj, acc.w);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float inv = 1.f / L;
  const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 packed;
  packed.x = *reinterpret_cast<const uint32_t*>(&lo);
  packed.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(out) = packed;
  if (lane == 0) p.lse[wid] = (M + log2f(L)) * 0.69314718055994531f;
}

size_t decode_workspace_bytes(int batch, int num_kv_heads, int group, int num_workers) {
  const size_t slots = static_cast<size_t>(num_workers) + static_cast<size_t>(batch) * num_kv_heads;
  const size_t part = slots * decode_slot_floats(group) * sizeof(float);
  const size_t pre = (static_cast<size_t>(batch) + 1) * sizeof(int32_t);
  return ((part + 255) / 256) * 256 + ((pre + 255) / 256) * 256;
}

int decode_workers_for_device(int sm_count) { return sm_count * kDecodeWarps; }

template <int G>
static cudaError_t launch_decode_g(const DecodeParams& p, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, int sm_count, cudaStream_t stream) {
  using C = DecodeCfg<G>;
  const size_t smem = C::smem_bytes(p.batch);
  static_assert(C::smem_bytes(kDecodeMaxBatch) <= 232448, "decode shared memory over budget");
  // The shared-memory opt-in is set once per device, so steady-state calls
  // (and calls under stream capture) only enqueue kernels.
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(decode_splitkv_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::smem_bytes(kDecodeMaxBatch)));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  e = launch_kernel(decode_splitkv_kernel<G>, dim3(sm_count), dim3(kDecodeWarps * 32), smem,
                    stream, /*programmatic=*/true, kmap, vmap, p);
  if (e != cudaSuccess) return e;
  const int rows = p.batch * p.num_q_heads;
  return launch_kernel(decode_merge_kernel<G>, dim3((rows + 7) / 8), dim3(256), 0, stream,
                       /*programmatic=*/true, p);
}

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          int sm_count, cudaStream_t stream) {
  switch (p.num_q_heads / p.num_kv_heads) {
    case 1: return launch_decode_g<1>(p, kmap, vmap, sm_count, stream);
    case 2: return launch_decode_g<2>(p, kmap, vmap, sm_count, stream);
    case 4: return launch_decode_g<4>(p, kmap, vmap, sm_count, stream);
    case 8: return launch_decode_g<8>(p, kmap, vmap, sm_count, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
