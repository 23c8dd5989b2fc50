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
// its range through a private two-stage ring of TMA stages (K tile, V tile
// and, at a segment start, the item's G query rows), so no barrier is shared
// between warps. An item that lies inside one warp's range is normalised and
// written by that warp. Every other (worker, item) segment leaves one partial
// (unnormalised o for the G heads, running max m and sum l in log2 units) in
// slot worker + item, unique because both indices grow along the list, and
// the merge kernel combines an item's segments by LSE. When the launch
// expects long items (few rows for the machine, kCombine), the CTAs first
// combine their warps' partials of items split over more than kLongItemSegs
// warps, so the merge reads one segment per CTA for those.
//
// Arithmetic per tile: all G query heads of a kv head use one load of each K
// and V row. The two products are small dense contractions and run as
// warp-level bf16 MMAs (m16n8k16, fp32 accumulate) in transposed form, so the
// 16 tokens and the head dims fill the MMA's 16 rows and the G <= 8 heads its
// 8 columns: S^T[16 x 8] = K Q^T over 8 k-steps, then O^T[128 x 8] += V^T P^T
// as 8 m-tiles of one k-step (16 MMAs a tile; with the heads as rows it would
// be 32, three quarters padding at G = 4). A warp first copies the tile's K
// and V fragments out of shared memory (ldmatrix on 128-byte-swizzled TMA
// boxes, conflict-free) and hands the stage back to TMA before any
// arithmetic. The online softmax stays in fp32 registers: per-head max over
// tokens is a 3-step shuffle reduction, exp2 with the scale folded in, O
// rescaled only when some head's max moved. P^T leaves the S^T accumulators
// as bf16 pairs and one register transpose (movmatrix) per 8 x 8 block makes
// it the B operand of the PV product, so the softmax never touches shared
// memory. Keys past a row's length are masked to -inf in S and their V rows
// are zeroed in shared memory before the fragments are read (stale slots of a
// page may hold any bits, NaN included).
#include <atomic>

#include "pkv_launch.h"

namespace pkv {

namespace {

constexpr int kKTileBytes = kDecodeTile * kHeadDim * 2;  // one head, 16 tokens (4 KB)

// The K/V stream of a call is read once: its TMA loads carry an L2
// evict-first policy, so the lines they bring in are the first replaced and
// the partials, q rows and page-table rows the call reuses stay in L2
// (decode call 37.70 -> 37.10 us on the B = 64 Qwen3-4B step).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_4d_evict_first(void* dst, const CUtensorMap* map,
                                                        uint64_t* bar, int x, int y, int z, int w,
                                                        uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w),
      "l"(pol)
      : "memory");
}

template <int G>
struct DecodeCfg {
  static constexpr int kStages = kDecodeStages;
  static constexpr int kQBytes = G * kHeadDim * 2;
  // stage: K tile (two 2 KB swizzled halves), V tile (same), q rows
  static constexpr int kOffV = kKTileBytes;
  static constexpr int kOffQ = 2 * kKTileBytes;
  static constexpr int kStageStride = ((2 * kKTileBytes + kQBytes) + 1023) / 1024 * 1024;
  static constexpr int kBarOffset = kDecodeWarps * kStages * kStageStride;
  static constexpr int kWarpSumOffset = kBarOffset + kDecodeWarps * kStages * 8;
  static constexpr int kRowsOffset = kWarpSumOffset + kDecodeWarps * 4;
  static constexpr size_t smem_bytes(int batch, bool list = false) {
    // seq_len and slot per row, the tile prefix over rows ([batch + 1]), the
    // row's token in list mode, and 1 KB to round the dynamic base up to the
    // swizzle-atom alignment
    return 1024 + kRowsOffset + static_cast<size_t>(batch) * (list ? 12 : 8) +
           static_cast<size_t>(batch + 1) * 4;
  }
};

constexpr int kHalfBytes = kDecodeTile * 128;  // 16 rows x 64 dims (bf16) TMA box

// Byte offset of 16-byte chunk `chunk` (0..15, eight dims each) of row `row`
// inside a [16 rows x 128 dims] tile stored as two 128-byte-swizzled halves.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * kHalfBytes + row * 128 +
                               (((chunk & 7) ^ (row & 7)) << 4));
}

// Slot c, keys attended n and token t of row r: the call's row r, or in
// list mode (kList) the packed token t = row_token[r], which attends
// input_pos[t] + 1 keys (a negative position counts as out of range).
template <bool kList>
__device__ __forceinline__ void row_input(const DecodeParams& p, int r, int& c, int& n, int& t) {
  if constexpr (kList) {
    t = p.row_token[r];
    c = p.batch_idx[t];
    const int pos = p.input_pos[t];
    n = pos < 0 ? -1 : pos + 1;
  } else {
    t = r;
    c = p.batch_idx[r];
    n = p.seq_lens[r];
  }
}

// Rows of the call: the batch, or in list mode the device-side count.
template <bool kList>
__device__ __forceinline__ int call_rows(const DecodeParams& p) {
  if constexpr (kList) return min(max(*p.row_count, 0), p.batch);
  return p.batch;
}

// Tiles of row r and the device error its entries raise (0 if none). Both
// kernels apply this one rule, so the merge can rebuild the split-KV pass's
// schedule from the call's inputs alone.
template <bool kList>
__device__ __forceinline__ int row_tiles(const DecodeParams& p, int r, int* err) {
  int c, n, t;
  row_input<kList>(p, r, c, n, t);
  *err = 0;
  if (c < 0 || c >= p.max_batch) *err = PKV_DEV_ERR_BAD_SLOT;
  else if (n < 0 || n > p.max_blocks * p.page_size) *err = PKV_DEV_ERR_BAD_POS;
  else if (c != 0) return (n + kDecodeTile - 1) / kDecodeTile;
  return 0;
}

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

// Fused append: the new token of item (b, kvh), at position seq_lens[b] - 1,
// copied from k_new/v_new into the pools (lanes 0-15 a K chunk of 16 bytes,
// lanes 16-31 a V chunk). Only the warp that reads the item's last tile does
// this, before its own TMA read of that tile.
// Split in two so that a warp can issue the loads of several items before
// their stores (k_new/v_new may be host memory, a link round trip away).
__device__ __forceinline__ uint4 append_load(const DecodeParams& p, int b, int kvh, int lane) {
  const int64_t src = (static_cast<int64_t>(b) * p.num_kv_heads + kvh) * kHeadDim + (lane & 15) * 8;
  return *reinterpret_cast<const uint4*>(
      static_cast<const __nv_bfloat16*>(lane < 16 ? p.k_new : p.v_new) + src);
}

__device__ __forceinline__ void append_store(const DecodeParams& p, const int32_t* s_slot,
                                             const int32_t* s_len, int b, int kvh, int lane,
                                             const uint4 val) {
  const int n = s_len[b];
  const int pos = n - 1;
  const int hkv = p.num_kv_heads;
  const int page = p.page_table[static_cast<int64_t>(s_slot[b]) * p.max_blocks + pos / p.page_size];
  if (page < 0 || page >= p.num_pages) {
    if (lane == 0) set_dev_err(p.dev_err, PKV_DEV_ERR_BAD_PAGE);
    return;
  }
  const int64_t row = static_cast<int64_t>(page) * p.page_size + pos % p.page_size;
  const int64_t dst = (row * hkv + kvh) * kHeadDim + (lane & 15) * 8;
  *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(lane < 16 ? p.k_pool : p.v_pool) + dst) =
      val;
}

// Producer-side view of the current row's pages (warp-uniform).
struct RowPages {
  int b;            // row these describe (-1: none yet)
  int slot;         // batch_idx[b]
  int base;         // first page when contiguous
  bool contiguous;  // page_table[slot, j] == base + j for every needed block
};

__device__ __forceinline__ void load_row_pages(RowPages& rp, const DecodeParams& p,
                                               const int32_t* s_slot, int b, int tiles,
                                               int lane) {
  rp.b = b;
  rp.slot = s_slot[b];
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

// An item split over more than this many warps ("long": few rows, many
// keys) has the partials of each CTA combined inside the CTA, so the merge
// kernel sees one segment per CTA instead of one per warp.
constexpr int kLongItemSegs = 24;

// Combines the k <= 8 partials that consecutive warps wa .. wa+k-1 of one CTA
// left for item (b, kvh) (slots wa + item ...), all G heads at once, by LSE in
// log2 units: lanes take segments for (m, l) and four head dims each for o.
// With final_out the item is complete (it lies inside the CTA): out and lse
// are written; otherwise the merged partial replaces the first slot's.
template <int G>
__device__ __forceinline__ void combine_segments(const DecodeParams& p, int b, int kvh, int wa,
                                                 int k, bool final_out, int lane) {
  constexpr int SF = decode_slot_floats(G);
  const int hkv = p.num_kv_heads;
  float* base = p.partials + (static_cast<int64_t>(wa) + static_cast<int64_t>(b) * hkv + kvh) * SF;
  float M[G], L[G], sc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float m = -INFINITY, l = 0.f;
    if (lane < k) {
      m = __ldcg(base + static_cast<int64_t>(lane) * SF + G * kHeadDim + h);
      l = __ldcg(base + static_cast<int64_t>(lane) * SF + G * kHeadDim + G + h);
    }
    float mx = m;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mx = __shfl_sync(0xffffffffu, mx, 0);
    sc[h] = lane < k ? exp2f(m - mx) : 0.f;
    float ls = l * sc[h];
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    M[h] = mx;
    L[h] = __shfl_sync(0xffffffffu, ls, 0);
  }
  float4 acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < kDecodeWarps; ++j) {
    if (j < k) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float s = __shfl_sync(0xffffffffu, sc[h], j);
        const float4 ov = __ldcg(reinterpret_cast<const float4*>(
            base + static_cast<int64_t>(j) * SF + h * kHeadDim + lane * 4));
        acc[h].x = fmaf(ov.x, s, acc[h].x);
        acc[h].y = fmaf(ov.y, s, acc[h].y);
        acc[h].z = fmaf(ov.z, s, acc[h].z);
        acc[h].w = fmaf(ov.w, s, acc[h].w);
      }
    }
  }
  if (final_out) {
    const int64_t head0 = static_cast<int64_t>(b) * p.num_q_heads + kvh * G;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float inv = 1.f / L[h];
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[h].x * inv, acc[h].y * inv);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[h].z * inv, acc[h].w * inv);
      uint2 packed;
      packed.x = *reinterpret_cast<const uint32_t*>(&lo);
      packed.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + (head0 + h) * kHeadDim +
                                lane * 4) = packed;
      if (lane == h) p.lse[head0 + h] = (M[h] + log2f(L[h])) * 0.69314718055994531f;
    }
  } else {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      *reinterpret_cast<float4*>(base + h * kHeadDim + lane * 4) = acc[h];
      if (lane == h) {
        base[G * kHeadDim + h] = M[h];
        base[G * kHeadDim + G + h] = L[h];
      }
    }
  }
}

}  // namespace

// kCombine: the launch expects long items (few rows for the machine) and the
// CTAs combine their partials of those; without it the code below it is
// compiled out and every item goes to the merge kernel one segment per warp.
// kHostQ: q is in mapped host memory (read by cp.async); device-resident q
// takes the bulk copy, and its instantiation carries no host-memory path
// (a smaller loop: decode call ~0.15 us and fused step ~0.3 us faster).
template <int G, bool kCombine, bool kList, bool kHostQ>
__global__ void __launch_bounds__(kDecodeWarps * 32, 1)
decode_splitkv_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  using C = DecodeCfg<G>;
  constexpr int S = C::kStages;
  static_assert(G <= 8, "GQA group must fit the MMA's 16 rows with the q rows of one head group");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int B = call_rows<kList>(p);
  const int hkv = p.num_kv_heads;

  uint8_t* stages = smem + warp * S * C::kStageStride;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset) + warp * S;
  int* s_warp_sum = reinterpret_cast<int*>(smem + C::kWarpSumOffset);
  int32_t* s_len = reinterpret_cast<int32_t*>(smem + C::kRowsOffset);
  int32_t* s_slot = s_len + B;
  int32_t* s_prefix = s_slot + B;
  int32_t* s_tok = s_prefix + B + 1;  // list mode: token of each row

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  if (tid == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  // Programmatic dependent launch: this prologue (row lengths, slots, the tile
  // prefix, the first page-table row) reads only arrays that no kernel of this
  // library writes, so it overlaps the previous kernel on the stream; the
  // pools, q and the workspace are touched only after pdl_wait_primary().
  pdl_launch_dependents();

  // ---- tiles per row and their exclusive prefix sum (every CTA, in smem) ----
  const int per_thread = (B + blockDim.x - 1) / blockDim.x;
  const int r0 = min(tid * per_thread, B);
  const int r1 = min(r0 + per_thread, B);
  int local = 0;
  for (int r = r0; r < r1; ++r) {
    int err, c, n, t;
    const int tiles = row_tiles<kList>(p, r, &err);
    if (err && blockIdx.x == 0) set_dev_err(p.dev_err, err);
    row_input<kList>(p, r, c, n, t);
    s_len[r] = n;
    s_slot[r] = c;
    if constexpr (kList) s_tok[r] = t;
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

  // ---- this warp's range of the tile list ----
  const int64_t total = static_cast<int64_t>(s_prefix[B]) * hkv;
  const int worker = blockIdx.x * kDecodeWarps + warp;
  const int64_t per = (total + p.num_workers - 1) / p.num_workers;
  const int64_t u_begin = static_cast<int64_t>(worker) * per;
  const int64_t u_end = min(u_begin + per, total);
  if constexpr (!kCombine) {
    if (u_begin >= u_end) return;
  }
  if (u_begin < u_end) {
  const int count = static_cast<int>(u_end - u_begin);

  const Cursor start = locate(s_prefix, B, hkv, u_begin);
  Cursor pc = start;  // producer: next tile to stage
  Cursor cc = start;  // consumer: tile being computed
  RowPages rp;
  rp.b = -1;
  bool bail = false;

  const uint8_t* qbase = static_cast<const uint8_t*>(p.q);
  const uint64_t kv_policy = l2_evict_first_policy();
  auto issue = [&](const Cursor& c, int k) {
    if (c.b != rp.b) load_row_pages(rp, p, s_slot, c.b, c.tiles, lane);
    const bool seg_start = (k == 0) || (c.tile == 0);
    if (seg_start && kHostQ) {
      // q in mapped host memory: every lane copies its 16-byte pieces of the
      // item's G rows with cp.async and counts them on the stage barrier
      // before lane 0 arms it for the K/V bytes, so the stage completes only
      // once q has landed too
      const int s = k % S;
      uint8_t* st = stages + s * C::kStageStride;
      const int qrow = kList ? s_tok[c.b] : c.b;
      const uint8_t* src =
          qbase + (static_cast<size_t>(qrow) * p.num_q_heads + static_cast<size_t>(c.kvh) * G) *
                      kHeadDim * 2;
      for (int o = lane * 16; o < C::kQBytes; o += 32 * 16) cp_async16(st + C::kOffQ + o, src + o);
      cp_async_mbar_arrive(&bars[s]);
      __syncwarp();
    }
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
      const bool q_bulk = seg_start && !kHostQ;
      mbar_arrive_expect_tx(&bars[s], 2 * kKTileBytes + (q_bulk ? C::kQBytes : 0));
      tma_load_4d_evict_first(st, &kmap, &bars[s], 0, row, 0, c.kvh, kv_policy);
      tma_load_4d_evict_first(st + C::kOffV, &vmap, &bars[s], 0, row, 0, c.kvh, kv_policy);
      if (q_bulk) {
        const int qrow = kList ? s_tok[c.b] : c.b;
        const size_t qoff =
            (static_cast<size_t>(qrow) * p.num_q_heads + static_cast<size_t>(c.kvh) * G) *
            kHeadDim * 2;
        bulk_load(st + C::kOffQ, qbase + qoff, C::kQBytes, &bars[s]);
      }
    }
  };

  load_row_pages(rp, p, s_slot, start.b, start.tiles, lane);
  pdl_wait_primary();
  // Fused append: this warp owns the new tokens of the items whose last tile
  // lies in its range, and they must reach the pools before its TMA read of
  // that tile. The loads of the first four go out now; their stores follow
  // once the first stages are issued, or before a stage that reads one of
  // those tiles, so streaming does not start a round trip (to the host, when
  // k_new/v_new live there) late. Items past the first four (their last
  // tiles lie past the first stages) are appended four at a time after that.
  Cursor ac = start;
  int64_t au = u_begin;
  bool amore = p.k_new != nullptr;
  int nb = 0;
  int ib[4], ik[4];
  int64_t ul[4];  // tile-list index of each pending item's last tile
  uint4 val[4];
  // the next up to four owned items from (ac, au)
  auto gather = [&]() {
    nb = 0;
    while (amore && nb < 4) {
      const int64_t u_last = au + (ac.tiles - 1 - ac.tile);
      if (u_last >= u_end) {
        amore = false;
        break;
      }
      ib[nb] = ac.b;
      ik[nb] = ac.kvh;
      ul[nb] = u_last;
      ++nb;
      au = u_last + 1;
      if (au >= u_end) {
        amore = false;
        break;
      }
      ac.tile = ac.tiles - 1;
      advance(ac, s_prefix, hkv);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < nb) val[e] = append_load(p, ib[e], ik[e], lane);
  };
  auto store_pending = [&]() {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < nb) append_store(p, s_slot, s_len, ib[e], ik[e], lane, val[e]);
    nb = 0;
  };
  bool appended = p.k_new == nullptr;
  auto finish_append = [&]() {
    if (appended) return;
    store_pending();
    while (amore) {
      gather();
      store_pending();
    }
    fence_proxy_async_global();
    __syncwarp();
    appended = true;
  };
  if (!appended) gather();
  const int prologue = min(S, count);
  for (int k = 0; k < prologue; ++k) {
    bool reads_pending = false;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < nb && ul[e] == u_begin + k) reads_pending = true;
    if (reads_pending) finish_append();
    issue(pc, k);
    if (k + 1 < count) advance(pc, s_prefix, hkv);
  }
  finish_append();

  // MMA fragment coordinates: g = this lane's accumulator row (a token in
  // S^T, a head dim in O^T), t = its column pair (query heads 2t, 2t+1).
  const int g = lane >> 2;
  const int t = lane & 3;
  const bool live_row = g < G;        // this lane loads q row g into the B fragments
  const bool live_h0 = 2 * t < G;     // heads this lane's columns hold
  const bool live_h1 = 2 * t + 1 < G;
  uint32_t qb[8][2];     // B fragments of Q^T (columns 0..G-1; columns >= G are zero)
  float acc[8][4];       // O^T accumulators, m-tile = 16 head dims
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  int n_row = 0;
  int seg_t0 = 0;  // first tile of the open segment
  int issued = prologue;
  // ldmatrix row addresses (per lane) within a K or V tile
  const int mtx = lane >> 3;       // which of the four 8x8 matrices this lane addresses
  const int mrow = lane & 7;

  for (int k = 0; k < count; ++k) {
    const int s = k % S;
    if (!mbar_wait_bounded(&bars[s], (k / S) & 1)) {
      if (lane == 0) set_dev_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
      bail = true;
      break;
    }
    uint8_t* st = stages + s * C::kStageStride;
    const uint32_t sK = smem_u32(st);
    const uint32_t sV = smem_u32(st + C::kOffV);
    const bool seg_start = (k == 0) || (cc.tile == 0);
    if (seg_start) {
      const uint32_t* qs = reinterpret_cast<const uint32_t*>(st + C::kOffQ);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qb[kk][0] = live_row ? qs[g * 64 + kk * 8 + t] : 0u;
        qb[kk][1] = live_row ? qs[g * 64 + kk * 8 + 4 + t] : 0u;
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
      m_run[0] = m_run[1] = -INFINITY;
      l_run[0] = l_run[1] = 0.f;
      n_row = s_len[cc.b];
      seg_t0 = cc.tile;
    }
    const int n_valid = min(kDecodeTile, n_row - cc.tile * kDecodeTile);
    if (n_valid < kDecodeTile) {
      // stale slots past the row's end may hold any bits (NaN included):
      // zero their V rows before they are read (their scores are masked)
      for (int r = n_valid; r < kDecodeTile; ++r) {
        uint4* vrow = reinterpret_cast<uint4*>(st + C::kOffV);
        if (lane < 16) vrow[(swz(r, lane)) >> 4] = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }

    // ---- the tile's K and V fragments into registers; the stage goes back
    // to TMA before any arithmetic, so all S stages stay in flight ----
    uint32_t kf[8][4], vf[8][4];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)  // A = K: (tokens 0-7 | 8-15) x (dims 16kk..+7 | +8..+15)
      ldsm_x4(sK + swz((mtx & 1) * 8 + mrow, 2 * kk + (mtx >> 1)), kf[kk][0], kf[kk][1],
              kf[kk][2], kf[kk][3]);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)  // A = V^T: (dims 16mt..+7 | +8..+15) x (tokens 0-7 | 8-15)
      ldsm_x4_trans(sV + swz((mtx >> 1) * 8 + mrow, 2 * mt + (mtx & 1)), vf[mt][0], vf[mt][1],
                    vf[mt][2], vf[mt][3]);
    // these shared-memory reads (and the zeroing) come before the refill's
    // async-proxy writes
    fence_proxy_async_smem();
    __syncwarp();
    if (k + S < count) {
      issue(pc, k + S);
      ++issued;
      if (k + S + 1 < count) advance(pc, s_prefix, hkv);
    }

    // ---- S^T = K Q^T: 16 tokens x 8 head columns, 8 k-steps of 16 dims; even
    // and odd k-steps accumulate separately to halve the dependent MMA chain ----
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    float sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; kk += 2) {
      mma_16816(sc, kf[kk][0], kf[kk][1], kf[kk][2], kf[kk][3], qb[kk][0], qb[kk][1]);
      mma_16816(sd, kf[kk + 1][0], kf[kk + 1][1], kf[kk + 1][2], kf[kk + 1][3], qb[kk + 1][0],
                qb[kk + 1][1]);
    }
    // ---- online softmax (log2 units): x[0..1] token g, x[2..3] token g + 8;
    // x[0], x[2] head 2t and x[1], x[3] head 2t + 1 ----
    float x[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] = (sc[e] + sd[e]) * p.qscale;
    if (g >= n_valid) x[0] = x[1] = -INFINITY;
    if (g + 8 >= n_valid) x[2] = x[3] = -INFINITY;
    float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
    const float alpha0 = exp2f(m_run[0] - mn0);  // 0 on the first tile
    const float alpha1 = exp2f(m_run[1] - mn1);
    const float pe0 = exp2f(x[0] - mn0), pe1 = exp2f(x[1] - mn1);
    const float pe2 = exp2f(x[2] - mn0), pe3 = exp2f(x[3] - mn1);
    l_run[0] = l_run[0] * alpha0 + (pe0 + pe2);
    l_run[1] = l_run[1] * alpha1 + (pe1 + pe3);
    m_run[0] = mn0;
    m_run[1] = mn1;
    if (__any_sync(0xffffffffu, alpha0 != 1.f || alpha1 != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        acc[mt][0] *= alpha0;
        acc[mt][1] *= alpha1;
        acc[mt][2] *= alpha0;
        acc[mt][3] *= alpha1;
      }
    }
    // P^T as the B operand: the S^T accumulator holds P^T[token][head]; a
    // register transpose of each 8 x 8 block gives P[head][token] pairs
    const uint32_t pb0 = movmatrix_trans(pack_bf16x2(pe0, pe1));  // tokens 0-7
    const uint32_t pb1 = movmatrix_trans(pack_bf16x2(pe2, pe3));  // tokens 8-15

    // ---- O^T += V^T P^T: 8 m-tiles of 16 dims, one k-step of 16 tokens ----
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
      mma_16816(acc[mt], vf[mt][0], vf[mt][1], vf[mt][2], vf[mt][3], pb0, pb1);

    // ---- segment end: leave the partial in slot worker + item ----
    const bool seg_end = (k == count - 1) || (cc.tile == cc.tiles - 1);
    if (seg_end) {
      float lt0 = l_run[0], lt1 = l_run[1];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        lt0 += __shfl_xor_sync(0xffffffffu, lt0, o);
        lt1 += __shfl_xor_sync(0xffffffffu, lt1, o);
      }
      if (seg_t0 == 0 && cc.tile == cc.tiles - 1) {
        // the item lies in this segment alone: normalise and write it out
        // here (the merge skips items of one segment)
        const float inv0 = 1.f / lt0, inv1 = 1.f / lt1;
        const int orow = kList ? s_tok[cc.b] : cc.b;
        const int64_t head0 = static_cast<int64_t>(orow) * p.num_q_heads + cc.kvh * G + 2 * t;
        __nv_bfloat16* o0 = static_cast<__nv_bfloat16*>(p.out) + head0 * kHeadDim + g;
        __nv_bfloat16* o1 = o0 + kHeadDim;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          if (live_h0) {
            o0[16 * mt] = __float2bfloat16_rn(acc[mt][0] * inv0);
            o0[16 * mt + 8] = __float2bfloat16_rn(acc[mt][2] * inv0);
          }
          if (live_h1) {
            o1[16 * mt] = __float2bfloat16_rn(acc[mt][1] * inv1);
            o1[16 * mt + 8] = __float2bfloat16_rn(acc[mt][3] * inv1);
          }
        }
        if (g == 0) {
          if (live_h0) p.lse[head0] = (m_run[0] + log2f(lt0)) * 0.69314718055994531f;
          if (live_h1) p.lse[head0 + 1] = (m_run[1] + log2f(lt1)) * 0.69314718055994531f;
        }
      } else {
        // leave the partial in slot worker + item
        const int64_t slot_id =
            static_cast<int64_t>(worker) + static_cast<int64_t>(cc.b) * hkv + cc.kvh;
        float* slot = p.partials + slot_id * decode_slot_floats(G);
        float* o0 = slot + (2 * t) * kHeadDim + g;
        float* o1 = o0 + kHeadDim;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          if (live_h0) {
            o0[16 * mt] = acc[mt][0];
            o0[16 * mt + 8] = acc[mt][2];
          }
          if (live_h1) {
            o1[16 * mt] = acc[mt][1];
            o1[16 * mt + 8] = acc[mt][3];
          }
        }
        if (g == 0) {
          if (live_h0) {
            slot[G * kHeadDim + 2 * t] = m_run[0];
            slot[G * kHeadDim + G + 2 * t] = lt0;
          }
          if (live_h1) {
            slot[G * kHeadDim + 2 * t + 1] = m_run[1];
            slot[G * kHeadDim + G + 2 * t + 1] = lt1;
          }
        }
      }
    }
    __syncwarp();

    if (k + 1 < count) advance(cc, s_prefix, hkv);
  }

  if (bail && lane == 0) {
    // Drain copies still in flight into this warp's stages before exiting.
    for (int k = 0; k < issued; ++k) {
      const int s = k % S;
      mbar_wait_bounded(&bars[s], (k / S) & 1);
    }
  }
  }  // this warp's range

  // ---- long items (split over more than kLongItemSegs warps) that two or
  // more warps of this CTA share are combined here into one partial, in the
  // slot of this CTA's first warp on the item. A long item always crosses
  // CTAs, so the merge kernel finishes it from one segment per CTA. Every
  // warp walks the CTA's items alike, so the barrier is taken CTA-uniformly
  // and only by CTAs that hold such an item.
  if constexpr (kCombine) {
    const int64_t span = static_cast<int64_t>(kDecodeWarps) * per;
    const int64_t U0 = static_cast<int64_t>(blockIdx.x) * span;
    const int64_t U1 = min(U0 + span, total);
    const int wlo = blockIdx.x * kDecodeWarps;
    const int whi = wlo + kDecodeWarps - 1;
    // visits the items overlapping this CTA's tiles; f(cursor, w0, w1, wa, wb)
    auto for_items = [&](auto&& f) {
      if (U0 >= U1) return;
      Cursor c = locate(s_prefix, B, hkv, U0);
      int64_t u_s = U0 - c.tile;  // the item's first tile
      while (true) {
        const int64_t u_e = u_s + c.tiles - 1;
        const int w0 = static_cast<int>(u_s / per);
        const int w1 = static_cast<int>(u_e / per);
        f(c, w0, w1, max(w0, wlo), min(w1, whi));
        if (u_e + 1 >= U1) break;
        c.tile = c.tiles - 1;
        advance(c, s_prefix, hkv);
        u_s = u_e + 1;
      }
    };
    // An item of t tiles spans at most (t - 1) / per + 2 warps: with no row
    // longer than (kLongItemSegs - 2) * per tiles there is nothing to combine
    // and the walk below is skipped (the common case).
    int longest = 0;
    for (int r = lane; r < B; r += 32) longest = max(longest, s_prefix[r + 1] - s_prefix[r]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) longest = max(longest, __shfl_xor_sync(0xffffffffu, longest, o));
    bool any = false;
    if (static_cast<int64_t>(longest) > static_cast<int64_t>(kLongItemSegs - 2) * per) {
      for_items([&](const Cursor&, int w0, int w1, int wa, int wb) {
        if (w1 - w0 + 1 > kLongItemSegs && wb > wa) any = true;
      });
    }
    if (any) {
      __syncthreads();    // every warp's partials are written
      pdl_wait_primary();  // idle warps skipped the wait above
      int q = 0;
      for_items([&](const Cursor& c, int w0, int w1, int wa, int wb) {
        if (w1 - w0 + 1 > kLongItemSegs && wb > wa) {
          if (q % kDecodeWarps == warp)
            combine_segments<G>(p, c.b, c.kvh, wa, wb - wa + 1, /*final_out=*/false, lane);
          ++q;
        }
      });
    }
  }
}

// One warp per (row, q head). Before waiting on the split-KV grid, the CTA
// rebuilds that grid's schedule from the call's inputs (each row's tile count
// and their prefix, one pass over the rows shared by the CTA's 256 threads),
// so after the wait only the partials are read: for items of up to kFast
// segments, (m, l) and all o rows go out in one round of loads. kFast is 8,
// 16 when long items were combined per CTA (kByCta), and 32 (kWide) for
// launches with few items for the workers, whose items have many segments;
// kWide keeps 32 o rows in registers, so it is a separate instantiation.
template <int G, bool kByCta, bool kList, bool kWide>
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeParams p) {
  constexpr int kFast = kWide ? 32 : (kByCta ? 16 : 8);
  __shared__ int32_t s_prefix[kDecodeMaxBatch + 1];
  __shared__ int32_t s_warp_sum[8];
  // The next launch may start its prologue now; it touches the workspace
  // only after this grid completes.
  pdl_launch_dependents();
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int wid = blockIdx.x * 8 + (tid >> 5);
  const int B = call_rows<kList>(p);  // at most kDecodeMaxBatch per launch
  {
    const int per_thread = (B + 255) / 256;
    const int r0 = min(tid * per_thread, B);
    const int r1 = min(r0 + per_thread, B);
    int local = 0;
    for (int r = r0; r < r1; ++r) {
      int err;
      const int t = row_tiles<kList>(p, r, &err);
      s_prefix[r] = t;
      local += t;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp_sum[tid >> 5] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < (tid >> 5); ++w) run += s_warp_sum[w];
    for (int r = r0; r < r1; ++r) {
      const int t = s_prefix[r];
      s_prefix[r] = run;
      run += t;
    }
    if (tid == 255) s_prefix[B] = run;
    __syncthreads();
  }
  const bool active = wid < B * p.num_q_heads;
  const int b = active ? wid / p.num_q_heads : 0;
  const int h = wid % p.num_q_heads;
  const int kvh = h / G;
  const int g = h % G;
  const int hkv = p.num_kv_heads;
  const int before = active ? s_prefix[b] : 0;
  const int tiles = active ? s_prefix[b + 1] - before : 0;
  const int total = s_prefix[B];
  pdl_wait_primary();
  if (!active) return;
  // output row of (b, h): wid itself, or in list mode that of b's token
  const int64_t oid =
      kList ? static_cast<int64_t>(p.row_token[b]) * p.num_q_heads + h : static_cast<int64_t>(wid);
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + oid * kHeadDim + lane * 4;
  if (tiles == 0) {
    *reinterpret_cast<uint2*>(out) = make_uint2(0u, 0u);
    if (lane == 0) p.lse[oid] = -INFINITY;
    return;
  }
  const int64_t per = (static_cast<int64_t>(total) * hkv + p.num_workers - 1) / p.num_workers;
  const int64_t u0 = static_cast<int64_t>(before) * hkv + static_cast<int64_t>(kvh) * tiles;
  const int w0 = static_cast<int>(u0 / per);
  const int w1 = static_cast<int>((u0 + tiles - 1) / per);
  if (w0 == w1) return;  // one warp: written by the split-KV pass
  // a long item was combined per CTA by the split-KV pass: one segment per
  // CTA, in the slot of that CTA's first warp on it; else one per warp
  const bool by_cta = kByCta && w1 - w0 + 1 > kLongItemSegs;
  const int c0 = w0 / kDecodeWarps;
  const int nseg = by_cta ? w1 / kDecodeWarps - c0 + 1 : w1 - w0 + 1;
  constexpr int SF = decode_slot_floats(G);
  const float* item_slots = p.partials + (static_cast<int64_t>(b) * hkv + kvh) * SF;
  auto seg = [&](int s) -> const float* {
    const int w = by_cta ? (s == 0 ? w0 : (c0 + s) * kDecodeWarps) : w0 + s;
    return item_slots + static_cast<int64_t>(w) * SF;
  };

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float M, L = 0.f;
  if (nseg <= kFast) {
    float ms = -INFINITY, ls = 0.f;
    if (lane < nseg) {
      ms = __ldcg(seg(lane) + G * kHeadDim + g);
      ls = __ldcg(seg(lane) + G * kHeadDim + G + g);
    }
    float4 ov[kFast];
#pragma unroll
    for (int j = 0; j < kFast; ++j)
      if (j < nseg)
        ov[j] = __ldcg(reinterpret_cast<const float4*>(seg(j) +
                                                       g * kHeadDim + lane * 4));
    M = ms;
#pragma unroll
    for (int o = kFast / 2; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    M = __shfl_sync(0xffffffffu, M, 0);
    const float sc = (lane < nseg) ? exp2f(ms - M) : 0.f;
    L = ls * sc;
#pragma unroll
    for (int j = 0; j < kFast; ++j) {
      const float scj = __shfl_sync(0xffffffffu, sc, j);
      if (j < nseg) {
        acc.x = fmaf(ov[j].x, scj, acc.x);
        acc.y = fmaf(ov[j].y, scj, acc.y);
        acc.z = fmaf(ov[j].z, scj, acc.z);
        acc.w = fmaf(ov[j].w, scj, acc.w);
      }
    }
  } else {
    M = -INFINITY;
    for (int s0 = 0; s0 < nseg; s0 += 32) {
      const int s = s0 + lane;
      if (s < nseg) M = fmaxf(M, __ldcg(seg(s) + G * kHeadDim + g));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    for (int s0 = 0; s0 < nseg; s0 += 32) {
      const int s = s0 + lane;
      float sc = 0.f;
      if (s < nseg) {
        const float* sl = seg(s);
        sc = exp2f(__ldcg(sl + G * kHeadDim + g) - M);
        L = fmaf(__ldcg(sl + G * kHeadDim + G + g), sc, L);
      }
      const int n = min(32, nseg - s0);
#pragma unroll 4
      for (int j = 0; j < n; ++j) {
        const float scj = __shfl_sync(0xffffffffu, sc, j);
        const float4 ov = __ldcg(reinterpret_cast<const float4*>(
            seg(s0 + j) + g * kHeadDim + lane * 4));
        acc.x = fmaf(ov.x, scj, acc.x);
        acc.y = fmaf(ov.y, scj, acc.y);
        acc.z = fmaf(ov.z, scj, acc.z);
        acc.w = fmaf(ov.w, scj, acc.w);
      }
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
  if (lane == 0) p.lse[oid] = (M + log2f(L)) * 0.69314718055994531f;
}

size_t decode_workspace_bytes(int batch, int num_kv_heads, int group, int num_workers) {
  const size_t slots = static_cast<size_t>(num_workers) + static_cast<size_t>(batch) * num_kv_heads;
  const size_t part = slots * decode_slot_floats(group) * sizeof(float);
  return ((part + 255) / 256) * 256;
}

int decode_workers_for_device(int sm_count) { return sm_count * kDecodeWarps; }

template <int G, bool kCombine, bool kList, bool kHostQ>
static cudaError_t launch_decode_gc(const DecodeParams& p, const CUtensorMap& kmap,
                                    const CUtensorMap& vmap, int sm_count, cudaStream_t stream) {
  using C = DecodeCfg<G>;
  const size_t smem = C::smem_bytes(p.batch, kList);
  static_assert(C::smem_bytes(kDecodeMaxBatch, true) <= 232448, "decode shared memory over budget");
  // The shared-memory opt-in is set once per device, so steady-state calls
  // (and calls under stream capture) only enqueue kernels.
  static std::atomic<bool> attr_set[64] = {};  // per device; host threads may race to set it
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(decode_splitkv_kernel<G, kCombine, kList, kHostQ>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::smem_bytes(kDecodeMaxBatch, kList)));
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  e = launch_kernel(decode_splitkv_kernel<G, kCombine, kList, kHostQ>, dim3(sm_count),
                    dim3(kDecodeWarps * 32), smem, stream, /*programmatic=*/true, kmap, vmap, p);
  if (e != cudaSuccess) return e;
  // Items with many segments (more than ~6 workers per item) take the merge
  // that loads up to 32 segments in one round.
  const int rows = p.batch * p.num_q_heads;
  const bool wide = !kCombine && static_cast<int64_t>(p.num_workers) >
                                     static_cast<int64_t>(6) * p.batch * p.num_kv_heads;
  if (wide)
    return launch_kernel(decode_merge_kernel<G, kCombine, kList, true>, dim3((rows + 7) / 8),
                         dim3(256), 0, stream, /*programmatic=*/true, p);
  return launch_kernel(decode_merge_kernel<G, kCombine, kList, false>, dim3((rows + 7) / 8),
                       dim3(256), 0, stream, /*programmatic=*/true, p);
}

// Few (row, kv head) items for the machine's workers means long items: then
// the CTAs combine their partials of those before the merge.
template <int G>
static cudaError_t launch_decode_g(const DecodeParams& p, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, int sm_count, cudaStream_t stream) {
  const bool combine =
      static_cast<int64_t>(p.batch) * p.num_kv_heads * kLongItemSegs < p.num_workers;
  // the token-list mode (pkv_mixed_attention) takes q from device memory only
  if (p.row_token != nullptr)
    return combine ? launch_decode_gc<G, true, true, false>(p, kmap, vmap, sm_count, stream)
                   : launch_decode_gc<G, false, true, false>(p, kmap, vmap, sm_count, stream);
  if (p.q_host)
    return combine ? launch_decode_gc<G, true, false, true>(p, kmap, vmap, sm_count, stream)
                   : launch_decode_gc<G, false, false, true>(p, kmap, vmap, sm_count, stream);
  return combine ? launch_decode_gc<G, true, false, false>(p, kmap, vmap, sm_count, stream)
                 : launch_decode_gc<G, false, false, false>(p, kmap, vmap, sm_count, stream);
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
