// pkv_prefill_paged.cu - K5 chunked prefill over the paged cache on tcgen05.
//
// Source: the step the pages leave on the table ("flex_vs_vllm.md", "What's
// left on the table", chunked prefill: prefill and decode interleaved in one
// pass, the earlier context read from the pages). Each packed query token i
// attends the logical keys 0..input_pos[i] of its batch slot batch_idx[i],
// read through the page table (the decode rule, "qwen3_flex_inference.py",
// _decode_block_mask / causal_offset, applied to every token of a chunk). The
// chunk's own K/V are appended to the pools first (pkv_append), so a token
// sees its own chunk up to itself. Tokens need no particular order: a decode
// token is a chunk of one.
//
// The kernel keeps the packed prefill's roles (pkv_prefill.cu): a persistent
// grid walks items of one 128-row query tile x two query heads of a GQA
// group, dealt by estimated cost, largest first, a sequence's tiles together
// (sched_build in pkv_prefill_common.cuh); warp 0 loads Q and a 5-slot ring of 128-key K/V tiles by TMA, warp 1
// issues the tcgen05 MMAs, warps 2..9 run the masked online softmax, one row
// per thread, and the epilogue. Two things differ in the tile loop:
//  * P stays in tensor memory: the softmax writes it as bf16 pairs over the
//    first half of S_h, and O_h += P_h V reads its A operand from there, so
//    the PV product reads only V from shared memory (the packed kernel writes
//    P to shared memory and the product reads it back). Because P_h sits on
//    S_h, the next tile's S_h is issued only after that PV has completed;
//    the two heads' chains (QK, softmax, PV) interleave on the tensor pipe.
//    This pays on the long key ranges of chunks over a cached prefix (561 ->
//    488 us on 16 chunks of 512 over prefixes U[512, 4096]); on the packed
//    workload's short documents, with a few key tiles per item, the serial
//    chain is exposed and the packed kernel keeps P in shared memory;
//  * output rows go straight from registers to global memory, and the
//    shared memory this frees deepens the K/V ring from 3 to 5 slots.
// What changes otherwise is where the keys come from:
//  * the rows of a query tile fall into runs of equal batch slot (ballots
//    over the tile's slots); a run with slot s whose largest position is M
//    reads the logical key tiles j = 0..M/128 of slot s;
//  * a key tile is staged from the pools through the page table: one box of
//    128 rows per head-dim half when a page holds whole tiles (page_size a
//    multiple of 128), else one box per page per half (page_size 16, 32 or
//    64); rows past the run's last position come from page 0 as filler;
//  * a row sees key tile j of its own run only, columns 0..pos-128j;
//  * V rows past the run's last position are zeroed in shared memory before
//    the PV product (stale slots of a page may hold any bits, NaN included;
//    their P is zero, but 0 * NaN is not).
// Every role recomputes the runs from the same tile metadata, so they agree
// on the key-tile sequence without sharing it through memory.
#include <atomic>
#include <cmath>

#include "pkv_prefill_common.cuh"

namespace pkv {

namespace {

using namespace prefill_detail;

// Each query tile is loaded once per item, while a chunk's K/V tiles are read
// by all its query tiles: Q's TMA loads carry an L2 evict-first policy, so
// its lines are the first replaced and the K/V tiles stay in L2 (16 chunks of
// 512 over prefixes U[512, 4096]: 380 -> 376 us, same box, two runs each).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_3d_evict_first(void* dst, const CUtensorMap* map,
                                                        uint64_t* bar, int x, int y, int z,
                                                        uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "l"(pol)
      : "memory");
}

// The output rows are written once and read by no later item: their stores
// carry the same evict-first policy (375.0 / 375.4 against 377.0 / 377.0 us
// on the chunks, same box).
__device__ __forceinline__ void st_global_v4_evict_first(void* a, const uint4 w, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(a), "r"(w.x),
               "r"(w.y), "r"(w.z), "r"(w.w), "l"(pol)
               : "memory");
}

// The epilogue of one row: O / l from this thread's TMEM lane (columns t_o ..
// t_o + 127) as bf16 into orow (zeros when `has` is false), 32 head dims at a
// time, straight from registers to global memory. Every lane of the warp must
// call it (the TMEM loads are warp-collective); only lanes with `store` set
// write.
__device__ __forceinline__ void store_o_row_evict_first(__nv_bfloat16* orow, uint32_t t_o,
                                                        float inv, bool has, bool store) {
  const uint64_t pol = l2_evict_first_policy();
#pragma unroll
  for (int c = 0; c < kHeadDim; c += 32) {
    uint32_t o[32];
    tmem_ld32(t_o + c, o);
    tmem_wait_ld();
    if (store) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (has) {
          const int e = 8 * q;
          w.x = pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
          w.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
          w.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
          w.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
        }
        st_global_v4_evict_first(orow + c + 8 * q, w, pol);
      }
    }
  }
}

// shared memory layout (offsets from a 1024-aligned base). P lives in tensor
// memory and the output rows are written straight from registers, so all but
// Q is K/V ring.
constexpr int kRing = 5;                              // K/V tile slots
constexpr int kOffQ = 0;                              // Q0, Q1
constexpr int kOffRing = kOffQ + 2 * kTileBytes;      // kRing slots
constexpr int kOffBar = kOffRing + kRing * kTileBytes;
// q_full, q_empty, ring_full[kRing], ring_empty[kRing], s_full[2], p_full[2],
// pv_done[2], o_free[2]
constexpr int kNumBars = 2 + 2 * kRing + 8;
constexpr int kOffMisc = kOffBar + kNumBars * 8;      // tmem slot, abort flag
constexpr int kOffSched = kOffMisc + 16;              // this CTA's item list
constexpr int kSmemBytes = kOffSched + kSchedBytes + 1024;  // + slack for 1024 alignment
static_assert(kRing * kTileBytes >= kSchedScratchBytes, "schedule scratch lives in the ring");
static_assert(kSmemBytes <= kMaxDynSmem, "shared memory above the opt-in limit");

struct PagedPrefillParams {
  const int32_t* page_table;
  const int32_t* batch_idx;
  const int32_t* input_pos;
  const uint8_t* skip;  // nullable: tokens served elsewhere (nothing written here)
  // nullable: query tiles start at seg_start[0, *seg_count) and cover the run
  // of equal slots from there (at most 128 rows), instead of 128-row windows
  const int32_t* seg_start;
  const int32_t* seg_count;
  void* out;
  float* lse;
  int32_t* dev_err;
  int n_tokens;
  int num_q_heads;
  int group;
  int heads_per_item;   // 2 when group >= 2, else 1
  int n_tiles;          // query tiles
  int n_items;          // n_tiles * num_q_heads / heads_per_item
  int page_size;
  int num_pages;
  int max_batch;
  int max_blocks;
  int box_rows;         // rows of one K/V TMA box: min(page_size, 128)
  float qscale;         // scale * log2(e)
};

// Slot and position of a row, or slot 0 for padding, for a rejected row
// (slot outside the table, position outside [0, max_blocks * page_size)) and
// for a token another kernel serves (skip).
__device__ __forceinline__ void row_meta(const PagedPrefillParams& p, int i, int& b, int& pos,
                                         int& err) {
  b = 0;
  pos = 0;
  err = 0;
  if (i < 0 || i >= p.n_tokens) return;
  if (p.skip != nullptr && __ldg(p.skip + i) != 0) return;
  const int bb = __ldg(p.batch_idx + i);
  const int pp = __ldg(p.input_pos + i);
  if (bb == 0) return;
  if (bb < 0 || bb >= p.max_batch) err = PKV_DEV_ERR_BAD_SLOT;
  else if (pp < 0 || pp >= p.max_blocks * p.page_size) err = PKV_DEV_ERR_BAD_POS;
  if (err) return;
  b = bb;
  pos = pp;
}

// One warp's view of a query tile's 128 rows: lane l holds rows l + 32 m.
// The tile starts at token r0; its first `len` rows are its own (all 128 for
// the usual tiles; with listed tile starts, the leading rows whose slot, as
// given, equals the first row's). Rows past len are no part of the tile.
struct TileRows {
  int b[4];
  int pos[4];
  int r0;
  int len;
};

template <bool kSeg>
__device__ __forceinline__ TileRows tile_rows_load(const PagedPrefillParams& p, int r0, int lane) {
  TileRows t;
  t.r0 = r0;
  t.len = kBM;
  if (kSeg && r0 >= 0) {
    const int b0 = __ldg(p.batch_idx + r0);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int i = r0 + lane + 32 * m;
      const uint32_t brk =
          __ballot_sync(0xffffffffu, i >= p.n_tokens || __ldg(p.batch_idx + i) != b0);
      if (brk != 0u) t.len = min(t.len, 32 * m + __ffs(brk) - 1);
    }
  }
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    int err;
    const int row = lane + 32 * m;
    row_meta(p, r0 >= 0 && row < t.len ? r0 + row : -1, t.b[m], t.pos[m], err);
  }
  return t;
}

// Rows that start a run of equal slots, as four 32-bit masks (row r is bit
// r % 32 of mask r / 32). Row 0 always starts one.
struct RunMasks {
  uint32_t start[4];
};

__device__ __forceinline__ RunMasks run_masks(const TileRows& t, int lane) {
  RunMasks rm;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    int prev = __shfl_up_sync(0xffffffffu, t.b[m], 1);
    const int wrap = __shfl_sync(0xffffffffu, m > 0 ? t.b[m > 0 ? m - 1 : 0] : -1, 31);
    if (lane == 0) prev = (m == 0) ? -1 : wrap;
    rm.start[m] = __ballot_sync(0xffffffffu, t.b[m] != prev);
  }
  return rm;
}

// First run start at or after row r (kBM if none).
__device__ __forceinline__ int next_start(const RunMasks& rm, int r) {
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    if (r >= 32 * (m + 1)) continue;
    uint32_t bits = rm.start[m];
    const int lo = r - 32 * m;
    if (lo > 0) bits &= ~((1u << lo) - 1u);
    if (bits) return 32 * m + __ffs(bits) - 1;
  }
  return kBM;
}

// Position in an item's key-tile sequence: run rows [s, e) of slot `slot`,
// largest position maxpos, nkv key tiles, current tile j. Warp-collective.
struct RunCursor {
  int s, e, slot, maxpos, nkv, j;
};

__device__ __forceinline__ void run_setup(RunCursor& c, const TileRows& t, const RunMasks& rm,
                                          int lane) {
  c.e = next_start(rm, c.s + 1);
  const int ms = c.s >> 5;
  const int bsel = ms == 0 ? t.b[0] : ms == 1 ? t.b[1] : ms == 2 ? t.b[2] : t.b[3];
  c.slot = __shfl_sync(0xffffffffu, bsel, c.s & 31);
  int mp = -1;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int r = lane + 32 * m;
    if (r >= c.s && r < c.e) mp = max(mp, t.pos[m]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mp = max(mp, __shfl_xor_sync(0xffffffffu, mp, o));
  c.maxpos = mp;
  c.nkv = (c.slot != 0 && mp >= 0) ? mp / kBN + 1 : 0;
  c.j = 0;
}

__device__ __forceinline__ void cursor_skip_empty(RunCursor& c, const TileRows& t,
                                                  const RunMasks& rm, int lane) {
  while (c.s < kBM) {
    run_setup(c, t, rm, lane);
    if (c.nkv > 0) return;
    c.s = c.e;
  }
}

__device__ __forceinline__ void cursor_first(RunCursor& c, const TileRows& t, const RunMasks& rm,
                                             int lane) {
  c.s = 0;
  cursor_skip_empty(c, t, rm, lane);
}

__device__ __forceinline__ void cursor_next(RunCursor& c, const TileRows& t, const RunMasks& rm,
                                            int lane) {
  if (++c.j < c.nkv) return;
  c.s = c.e;
  cursor_skip_empty(c, t, rm, lane);
}

// Key tiles of an item (all runs).
__device__ __forceinline__ int count_tiles(const TileRows& t, const RunMasks& rm, int lane) {
  int n = 0;
  RunCursor c;
  c.s = 0;
  while (c.s < kBM) {
    run_setup(c, t, rm, lane);
    n += c.nkv;
    c.s = c.e;
  }
  return n;
}

// Items of the call: tiles x head groups; with listed tile starts the tile
// count is read on the device.
template <bool kSeg>
__device__ __forceinline__ int call_items(const PagedPrefillParams& p, int items_per_tile) {
  return kSeg ? *p.seg_count * items_per_tile : p.n_items;
}

// First token of an item's query tile (-1 past the last item).
template <bool kSeg>
__device__ __forceinline__ int item_r0(const PagedPrefillParams& p, int item, int items_per_tile,
                                       int n_items) {
  if (item < 0 || item >= n_items) return -1;
  const int tile = item / items_per_tile;
  return kSeg ? __ldg(p.seg_start + tile) : tile * kBM;
}

}  // namespace

// 10 warps: two of the four SM sub-partitions hold three warps, so at most
// 16384 / 96 = 170 registers per thread
// kSeg: query tiles start at the listed tokens (p.seg_start) and cover one
// run piece each; else they are fixed 128-row windows of the packing.
template <bool kSeg>
__global__ void __launch_bounds__(kThreads, 1)
prefill_paged_tcgen05_kernel(const __grid_constant__ CUtensorMap qmap,
                             const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap vmap,
                             const PagedPrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* ring_full = bars + 2;               // [kRing]
  uint64_t* ring_empty = bars + 2 + kRing;      // [kRing]
  uint64_t* s_full = bars + 2 + 2 * kRing;      // [2]
  uint64_t* p_full = s_full + 2;                // [2]: P_h in TMEM, O_h rescaled
  uint64_t* pv_done = s_full + 4;               // [2]
  uint64_t* o_free = s_full + 6;                // [2]: epilogue has read O_h
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int hpi = p.heads_per_item;
  const int items_per_tile = p.num_q_heads / hpi;
  const int n_tiles = kSeg ? *p.seg_count : p.n_tiles;
  const int n_items = call_items<kSeg>(p, items_per_tile);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&ring_full[s], 1);
      mbar_init(&ring_empty[s], 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&s_full[h], 1);
      mbar_init(&p_full[h], kGroupThreads);
      mbar_init(&pv_done[h], 1);
      mbar_init(&o_free[h], kGroupThreads);
    }
    *s_abort = (p.dev_err != nullptr &&
                (*reinterpret_cast<volatile int32_t*>(p.dev_err) & PKV_DEV_ERR_TIMEOUT)) ? 1 : 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // tile cost: key tiles of the run at the tile's first row, plus those of
  // the run at its last row when that is another run of a fixed window, plus
  // one for the item's Q load and epilogue
  const uint16_t* s_list = reinterpret_cast<const uint16_t*>(smem + kOffSched);
  const ItemSched S = sched_build(
      reinterpret_cast<uint16_t*>(smem + kOffSched), smem + kOffRing, n_tiles, items_per_tile,
      [&](int t) -> int {
        const int r0 = kSeg ? __ldg(p.seg_start + t) : t * kBM;
        if (r0 < 0 || r0 >= p.n_tokens) return 0;
        const int rl = min(r0 + kBM, p.n_tokens) - 1;
        const int b0 = __ldg(p.batch_idx + r0), bl = __ldg(p.batch_idx + rl);
        const int q0 = __ldg(p.input_pos + r0), ql = __ldg(p.input_pos + rl);
        auto tiles = [](int b, int pos) { return (b != 0 && pos >= 0) ? pos / kBN + 1 : 0; };
        if (b0 == bl) return tiles(b0, max(q0, ql)) + 1;
        return tiles(b0, q0) + (kSeg ? 0 : tiles(bl, ql)) + 1;
      },
      [&](int t) -> bool {  // the next tile's first row is in this tile's last run
        const int r1 = kSeg ? __ldg(p.seg_start + t + 1) : (t + 1) * kBM;
        if (r1 <= 0 || r1 >= p.n_tokens) return false;
        const int b1 = __ldg(p.batch_idx + r1);
        return b1 != 0 && b1 == __ldg(p.batch_idx + r1 - 1);
      });

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer ----
    uint32_t L = 0;   // ring loads issued
    uint32_t qi = 0;  // non-empty items
    const int R = p.box_rows;
    const int nsub = kBN / R;  // boxes per head-dim half of a key tile (1..8)
    int item = sched_item(S, s_list, 0);
    TileRows nxt = tile_rows_load<kSeg>(p, item_r0<kSeg>(p, item, items_per_tile, n_items), lane);
    for (int r = 0; item >= 0 && !*s_abort; item = sched_item(S, s_list, ++r)) {
      const int h0 = (item % items_per_tile) * hpi;
      const int kvh = h0 / p.group;
      const TileRows cur = nxt;
      const int r0 = cur.r0;
      nxt = tile_rows_load<kSeg>(p, item_r0<kSeg>(p, sched_item(S, s_list, r + 1), items_per_tile, n_items), lane);
      const RunMasks rm = run_masks(cur, lane);
      const int n_kv = count_tiles(cur, rm, lane);
      if (n_kv == 0) continue;
      bool ok = true;
      if (lane == 0) {
        ok = qi == 0 || wait_or_abort(q_empty, (qi - 1) & 1, s_abort);
        if (ok) {
          const uint64_t q_policy = l2_evict_first_policy();
          mbar_arrive_expect_tx(q_full, hpi * kTileBytes);
          for (int h = 0; h < hpi; ++h) {
            uint8_t* qd = smem + kOffQ + h * kTileBytes;
            tma_load_3d_evict_first(qd, &qmap, q_full, 0, h0 + h, r0, q_policy);
            tma_load_3d_evict_first(qd + kHalf, &qmap, q_full, 64, h0 + h, r0, q_policy);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // One 128-key tile of run c through the page table. Lane k < nsub finds
      // the pool row of box k; positions past the run's last key (and an
      // unreserved entry, flagged) read page 0 as filler.
      auto load = [&](const CUtensorMap* map, const RunCursor& c) -> bool {
        int rowk = 0;
        bool bad = false;
        if (lane < nsub) {
          const int l0 = c.j * kBN + lane * R;
          if (l0 <= c.maxpos) {
            const int blk = l0 / p.page_size;
            const int pg = __ldg(p.page_table + static_cast<int64_t>(c.slot) * p.max_blocks + blk);
            if (pg < 0 || pg >= p.num_pages) bad = true;
            else rowk = pg * p.page_size + l0 % p.page_size;
          }
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) set_dev_err(p.dev_err, PKV_DEV_ERR_BAD_PAGE);
        int rows[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) rows[k] = __shfl_sync(0xffffffffu, rowk, k);
        bool good = true;
        if (lane == 0) {
          const uint32_t slot = L % kRing;
          if (L >= kRing && !wait_or_abort(&ring_empty[slot], ((L / kRing) - 1) & 1, s_abort)) {
            good = false;
          } else {
            uint8_t* dst = smem + kOffRing + slot * kTileBytes;
            mbar_arrive_expect_tx(&ring_full[slot], kTileBytes);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              if (k < nsub) {
                tma_load_4d(dst + k * R * 128, map, &ring_full[slot], 0, rows[k], 0, kvh);
                tma_load_4d(dst + kHalf + k * R * 128, map, &ring_full[slot], 0, rows[k], 1, kvh);
              }
            }
          }
        }
        ++L;
        return __shfl_sync(0xffffffffu, good, 0);
      };
      // ring order = the MMA thread's consumption order:
      // K_0, then for each tile t: K_{t+1} (if any), V_t
      RunCursor kc, vc;
      cursor_first(kc, cur, rm, lane);
      vc = kc;
      ok = ok && load(&kmap, kc);
      cursor_next(kc, cur, rm, lane);
      for (int t = 0; ok && t < n_kv; ++t) {
        if (t + 1 < n_kv) {
          ok = load(&kmap, kc);
          cursor_next(kc, cur, rm, lane);
        }
        ok = ok && load(&vmap, vc);
        cursor_next(vc, cur, rm, lane);
      }
      if (!ok && lane == 0) *s_abort = 1;
      __syncwarp();
      ++qi;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer ----
    // The whole warp runs this loop (warp-uniform bookkeeping; all lanes zero
    // stale V rows) and one elected lane issues every tensor instruction
    // (always the same lane: a commit tracks only the MMAs of the thread that
    // commits), with every descriptor word computed before each burst:
    // anything issued between two MMAs leaves the tensor pipe idle. Per tile
    // and head: PV_h, then the head's next QK once that PV has read P_h (P_h
    // sits on S_h). (PV of both heads first, then the QKs, measured slower.)
    uint32_t C = 0;       // ring slots consumed
    uint32_t qi = 0;      // non-empty items
    uint32_t tc = 0;      // KV tiles processed (all items)
    const uint32_t sR = smem_u32(smem + kOffRing);
    uint32_t qd[2][8];
    kmajor_steps(smem_u32(smem + kOffQ), qd[0]);
    kmajor_steps(smem_u32(smem + kOffQ + kTileBytes), qd[1]);
    // every lane tests the barrier; lane 0's outcome is the warp's
    auto wait_w = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __shfl_sync(0xffffffffu, wait_or_abort(bar, parity, s_abort) ? 1 : 0, 0) != 0;
    };
    auto issue_qk = [&](int h, const uint32_t (&kb)[8]) {  // S_h = Q_h K^T
      if (elect_one()) {
        umma8_ss(tmem + static_cast<uint32_t>(h * kBN), qd[h], kb, kIdescQK, 0u);
        umma_commit(&s_full[h]);
      }
      __syncwarp();
    };
    auto issue_pv = [&](int h, const uint32_t (&vb)[8], uint32_t acc) {  // O_h (+)= P_h V
      if (elect_one()) {
        umma8_ts(tmem + static_cast<uint32_t>(256 + h * kHeadDim),  // O_h
                 tmem + static_cast<uint32_t>(h * kBN), vb, kIdescPV, acc);  // P_h, over S_h
        umma_commit(&pv_done[h]);
      }
      __syncwarp();
    };
    auto commit_w = [&](uint64_t* bar) {
      if (elect_one()) umma_commit(bar);
      __syncwarp();
    };
    int item = sched_item(S, s_list, 0);
    TileRows nxt = tile_rows_load<kSeg>(p, item_r0<kSeg>(p, item, items_per_tile, n_items), lane);
    for (int r = 0; item >= 0 && !*s_abort; item = sched_item(S, s_list, ++r)) {
      const TileRows cur = nxt;
      nxt = tile_rows_load<kSeg>(p, item_r0<kSeg>(p, sched_item(S, s_list, r + 1), items_per_tile, n_items), lane);
      const RunMasks rm = run_masks(cur, lane);
      const int n_kv = count_tiles(cur, rm, lane);
      if (n_kv == 0) continue;
      RunCursor vc;
      cursor_first(vc, cur, rm, lane);
      const uint32_t k0slot = C % kRing;
      bool ok = wait_w(q_full, qi & 1) && wait_w(&ring_full[k0slot], (C / kRing) & 1);
      if (ok) {
        uint32_t kb[8];
        kmajor_steps(sR + k0slot * kTileBytes, kb);
        // S_h is free once the previous item's last PV_h has read P_h from it
        for (int h = 0; ok && h < hpi; ++h) {
          if (tc > 0) ok = wait_w(&pv_done[h], (tc - 1) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_qk(h, kb);
        }
        if (ok) {
          commit_w(&ring_empty[k0slot]);
          if (n_kv == 1) commit_w(q_empty);
        }
      }
      ++C;
      for (int t = 0; ok && t < n_kv; ++t) {
        // ring order: K_{t+1} (if any), then V_t
        const bool more = t + 1 < n_kv;
        const uint32_t ck = C;
        if (more) ++C;
        const uint32_t cv = C++;
        const uint32_t kslot = ck % kRing;
        const uint32_t vslot = cv % kRing;
        // the V tile has landed: zero its rows past the run's last key
        if (!__all_sync(0xffffffffu,
                        wait_or_abort(&ring_full[vslot], (cv / kRing) & 1, s_abort))) {
          ok = false;
          break;
        }
        const int nvalid = min(kBN, vc.maxpos + 1 - vc.j * kBN);
        if (nvalid < kBN) {
          uint8_t* vt = smem + kOffRing + vslot * kTileBytes;
          const int chunks = (kBN - nvalid) * 16;  // 16-byte chunks: 2 halves x 8 per row
          for (int q = lane; q < chunks; q += 32) {
            const int r = nvalid + (q >> 4);
            const int c = q & 15;
            *reinterpret_cast<uint4*>(vt + (c >> 3) * kHalf + r * 128 + (c & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        uint32_t vb[8], kb[8];
        vmn_steps(sR + vslot * kTileBytes, vb);
        kmajor_steps(sR + kslot * kTileBytes, kb);
        if (more) ok = wait_w(&ring_full[kslot], (ck / kRing) & 1);
        for (int h = 0; h < hpi && ok; ++h) {
          ok = wait_w(&p_full[h], tc & 1);
          if (ok && t == 0 && qi > 0) ok = wait_w(&o_free[h], (qi - 1) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_pv(h, vb, t > 0 ? 1u : 0u);
          if (more) {
            ok = wait_w(&pv_done[h], tc & 1);
            if (!ok) break;
            tc_fence_after();
            issue_qk(h, kb);
          }
        }
        if (!ok) break;
        commit_w(&ring_empty[vslot]);
        if (more) {
          commit_w(&ring_empty[kslot]);
          if (t + 2 == n_kv) commit_w(q_empty);
        }
        ++tc;
        cursor_next(vc, cur, rm, lane);
      }
      if (!ok && lane == 0) *s_abort = 1;
      __syncwarp();
      ++qi;
    }
  } else {
    // ---------------------------------------------------- softmax rows ----
    const int grp = (warp - 2) >> 2;      // which head of the item
    const int lane_base = 32 * (warp & 3);
    const int row = lane_base + lane;
    const uint32_t t_s = tmem + (static_cast<uint32_t>(lane_base) << 16) + grp * kBN;
    const uint32_t t_o = tmem + (static_cast<uint32_t>(lane_base) << 16) + 256 + grp * kHeadDim;
    uint32_t tc = 0, qi = 0;
    const bool active = grp < hpi;
    int item = sched_item(S, s_list, 0);
    TileRows nxt = tile_rows_load<kSeg>(p, item_r0<kSeg>(p, item, items_per_tile, n_items), lane);
    for (int r = 0; active && item >= 0; item = sched_item(S, s_list, ++r)) {
      if (__any_sync(0xffffffffu, *s_abort != 0)) break;  // warp-uniform exit
      const int head = (item % items_per_tile) * hpi + grp;
      const TileRows cur = nxt;
      const int r0 = cur.r0;
      nxt = tile_rows_load<kSeg>(p, item_r0<kSeg>(p, sched_item(S, s_list, r + 1), items_per_tile, n_items), lane);
      const RunMasks rm = run_masks(cur, lane);
      const int n_kv = count_tiles(cur, rm, lane);
      const int i = r0 + row;
      const bool mine = row < cur.len;  // the row belongs to this tile
      int my_b, my_pos, my_err;
      row_meta(p, mine ? i : -1, my_b, my_pos, my_err);
      if (my_err && grp == 0) set_dev_err(p.dev_err, my_err);
      float m_run = -INFINITY;  // running max, raw score units
      float l_run = 0.f;
      bool ok = true;
      RunCursor c;
      cursor_first(c, cur, rm, lane);
      for (int j = 0; j < n_kv && ok; ++j) {
        if (!__all_sync(0xffffffffu, wait_or_abort(&s_full[grp], tc & 1, s_abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[128];
        {
          uint32_t (&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
          uint32_t (&b)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
          uint32_t (&cc)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[64]);
          uint32_t (&d)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[96]);
          tmem_ld32(t_s + 0, a);
          tmem_ld32(t_s + 32, b);
          tmem_ld32(t_s + 64, cc);
          tmem_ld32(t_s + 96, d);
          tmem_wait_ld();
        }
        // this row sees key tile j of its own run, columns 0 .. pos - 128j
        const bool in_run = row >= c.s && row < c.e;
        const int c_hi = in_run ? min(my_pos - c.j * kBN, kBN - 1) : -1;
        const bool full = c_hi == kBN - 1;
        cursor_next(c, cur, rm, lane);
        // masked columns become -inf (all of them when nothing is visible, c_hi
        // < 0), so every lane takes the same P path (the TMEM store is
        // warp-collective)
        float mx;
        if (full) {
          mx = row_max_full(sr);
        } else {
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int q = 0; q < kBN; ++q) {
            const float v = q <= c_hi ? __uint_as_float(sr[q]) : -INFINITY;
            sr[q] = __float_as_uint(v);
            m4[q & 3] = fmaxf(m4[q & 3], v);
          }
          mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        const float m_cand = fmaxf(m_run, mx);
        const bool grow = (m_run == -INFINITY)
                              ? (m_cand != -INFINITY)
                              : ((m_cand - m_run) * p.qscale > kRescaleThreshold);
        const float m_use = grow ? m_cand : m_run;
        const float alpha = grow ? ex2((m_run - m_use) * p.qscale) : 1.f;  // 0 if m_run=-inf
        const float neg_m = (m_use == -INFINITY) ? 0.f : -m_use * p.qscale;
        const bool got = (j == 0) || wait_or_abort(&pv_done[grp], (tc - 1) & 1, s_abort);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // P over the first 64 columns of S_h (already in registers)
        const float psum = softmax_row_to_tmem(sr, p.qscale, neg_m, t_s);
        l_run = l_run * alpha + psum;
        m_run = m_use;
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
          for (int q = 0; q < kHeadDim; q += 32) {
            uint32_t o[32];
            tmem_ld32(t_o + q, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(t_o + q, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[grp]);
        ++tc;
      }
      // ---- epilogue: O / l, LSE ----
      if (ok && n_kv > 0) {
        const bool got = wait_or_abort(&pv_done[grp], (tc - 1) & 1, s_abort);
        if (!__all_sync(0xffffffffu, got)) ok = false;
      }
      tc_fence_after();
      // tokens served by another kernel are not written here
      const bool in_range =
          mine && i < p.n_tokens && !(p.skip != nullptr && __ldg(p.skip + i) != 0);
      const bool has = in_range && my_b != 0 && ok && l_run > 0.f;
      const float inv = has ? 1.f / l_run : 0.f;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                            (static_cast<int64_t>(i) * p.num_q_heads + head) * kHeadDim;
      if (n_kv > 0 && ok) {
        // O / l as bf16 straight from TMEM to this row of the output (the
        // item's last PV has completed)
        store_o_row_evict_first(orow, t_o, inv, has, in_range);
      } else if (in_range) {
        // no key tile at all (padding-only tile) or an aborted item: zeros
#pragma unroll
        for (int q = 0; q < kHeadDim; q += 8)
          *reinterpret_cast<uint4*>(orow + q) = make_uint4(0u, 0u, 0u, 0u);
      }
      if (in_range)
        p.lse[static_cast<int64_t>(i) * p.num_q_heads + head] =
            has ? (m_run * p.qscale + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
      if (n_kv > 0) {
        tc_fence_before();
        mbar_arrive(&o_free[grp]);
        ++qi;
      }
      if (!ok) {
        set_dev_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
        *s_abort = 1;
        break;
      }
    }
  }
  if (*s_abort && threadIdx.x == 0) set_dev_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

using namespace prefill_host;

namespace {
// 4-D view {64 dims, rows, 2 halves of the head dims, H_kv} of a pool; one box
// is `box_rows` rows of one half of one head, 128-byte swizzled, so a box of
// page k of a 128-key tile lands at rows k * box_rows.. of that half.
bool encode_pool_box_map(CUtensorMap* map, const void* pool, const pkv_cache_desc* c,
                         int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {64u, static_cast<cuuint64_t>(c->num_pages) * c->page_size, 2u,
                              static_cast<cuuint64_t>(c->num_kv_heads)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(c->num_kv_heads) * c->head_dim * 2,
                                 128u, static_cast<cuuint64_t>(c->head_dim) * 2};
  const cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(box_rows), 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

pkv_status prefill_paged_entry(const pkv_cache_desc* cache, const void* k_pool,
                               const void* v_pool, const int32_t* page_table, const void* q,
                               int num_q_heads, const int32_t* batch_idx,
                               const int32_t* input_pos, int n_tokens, float scale, void* out,
                               float* lse, int32_t* dev_err, cudaStream_t stream,
                               const uint8_t* skip, const int32_t* seg_start,
                               const int32_t* seg_count) {
  if (cache == nullptr || cache->head_dim != kHeadDim || cache->num_pages <= 0 ||
      cache->num_kv_heads <= 0 || cache->max_batch <= 0 || cache->max_blocks <= 0)
    return PKV_ERR_ARG;
  const int ps = cache->page_size;
  if (!(ps == 16 || ps == 32 || ps == 64 || (ps > 0 && ps % 128 == 0))) return PKV_ERR_ARG;
  if (static_cast<long long>(cache->num_pages) * ps > INT32_MAX ||
      static_cast<long long>(cache->max_blocks) * ps > INT32_MAX ||
      static_cast<long long>(cache->max_batch) * cache->max_blocks > INT32_MAX)
    return PKV_ERR_ARG;
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads != 0) return PKV_ERR_ARG;
  const int g = num_q_heads / cache->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return PKV_ERR_ARG;
  if (n_tokens < 0 || !std::isfinite(scale) || !(scale > 0.f)) return PKV_ERR_ARG;
  if (n_tokens == 0) return PKV_OK;
  if (!k_pool || !v_pool || !page_table || !q || !batch_idx || !input_pos || !out || !lse)
    return PKV_ERR_ARG;
  if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(q, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(page_table, 4) || !aligned(batch_idx, 4) ||
      !aligned(input_pos, 4) || !aligned(dev_err, 4))
    return PKV_ERR_ALIGN;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (major != 10 || minor != 3) return PKV_ERR_DEVICE;
  if (static_cast<long long>(((n_tokens + kBM - 1) / kBM)) * num_q_heads > INT32_MAX)
    return PKV_ERR_ARG;
  const int box_rows = ps < kBN ? ps : kBN;

  CUtensorMap qmap, kmap, vmap;
  if (!encode_packed_map(&qmap, q, num_q_heads, n_tokens) ||
      !encode_pool_box_map(&kmap, k_pool, cache, box_rows) ||
      !encode_pool_box_map(&vmap, v_pool, cache, box_rows))
    return PKV_ERR_ARG;

  static std::atomic<bool> attr_set[64] = {};  // per device; host threads may race to set it
  if (dev < 0 || dev >= 64) return PKV_ERR_DEVICE;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t ea = cudaFuncSetAttribute(prefill_paged_tcgen05_kernel<false>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (ea == cudaSuccess)
      ea = cudaFuncSetAttribute(prefill_paged_tcgen05_kernel<true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (ea != cudaSuccess) return record_cuda_status(ea);
    attr_set[dev].store(true, std::memory_order_release);
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PKV_ERR_CUDA;
  PagedPrefillParams prm;
  prm.page_table = page_table;
  prm.batch_idx = batch_idx;
  prm.input_pos = input_pos;
  prm.skip = skip;
  prm.seg_start = seg_count != nullptr ? seg_start : nullptr;
  prm.seg_count = seg_count;
  prm.out = out;
  prm.lse = lse;
  prm.dev_err = dev_err;
  prm.n_tokens = n_tokens;
  prm.num_q_heads = num_q_heads;
  prm.group = g;
  prm.heads_per_item = g >= 2 ? 2 : 1;
  prm.n_tiles = (n_tokens + kBM - 1) / kBM;
  prm.n_items = prm.n_tiles * (num_q_heads / prm.heads_per_item);
  prm.page_size = ps;
  prm.num_pages = cache->num_pages;
  prm.max_batch = cache->max_batch;
  prm.max_blocks = cache->max_blocks;
  prm.box_rows = box_rows;
  prm.qscale = scale * 1.4426950408889634f;
  // with listed tile starts there are at most n_tokens tiles
  const long long items_max =
      prm.seg_start != nullptr ? static_cast<long long>(n_tokens) * (num_q_heads / prm.heads_per_item)
                               : prm.n_items;
  const int grid = items_max < sms ? static_cast<int>(items_max) : sms;
  const cudaError_t e =
      prm.seg_start != nullptr
          ? launch_kernel(prefill_paged_tcgen05_kernel<true>, dim3(grid), dim3(kThreads),
                          kSmemBytes, stream, false, qmap, kmap, vmap, prm)
          : launch_kernel(prefill_paged_tcgen05_kernel<false>, dim3(grid), dim3(kThreads),
                          kSmemBytes, stream, false, qmap, kmap, vmap, prm);
  return record_cuda_status(e);
}

}  // namespace pkv
