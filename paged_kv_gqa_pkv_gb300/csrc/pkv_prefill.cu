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
// Schedule: a persistent grid (one CTA per SM) walks the work items, sorted
// by estimated cost within windows of eight rounds and dealt in snake order
// (sched_build_windowed in pkv_prefill_common.cuh); an item is one 128-row
// query tile for TWO query heads of the same GQA group, so every K/V tile is loaded once for both heads (a group of
// one head, G == 1, gives one-head items). Warp roles:
//  * warp 0 issues TMA: each item's Q tiles, then K and V tiles of 128 keys
//    into a 3-slot ring of 32 KB half-stages, in the MMA thread's order
//    (K_0, then K_j+1 and V_j for each j, continuing across items), starting
//    at the first key any row of the tile can see;
//  * warp 1 issues tcgen05 MMAs (one elected lane): S_h = Q_h K^T into TMEM
//    and O_h += P_h V. The next tile's S_h is computed as soon as the softmax
//    has read the current S_h into registers (s_free), so QK of tile j+1 runs
//    while the softmax of tile j computes its exponentials;
//  * warps 2..5 and 6..9 are the softmax warpgroups of the two heads, one
//    query row per thread (its TMEM lane): masked online softmax in fp32 with
//    exp2 and the scale folded in, P written to shared memory as bf16 in the
//    MMA's K-major 128-byte-swizzled layout, O rescaled in TMEM only when the
//    running max grows by more than 2^8, and the epilogue O / l -> bf16 + LSE,
//    staged in the head's P buffer and written with TMA stores.
// Barrier phases are running counters kept identically by every role.
// Shared-memory operands (all 128-byte swizzled, 1024-byte aligned atoms):
// Q, K and P are K-major (64 elements per 128-byte row, two 16 KB halves of
// D or of the key block); V is used MN-major straight from its TMA tile
// (64 head dims per 128-byte row, one row per key).
#include <atomic>
#include <cmath>

#include "pkv_prefill_common.cuh"

namespace pkv {

namespace {

using namespace prefill_detail;

// shared memory layout (offsets from a 1024-aligned base)
constexpr int kRing = 3;                              // K/V tile slots
constexpr int kOffQ = 0;                              // Q0, Q1
constexpr int kOffP = kOffQ + 2 * kTileBytes;         // P0, P1 (also output staging)
constexpr int kOffRing = kOffP + 2 * kTileBytes;      // kRing slots
constexpr int kOffBar = kOffRing + kRing * kTileBytes;
// q_full, q_empty, ring_full[3], ring_empty[3], s_full[2], p_full[2],
// pv_done[2], o_free[2], s_free[2], grp_sync[2]
constexpr int kNumBars = 20;
constexpr int kOffMisc = kOffBar + kNumBars * 8;      // tmem slot, abort flag
constexpr int kOffSched = kOffMisc + 16;              // this CTA's item list
constexpr int kSmemBytes = kOffSched + kSchedBytes + 1024;  // + slack for 1024 alignment
static_assert(kRing * kTileBytes >= kSchedScratchBytes, "schedule scratch lives in the ring");
static_assert(kSmemBytes <= kMaxDynSmem, "shared memory above the opt-in limit");

struct PrefillParams {
  const int32_t* batch_idx;
  const int32_t* input_pos;
  void* out;
  float* lse;
  int32_t* dev_err;
  int n_tokens;
  int num_q_heads;
  int group;
  int heads_per_item;   // 2 when group >= 2, else 1
  int n_tiles;          // query tiles
  int n_items;          // n_tiles * num_q_heads / heads_per_item
  float qscale;         // scale * log2(e)
};

// Keys [kv_lo, kv_hi) that rows r0..r0+127 can see, found by one warp with
// four rows per lane. Under the packing precondition a valid row i sees
// [i - pos_i, i]. The loads (TileRaw) are issued one item ahead of their use
// so their latency hides behind the current item.
struct TileRaw {
  int b[4];
  int pos[4];
};

__device__ __forceinline__ TileRaw tile_raw_load(const PrefillParams& p, int r0, int lane) {
  TileRaw t;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int i = r0 + lane + 32 * m;
    t.b[m] = (r0 >= 0 && i < p.n_tokens) ? __ldg(p.batch_idx + i) : 0;
    t.pos[m] = (r0 >= 0 && i < p.n_tokens) ? __ldg(p.input_pos + i) : 0;
  }
  return t;
}

__device__ __forceinline__ void tile_key_range(const TileRaw& t, int r0, int lane, int& kv_lo,
                                               int& kv_hi) {
  int lo = 0x7fffffff, hi = -1;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int i = r0 + lane + 32 * m;
    if (t.b[m] != 0) {
      const int pos = t.pos[m];
      lo = min(lo, (pos >= 0 && pos <= i) ? i - pos : i);
      hi = max(hi, i + 1);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  kv_lo = lo;
  kv_hi = hi;
}

// This thread's own row of an item: slot/position of the row and of the row
// before it (for the packing check), loaded one item ahead.
struct RowRaw {
  int b, pos, b_prev, pos_prev;
};

__device__ __forceinline__ RowRaw row_raw_load(const PrefillParams& p, int i) {
  RowRaw r{0, 0, 0, 0};
  if (i >= 0 && i < p.n_tokens) {
    r.b = __ldg(p.batch_idx + i);
    r.pos = __ldg(p.input_pos + i);
    if (i > 0) {
      r.b_prev = __ldg(p.batch_idx + i - 1);
      r.pos_prev = __ldg(p.input_pos + i - 1);
    }
  }
  return r;
}

__device__ __forceinline__ int item_r0(const PrefillParams& p, int item, int items_per_tile) {
  return (item >= 0 && item < p.n_items) ? (item / items_per_tile) * kBM : -1;
}

}  // namespace

// 10 warps: two of the four SM sub-partitions hold three warps, so at most
// 16384 / 96 = 170 registers per thread (ptxas settles on 168)
__global__ void __launch_bounds__(kThreads, 1)
prefill_tcgen05_kernel(const __grid_constant__ CUtensorMap qmap,
                       const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap,
                       const __grid_constant__ CUtensorMap omap, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* ring_full = bars + 2;   // [3]
  uint64_t* ring_empty = bars + 5;  // [3]
  uint64_t* s_full = bars + 8;      // [2]
  uint64_t* p_full = bars + 10;     // [2]
  uint64_t* pv_done = bars + 12;    // [2]
  uint64_t* o_free = bars + 14;     // [2]
  uint64_t* s_free = bars + 16;     // [2]: S_h read into registers, TMEM free
  uint64_t* grp_sync = bars + 18;   // [2]: barrier of one softmax warpgroup
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int hpi = p.heads_per_item;
  const int items_per_tile = p.num_q_heads / hpi;

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
      mbar_init(&s_free[h], kGroupThreads);
      mbar_init(&grp_sync[h], kGroupThreads);
    }
    // After a timeout anywhere in the grid, this CTA does no work (results
    // are unspecified then) instead of waiting out its own limits.
    *s_abort = (p.dev_err != nullptr &&
                (*reinterpret_cast<volatile int32_t*>(p.dev_err) & PKV_DEV_ERR_TIMEOUT)) ? 1 : 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&omap);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // tile cost: key tiles from the first row's document start to the last row
  // (the packing precondition), plus one for the item's Q load and epilogue
  const uint16_t* s_list = reinterpret_cast<const uint16_t*>(smem + kOffSched);
  const ItemSched S = sched_build_windowed(
      reinterpret_cast<uint16_t*>(smem + kOffSched), smem + kOffRing, p.n_tiles, items_per_tile,
      (8 * static_cast<int>(gridDim.x)) / items_per_tile, [&](int t) -> int {
        const int r0 = t * kBM;
        const int rl = min(r0 + kBM, p.n_tokens) - 1;
        const int b0 = __ldg(p.batch_idx + r0);
        const int p0 = __ldg(p.input_pos + r0);
        const int lo = (b0 != 0 && p0 >= 0 && p0 <= r0) ? r0 - p0 : r0;
        return (rl + 1 - lo + kBN - 1) / kBN + 1;
      });

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer ----
    uint32_t L = 0;   // ring loads issued
    uint32_t qi = 0;  // non-empty items
    int item = sched_item(S, s_list, 0);
    TileRaw raw = tile_raw_load(p, item_r0(p, item, items_per_tile), lane);
    for (int r = 0; item >= 0 && !*s_abort; item = sched_item(S, s_list, ++r)) {
      const int tile = item / items_per_tile;
      const int h0 = (item % items_per_tile) * hpi;
      const int kvh = h0 / p.group;
      const int r0 = tile * kBM;
      int kv_lo, kv_hi;
      tile_key_range(raw, r0, lane, kv_lo, kv_hi);
      raw = tile_raw_load(p, item_r0(p, sched_item(S, s_list, r + 1), items_per_tile), lane);
      if (kv_hi <= kv_lo) continue;
      const int n_kv = (kv_hi - kv_lo + kBN - 1) / kBN;
      if (lane == 0) {
        bool ok = qi == 0 || wait_or_abort(q_empty, (qi - 1) & 1, s_abort);
        if (ok) {
          mbar_arrive_expect_tx(q_full, hpi * kTileBytes);
          for (int h = 0; h < hpi; ++h) {
            uint8_t* qd = smem + kOffQ + h * kTileBytes;
            tma_load_3d(qd, &qmap, q_full, 0, h0 + h, r0);
            tma_load_3d(qd + kHalf, &qmap, q_full, 64, h0 + h, r0);
          }
        }
        // ring order = the MMA thread's consumption order:
        // K_0, then for each j: K_{j+1} (if any), V_j
        auto load = [&](const CUtensorMap* map, int j) -> bool {
          const uint32_t slot = L % kRing;
          if (L >= kRing && !wait_or_abort(&ring_empty[slot], ((L / kRing) - 1) & 1, s_abort))
            return false;
          uint8_t* dst = smem + kOffRing + slot * kTileBytes;
          mbar_arrive_expect_tx(&ring_full[slot], kTileBytes);
          tma_load_3d(dst, map, &ring_full[slot], 0, kvh, kv_lo + j * kBN);
          tma_load_3d(dst + kHalf, map, &ring_full[slot], 64, kvh, kv_lo + j * kBN);
          ++L;
          return true;
        };
        ok = ok && load(&kmap, 0);
        for (int j = 0; ok && j < n_kv; ++j) {
          if (j + 1 < n_kv) ok = load(&kmap, j + 1);
          ok = ok && load(&vmap, j);
        }
        if (!ok) *s_abort = 1;
      }
      __syncwarp();
      ++qi;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer ----
    // The whole warp runs this loop, so its bookkeeping stays warp-uniform,
    // and one elected lane issues every tensor instruction (always the same
    // lane: a commit tracks only the MMAs of the thread that commits). Per
    // tile: QK_0, QK_1 of the next key tile, then PV_0, PV_1 of this one, each
    // once its own head's barrier passes (waiting for both heads before
    // either was 0.7 % slower), each head's eight K-steps as one asm burst
    // with every descriptor word computed before it: the tensor pipe accepts
    // one MMA at a time, so anything issued between two MMAs (the warp shares
    // its SM sub-partition with busy softmax warps) leaves the pipe idle.
    uint32_t slot = 0, phase = 0;  // ring slot and parity of the next tile consumed
    uint32_t qi = 0;               // non-empty items
    uint32_t tc = 0;               // KV tiles processed (all items)
    const uint32_t sR = smem_u32(smem + kOffRing);
    const bool two = hpi == 2;
    uint32_t qd[2][8], pd[2][8];
    kmajor_steps(smem_u32(smem + kOffQ), qd[0]);
    kmajor_steps(smem_u32(smem + kOffQ + kTileBytes), qd[1]);
    kmajor_steps(smem_u32(smem + kOffP), pd[0]);
    kmajor_steps(smem_u32(smem + kOffP + kTileBytes), pd[1]);
    // every lane tests the barrier; lane 0's outcome is the warp's
    auto wait_w = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __shfl_sync(0xffffffffu, wait_or_abort(bar, parity, s_abort) ? 1 : 0, 0) != 0;
    };
    auto next_slot = [&]() {
      if (++slot == kRing) {
        slot = 0;
        phase ^= 1u;
      }
    };
    // one head's products; the second (or only) head's commit releases the
    // ring slot
    auto qk_h = [&](uint32_t kslot, bool second, bool release, bool last_k) {
      uint32_t kb[8];
      kmajor_steps(sR + kslot * kTileBytes, kb);
      if (elect_one()) {
        if (second) {
          umma8_ss(tmem + kBN, qd[1], kb, kIdescQK, 0u);
          umma_commit(&s_full[1]);
        } else {
          umma8_ss(tmem, qd[0], kb, kIdescQK, 0u);
          umma_commit(&s_full[0]);
        }
        if (release) {
          umma_commit(&ring_empty[kslot]);
          if (last_k) umma_commit(q_empty);
        }
      }
      __syncwarp();
    };
    auto pv_h = [&](uint32_t vslot, bool second, bool release, uint32_t acc) {
      uint32_t vb[8];
      vmn_steps(sR + vslot * kTileBytes, vb);
      if (elect_one()) {
        if (second) {
          umma8_ss(tmem + 256 + kHeadDim, pd[1], vb, kIdescPV, acc);
          umma_commit(&pv_done[1]);
        } else {
          umma8_ss(tmem + 256, pd[0], vb, kIdescPV, acc);
          umma_commit(&pv_done[0]);
        }
        if (release) umma_commit(&ring_empty[vslot]);
      }
      __syncwarp();
    };
    int item = sched_item(S, s_list, 0);
    TileRaw raw = tile_raw_load(p, item_r0(p, item, items_per_tile), lane);
    for (int r = 0; item >= 0 && !*s_abort; item = sched_item(S, s_list, ++r)) {
      const int r0 = (item / items_per_tile) * kBM;
      int kv_lo, kv_hi;
      tile_key_range(raw, r0, lane, kv_lo, kv_hi);
      raw = tile_raw_load(p, item_r0(p, sched_item(S, s_list, r + 1), items_per_tile), lane);
      if (kv_hi <= kv_lo) continue;
      const int n_kv = (kv_hi - kv_lo + kBN - 1) / kBN;
      // K_0: S_h must have been read by the softmax of the previous tile
      bool ok = wait_w(q_full, qi & 1);
      uint32_t kslot = slot;
      ok = ok && wait_w(&ring_full[kslot], phase);
      next_slot();
      if (ok && tc > 0) ok = wait_w(&s_free[0], (tc - 1) & 1);
      if (ok) {
        tc_fence_after();
        qk_h(kslot, false, !two, n_kv == 1);
      }
      if (ok && two) {
        if (tc > 0) ok = wait_w(&s_free[1], (tc - 1) & 1);
        if (ok) {
          tc_fence_after();
          qk_h(kslot, true, true, n_kv == 1);
        }
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv) {
          // K_{j+1}: S of the next tile while this tile's softmax runs
          kslot = slot;
          ok = wait_w(&ring_full[kslot], phase);
          next_slot();
          ok = ok && wait_w(&s_free[0], tc & 1);
          if (!ok) break;
          tc_fence_after();
          qk_h(kslot, false, !two, j + 2 == n_kv);
          if (two) {
            ok = wait_w(&s_free[1], tc & 1);
            if (!ok) break;
            tc_fence_after();
            qk_h(kslot, true, true, j + 2 == n_kv);
          }
        }
        const uint32_t vslot = slot;
        ok = wait_w(&ring_full[vslot], phase);
        next_slot();
        ok = ok && wait_w(&p_full[0], tc & 1);
        // the first PV of an item overwrites O_h: its previous epilogue is done
        if (ok && j == 0 && qi > 0) ok = wait_w(&o_free[0], (qi - 1) & 1);
        if (!ok) break;
        tc_fence_after();
        pv_h(vslot, false, !two, j > 0 ? 1u : 0u);
        if (two) {
          ok = wait_w(&p_full[1], tc & 1);
          if (ok && j == 0 && qi > 0) ok = wait_w(&o_free[1], (qi - 1) & 1);
          if (!ok) break;
          tc_fence_after();
          pv_h(vslot, true, true, j > 0 ? 1u : 0u);
        }
        ++tc;
      }
      if (!ok) *s_abort = 1;
      ++qi;
    }
  } else {
    // ---------------------------------------------------- softmax rows ----
    const int grp = (warp - 2) >> 2;      // which head of the item
    const int lane_base = 32 * (warp & 3);
    const int row = lane_base + lane;
    const uint32_t t_s = tmem + (static_cast<uint32_t>(lane_base) << 16) + grp * kBN;
    const uint32_t t_o = tmem + (static_cast<uint32_t>(lane_base) << 16) + 256 + grp * kHeadDim;
    uint8_t* sP = smem + kOffP + grp * kTileBytes;
    const bool store_thread = (warp & 3) == 2 && lane == 0;  // first warp of the group
    uint32_t tc = 0, qi = 0, gs = 0;
    // all 128 threads of this warpgroup; bounded, warp-uniform outcome
    auto group_sync = [&]() -> bool {
      mbar_arrive(&grp_sync[grp]);
      const bool w = wait_or_abort(&grp_sync[grp], gs & 1, s_abort);
      ++gs;
      return __all_sync(0xffffffffu, w);
    };
    const bool active = grp < hpi;
    int item = sched_item(S, s_list, 0);
    TileRaw raw = tile_raw_load(p, item_r0(p, item, items_per_tile), lane);
    const int r0_first = item_r0(p, item, items_per_tile);
    RowRaw rr = row_raw_load(p, r0_first >= 0 ? r0_first + row : -1);
    for (int r = 0; active && item >= 0; item = sched_item(S, s_list, ++r)) {
      if (__any_sync(0xffffffffu, *s_abort != 0)) break;  // warp-uniform exit
      const int tile = item / items_per_tile;
      const int head = (item % items_per_tile) * hpi + grp;
      const int r0 = tile * kBM;
      int kv_lo, kv_hi;
      tile_key_range(raw, r0, lane, kv_lo, kv_hi);
      const int n_kv = (kv_hi > kv_lo) ? (kv_hi - kv_lo + kBN - 1) / kBN : 0;
      const int i = r0 + row;
      bool valid = false;
      int start = 0;
      if (i < p.n_tokens && rr.b != 0) {
        valid = true;
        bool okl = rr.pos >= 0 && rr.pos <= i;
        if (okl && rr.pos > 0) okl = (rr.b_prev == rr.b) && (rr.pos_prev == rr.pos - 1);
        if (!okl && grp == 0) set_dev_err(p.dev_err, PKV_DEV_ERR_LAYOUT);
        start = (rr.pos >= 0 && rr.pos <= i) ? i - rr.pos : i;
      }
      // next item's metadata, in flight while this item computes
      {
        const int r0n = item_r0(p, sched_item(S, s_list, r + 1), items_per_tile);
        raw = tile_raw_load(p, r0n, lane);
        rr = row_raw_load(p, r0n >= 0 ? r0n + row : -1);
      }
      float m_run = -INFINITY;  // running max, raw score units
      float l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < n_kv && ok; ++j) {
        // wait outcomes are warp-uniform: the TMEM accesses are warp-collective
        if (!__all_sync(0xffffffffu, wait_or_abort(&s_full[grp], tc & 1, s_abort))) {
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
          tmem_ld32(t_s + 0, a);
          tmem_ld32(t_s + 32, b);
          tmem_ld32(t_s + 64, c);
          tmem_ld32(t_s + 96, d);
          tmem_wait_ld();
        }
        // S_h is in registers: the next tile's QK may overwrite it
        tc_fence_before();
        mbar_arrive(&s_free[grp]);
        // columns [c_lo, c_hi] of this tile are visible to this row
        const int k0 = kv_lo + j * kBN;
        const int c_lo = max(start - k0, 0);
        const int c_hi = min(i - k0, kBN - 1);
        const bool none = !valid || c_lo > c_hi;
        const bool full = !none && c_lo == 0 && c_hi == kBN - 1;
        float mx = -INFINITY;
        if (!none) {
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          if (full) {
            m4[0] = row_max_full(sr);
          } else {
            const unsigned span = static_cast<unsigned>(c_hi - c_lo);
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
              const bool vis = static_cast<unsigned>(c - c_lo) <= span;
              const float v = vis ? __uint_as_float(sr[c]) : -INFINITY;
              sr[c] = __float_as_uint(v);
              m4[c & 3] = fmaxf(m4[c & 3], v);
            }
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
        // P and O of this head are free once its previous PV has completed
        const bool got = (j == 0) || wait_or_abort(&pv_done[grp], (tc - 1) & 1, s_abort);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (j == 0) {
          // the previous item's output store may still be reading this buffer
          if (store_thread) bulk_wait_read_all();
          if (!group_sync()) {
            ok = false;
            break;
          }
        }
        float psum = 0.f;
        if (none) {
          // nothing visible: a zero P row (masked keys contribute nothing)
#pragma unroll
          for (int q = 0; q < 16; ++q)
            *reinterpret_cast<uint4*>(sP + (q >> 3) * kHalf + row * 128 +
                                      (((q & 7) ^ (row & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
        } else {
          psum = softmax_row_to_p(sr, p.qscale, neg_m, sP, row);
        }
        l_run = l_run * alpha + psum;
        m_run = m_use;
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
          for (int c = 0; c < kHeadDim; c += 32) {
            uint32_t o[32];
            tmem_ld32(t_o + c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(t_o + c, o);
          }
          tmem_wait_st();
        }
        fence_proxy_async_smem();
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
      const bool in_range = i < p.n_tokens;
      const bool has = in_range && valid && ok && l_run > 0.f;
      const float inv = has ? 1.f / l_run : 0.f;
      if (n_kv > 0 && ok) {
        // O / l as bf16 into this head's P buffer (same swizzled layout; the
        // item's last PV has completed), then two TMA stores of 64 head dims
        // x 128 rows; rows past the end are clipped by the tensor map
        uint32_t o[128];
        {
          uint32_t (&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(&o[0]);
          uint32_t (&b)[32] = *reinterpret_cast<uint32_t(*)[32]>(&o[32]);
          uint32_t (&c)[32] = *reinterpret_cast<uint32_t(*)[32]>(&o[64]);
          uint32_t (&d)[32] = *reinterpret_cast<uint32_t(*)[32]>(&o[96]);
          tmem_ld32(t_o + 0, a);
          tmem_ld32(t_o + 32, b);
          tmem_ld32(t_o + 64, c);
          tmem_ld32(t_o + 96, d);
          tmem_wait_ld();
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          uint4 w = make_uint4(0u, 0u, 0u, 0u);
          if (has) {
            const int e = 8 * q;
            w.x = pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
          }
          *reinterpret_cast<uint4*>(sP + (q >> 3) * kHalf + row * 128 +
                                    (((q & 7) ^ (row & 7)) << 4)) = w;
        }
        fence_proxy_async_smem();
        const bool synced = group_sync();
        if (synced && store_thread) {
          tma_store_3d(&omap, sP, 0, head, r0);
          tma_store_3d(&omap, sP + kHalf, 64, head, r0);
          bulk_commit_group();
        }
        if (!synced) ok = false;
      } else if (in_range) {
        // no key range at all (padding-only tile) or an aborted item: zeros
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                              (static_cast<int64_t>(i) * p.num_q_heads + head) * kHeadDim;
#pragma unroll
        for (int c = 0; c < kHeadDim; c += 8)
          *reinterpret_cast<uint4*>(orow + c) = make_uint4(0u, 0u, 0u, 0u);
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
  if (warp >= 2 && (warp & 3) == 2 && lane == 0) bulk_wait_all();  // output stores done
  if (*s_abort && threadIdx.x == 0) set_dev_err(p.dev_err, PKV_DEV_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

using namespace prefill_host;

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

  CUtensorMap qmap, kmap, vmap, omap;
  if (!encode_packed_map(&qmap, q, num_q_heads, n_tokens) ||
      !encode_packed_map(&kmap, k, num_kv_heads, n_tokens) ||
      !encode_packed_map(&vmap, v, num_kv_heads, n_tokens) ||
      !encode_packed_map(&omap, out, num_q_heads, n_tokens))
    return PKV_ERR_ARG;

  static std::atomic<bool> attr_set[64] = {};  // per device; host threads may race to set it
  if (dev < 0 || dev >= 64) return PKV_ERR_DEVICE;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    const cudaError_t ea = cudaFuncSetAttribute(
        prefill_tcgen05_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (ea != cudaSuccess) return record_cuda_status(ea);
    attr_set[dev].store(true, std::memory_order_release);
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PKV_ERR_CUDA;
  PrefillParams prm;
  prm.batch_idx = batch_idx;
  prm.input_pos = input_pos;
  prm.out = out;
  prm.lse = lse;
  prm.dev_err = dev_err;
  prm.n_tokens = n_tokens;
  prm.num_q_heads = num_q_heads;
  prm.group = g;
  prm.heads_per_item = g >= 2 ? 2 : 1;
  prm.n_tiles = (n_tokens + kBM - 1) / kBM;
  prm.n_items = prm.n_tiles * (num_q_heads / prm.heads_per_item);
  prm.qscale = scale * 1.4426950408889634f;
  const int grid = prm.n_items < sms ? prm.n_items : sms;
  const cudaError_t e = launch_kernel(prefill_tcgen05_kernel, dim3(grid), dim3(kThreads),
                                      kSmemBytes, stream, false, qmap, kmap, vmap, omap, prm);
  return record_cuda_status(e);
}

}  // namespace pkv
