// pkv_prefill_common.cuh - what the two tcgen05 prefill kernels share: tile
// sizes, the tensor-memory layout, the MMA instruction descriptors, the
// softmax row (P into shared memory for the packed kernel, into tensor memory
// for the paged one), the bounded wait that honours a grid-wide abort flag,
// the cost-sorted item schedule, and the host-side cuTensorMapEncodeTiled
// lookup. Each kernel file lays out
// its own shared memory.
#pragma once

#include "pkv_launch.h"

namespace pkv {
namespace prefill_detail {

constexpr int kBM = 128;                 // query rows per tile
constexpr int kBN = 128;                 // keys per KV tile
constexpr int kHalf = 128 * 128;         // one [128 rows x 64 elems] bf16 block, bytes
constexpr int kTileBytes = 2 * kHalf;    // 128 x 128 bf16 (32 KB)
constexpr int kThreads = 10 * 32;
constexpr int kGroupThreads = 128;       // one softmax warpgroup
// TMEM columns: S0 S1 O0 O1, 128 each. Where P lives in TMEM, P_h (bf16
// pairs, 64 columns) is written over the first half of S_h once the softmax
// has read S_h.
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, /*b_mn_major=*/false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kHeadDim, /*b_mn_major=*/true);
constexpr int kMaxDynSmem = 232448;  // 227 KB opt-in limit per block

// D[tmem] (+)= A[tmem] * B[smem desc]: the A operand (M x K, bf16) is read
// from tensor memory, row m in lane m, two consecutive K elements packed per
// 32-bit column, so one K = 16 step spans 8 columns. Only A may come from
// tensor memory.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Shared-memory descriptors (tcgen05 format, as sw128_desc) split in 32-bit
// words. Every operand here has 8-row groups 1024 bytes apart and 128-byte
// swizzle, so the high word is one constant; the low word holds the start
// address (>> 4) and the leading byte offset.
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo >> 4) & 0x3FFFu) << 16);
}

// The eight K-steps of one 128 x 128 x 128 product, D (+)= sum_k A_k B_k, as
// eight tcgen05.mma from one asm block with nothing issued between them. The
// issuing warp shares its SM sub-partition with busy softmax warps; with the
// descriptor arithmetic done before the block, each MMA needs one issue slot
// and the tensor pipe is fed close to its rate (issued one by one with the
// arithmetic in between, a 128 x 128 x 16 MMA took ~150 cycles to issue
// against the 64 it executes in). a_lo/b_lo: low descriptor words per K-step
// (shared-memory A and B); the first MMA accumulates iff `accumulate`.
__device__ __forceinline__ void umma8_ss(uint32_t d, const uint32_t (&a_lo)[8],
                                         const uint32_t (&b_lo)[8], uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 a<8>, b<8>;\n\t"
      "setp.ne.b32 p0, %17, 0;\n\tsetp.eq.b32 p1, %17, %17;\n\t"
      "mov.b64 a0, {%1, %19};\n\tmov.b64 b0, {%9, %19};\n\t"
      "mov.b64 a1, {%2, %19};\n\tmov.b64 b1, {%10, %19};\n\t"
      "mov.b64 a2, {%3, %19};\n\tmov.b64 b2, {%11, %19};\n\t"
      "mov.b64 a3, {%4, %19};\n\tmov.b64 b3, {%12, %19};\n\t"
      "mov.b64 a4, {%5, %19};\n\tmov.b64 b4, {%13, %19};\n\t"
      "mov.b64 a5, {%6, %19};\n\tmov.b64 b5, {%14, %19};\n\t"
      "mov.b64 a6, {%7, %19};\n\tmov.b64 b6, {%15, %19};\n\t"
      "mov.b64 a7, {%8, %19};\n\tmov.b64 b7, {%16, %19};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a0, b0, %18, p0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %18, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %18, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %18, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a4, b4, %18, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a5, b5, %18, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a6, b6, %18, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a7, b7, %18, p1;\n\t}" ::"r"(d),
      "r"(a_lo[0]), "r"(a_lo[1]), "r"(a_lo[2]), "r"(a_lo[3]), "r"(a_lo[4]), "r"(a_lo[5]),
      "r"(a_lo[6]), "r"(a_lo[7]), "r"(b_lo[0]), "r"(b_lo[1]), "r"(b_lo[2]), "r"(b_lo[3]),
      "r"(b_lo[4]), "r"(b_lo[5]), "r"(b_lo[6]), "r"(b_lo[7]), "r"(accumulate), "r"(idesc),
      "n"(kDescHi)
      : "memory");
}

// The same with A read from tensor memory: K-step k takes its A operand at
// TMEM address a_tmem + 8k (bf16 pairs, 16 keys per 8 columns).
__device__ __forceinline__ void umma8_ts(uint32_t d, uint32_t a_tmem, const uint32_t (&b_lo)[8],
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p0, p1;\n\t.reg .b64 b<8>;\n\t.reg .b32 t<8>;\n\t"
      "setp.ne.b32 p0, %10, 0;\n\tsetp.eq.b32 p1, %10, %10;\n\t"
      "mov.b64 b0, {%2, %12};\n\tadd.u32 t0, %1, 0;\n\t"
      "mov.b64 b1, {%3, %12};\n\tadd.u32 t1, %1, 8;\n\t"
      "mov.b64 b2, {%4, %12};\n\tadd.u32 t2, %1, 16;\n\t"
      "mov.b64 b3, {%5, %12};\n\tadd.u32 t3, %1, 24;\n\t"
      "mov.b64 b4, {%6, %12};\n\tadd.u32 t4, %1, 32;\n\t"
      "mov.b64 b5, {%7, %12};\n\tadd.u32 t5, %1, 40;\n\t"
      "mov.b64 b6, {%8, %12};\n\tadd.u32 t6, %1, 48;\n\t"
      "mov.b64 b7, {%9, %12};\n\tadd.u32 t7, %1, 56;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], b0, %11, p0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t1], b1, %11, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t2], b2, %11, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t3], b3, %11, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t4], b4, %11, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t5], b5, %11, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t6], b6, %11, p1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t7], b7, %11, p1;\n\t}" ::"r"(d),
      "r"(a_tmem), "r"(b_lo[0]), "r"(b_lo[1]), "r"(b_lo[2]), "r"(b_lo[3]), "r"(b_lo[4]),
      "r"(b_lo[5]), "r"(b_lo[6]), "r"(b_lo[7]), "r"(accumulate), "r"(idesc), "n"(kDescHi)
      : "memory");
}

// Low descriptor words of the eight K-steps of a K-major 128 x 128 tile at
// `base` (two 16 KB halves of 64 elements; K-step k at half k / 4, 32 bytes
// per step within it).
__device__ __forceinline__ void kmajor_steps(uint32_t base, uint32_t (&lo)[8]) {
  const uint32_t b = desc_lo(base, 0);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) lo[kk] = b + ((((kk >> 2) * kHalf) + (kk & 3) * 32) >> 4);
}

// ... of an MN-major V tile at `base` used as the B operand of PV: K-step k
// (16 keys) starts 2 KB in; the two 64-dim halves are kHalf apart (LBO).
__device__ __forceinline__ void vmn_steps(uint32_t base, uint32_t (&lo)[8]) {
  const uint32_t b = desc_lo(base, kHalf);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) lo[kk] = b + ((kk * 2048) >> 4);
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}


__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Two fp32 lanes per instruction (Blackwell's paired FMA/ADD).
__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Maximum of a fully visible 128-column S row (three-input max, four chains).
__device__ __forceinline__ float row_max_full(const uint32_t (&sr)[128]) {
  float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int c = 0; c < 128; c += 8) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      m[k] = fmax3(m[k], __uint_as_float(sr[c + 2 * k]), __uint_as_float(sr[c + 2 * k + 1]));
  }
  return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// One softmax row of a 128-key tile: P = exp2(s * qscale - m) written as bf16
// into this row of the K-major 128-byte-swizzled P tile (16-byte chunk q at
// half q >> 3, position (q & 7) ^ (row & 7)); returns the row's sum of P in
// fp32. Masked columns hold -inf, which ex2.approx maps to +0 exactly. The
// scale-and-shift and the sum run two lanes per instruction: the softmax is
// bound by instruction issue, not by the exponential unit (moving a quarter
// of the exponentials to an FMA-pipe polynomial made the kernel 8 % slower).
__device__ __forceinline__ float softmax_row_to_p(const uint32_t (&sr)[128], float qscale,
                                                  float neg_m, uint8_t* sP, int row) {
  const unsigned long long qs2 = pack_f32x2(qscale, qscale);
  const unsigned long long nm2 = pack_f32x2(neg_m, neg_m);
  unsigned long long acc0 = 0ull, acc1 = 0ull;  // two paired partial sums (0.0f, 0.0f)
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    float e[8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const unsigned long long x2 = ffma2(
          pack_f32x2(__uint_as_float(sr[8 * q + 2 * u]), __uint_as_float(sr[8 * q + 2 * u + 1])),
          qs2, nm2);
      float x0, x1;
      unpack_f32x2(x2, x0, x1);
      e[2 * u] = ex2(x0);
      e[2 * u + 1] = ex2(x1);
    }
    acc0 = fadd2(acc0, fadd2(pack_f32x2(e[0], e[1]), pack_f32x2(e[2], e[3])));
    acc1 = fadd2(acc1, fadd2(pack_f32x2(e[4], e[5]), pack_f32x2(e[6], e[7])));
    *reinterpret_cast<uint4*>(sP + (q >> 3) * kHalf + row * 128 + (((q & 7) ^ (row & 7)) << 4)) =
        make_uint4(pack_bf16x2(e[0], e[1]), pack_bf16x2(e[2], e[3]), pack_bf16x2(e[4], e[5]),
                   pack_bf16x2(e[6], e[7]));
  }
  float a, b, c, d;
  unpack_f32x2(acc0, a, b);
  unpack_f32x2(acc1, c, d);
  return (a + b) + (c + d);
}

// The same row with P written to tensor memory: bf16 pairs into 64 columns of
// this thread's TMEM lane starting at t_p (keys 2c and 2c + 1 in column c,
// the A-operand layout of a PV product read from tensor memory); returns the
// row's sum of P in fp32. A row with every column masked (-inf) writes a zero
// P row. Every lane of the warp must call it (the TMEM store is
// warp-collective).
__device__ __forceinline__ float softmax_row_to_tmem(const uint32_t (&sr)[128], float qscale,
                                                     float neg_m, uint32_t t_p) {
  const unsigned long long qs2 = pack_f32x2(qscale, qscale);
  const unsigned long long nm2 = pack_f32x2(neg_m, neg_m);
  unsigned long long acc0 = 0ull, acc1 = 0ull;  // two paired partial sums (0.0f, 0.0f)
#pragma unroll
  for (int c = 0; c < 4; ++c) {  // 32 keys -> 16 columns
    uint32_t pk[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int k0 = 32 * c + 8 * q;
      float e[8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const unsigned long long x2 = ffma2(
            pack_f32x2(__uint_as_float(sr[k0 + 2 * u]), __uint_as_float(sr[k0 + 2 * u + 1])),
            qs2, nm2);
        float x0, x1;
        unpack_f32x2(x2, x0, x1);
        e[2 * u] = ex2(x0);
        e[2 * u + 1] = ex2(x1);
      }
      acc0 = fadd2(acc0, fadd2(pack_f32x2(e[0], e[1]), pack_f32x2(e[2], e[3])));
      acc1 = fadd2(acc1, fadd2(pack_f32x2(e[4], e[5]), pack_f32x2(e[6], e[7])));
#pragma unroll
      for (int u = 0; u < 4; ++u) pk[4 * q + u] = pack_bf16x2(e[2 * u], e[2 * u + 1]);
    }
    tmem_st16(t_p + 16 * c, pk);
  }
  float a, b, c, d;
  unpack_f32x2(acc0, a, b);
  unpack_f32x2(acc1, c, d);
  return (a + b) + (c + d);
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Item schedule of the persistent paged-prefill grid. An item is (query tile,
// head group); its cost is mostly its number of key tiles, which varies
// several-fold across the tiles of a step (a chunk over a 4 K prefix against
// one over 512 keys). Dealt round-robin, the busiest CTA of 16 chunks of 512
// tokens over prefixes U[512, 4096] carries 1.27x the mean load. Sorting
// tiles by cost alone brings that to 1.02x but scatters the tiles of one
// sequence, which share its K/V in L2, over the whole call (the mean CTA time
// grew 7 %). So tiles are grouped: consecutive tiles that continue one run of
// equal slots form a group, groups are sorted by their largest tile cost,
// largest first (a stable counting sort, identical in every CTA), and a
// group's tiles follow each other, last (costliest) tile first. The items in
// that order (a tile's head groups side by side) are dealt in snake order:
// round r gives position r*G + b to CTA b, reversed in odd rounds. The
// estimate only orders the work; which CTA computes an item changes nothing
// in its result. Calls with more than kSchedMaxTiles query tiles are dealt
// round-robin.
constexpr int kSchedMaxTiles = 768;
constexpr int kSchedListMax = 768;                 // this CTA's items + end mark
constexpr int kSchedBytes = kSchedListMax * 2;     // uint16 item list
constexpr int kSchedMaxCost = 255;
constexpr uint16_t kSchedEnd = 0xFFFFu;
// transient scratch (in the K/V ring, before any load): 256 bins, per tile
// its cost, its link to the next tile and its group's sort key, then the
// tile order
constexpr int kSchedScratchBytes = 1024 + 3 * kSchedMaxTiles + 2 * kSchedMaxTiles;

// listed: this CTA's items are list[0..] up to kSchedEnd; else round-robin
struct ItemSched {
  bool listed;
  int n_items;
};

// This CTA's r-th item (r = 0, 1, ... up to one past its last), or -1.
__device__ __forceinline__ int sched_item(const ItemSched& s, const uint16_t* list, int r) {
  if (s.listed) {
    const uint16_t v = list[r];
    return v == kSchedEnd ? -1 : static_cast<int>(v);
  }
  const long long it = static_cast<long long>(r) * gridDim.x + blockIdx.x;
  return it < s.n_items ? static_cast<int>(it) : -1;
}

// A sorted schedule needs at most kSchedMaxTiles tiles and item indices
// below the end mark, and this CTA's list must fit.
__device__ __forceinline__ bool sched_fits(int n_tiles, int n_items) {
  const int g = static_cast<int>(gridDim.x);
  return n_tiles > 1 && n_tiles <= kSchedMaxTiles && n_items < kSchedEnd &&
         (n_items + g - 1) / g < kSchedListMax;
}

// Warp 0: this CTA's items (position r*G + b of the ordered items in even
// rounds, r*G + G-1-b in odd ones, a tile's head groups side by side), then
// the end mark.
__device__ __forceinline__ void sched_fill_list(uint16_t* list, const uint16_t* order,
                                                int n_items, int items_per_tile, int lane) {
  const int g = static_cast<int>(gridDim.x);
  const int b = static_cast<int>(blockIdx.x);
  for (int r = lane; r < kSchedListMax; r += 32) {
    const long long pos = static_cast<long long>(r) * g + ((r & 1) ? g - 1 - b : b);
    uint16_t v = kSchedEnd;
    if (pos < n_items) {
      const int ps = static_cast<int>(pos);
      v = static_cast<uint16_t>(static_cast<int>(order[ps / items_per_tile]) * items_per_tile +
                                ps % items_per_tile);
    }
    list[r] = v;
    if (__all_sync(0xffffffffu, v == kSchedEnd)) break;
  }
}

// Called by every thread of the CTA (it holds block barriers). cost(t) is the
// estimated cost of tile t (clamped to [0, kSchedMaxCost]); link(t) says that
// tile t + 1 continues tile t's last run (t + 1 < n_tiles). scratch holds
// kSchedScratchBytes that nothing else uses until this returns; list gets
// this CTA's items.
template <class CostFn, class LinkFn>
__device__ ItemSched sched_build(uint16_t* list, uint8_t* scratch, int n_tiles,
                                 int items_per_tile, CostFn cost, LinkFn link) {
  ItemSched s;
  s.listed = false;
  s.n_items = n_tiles * items_per_tile;
  if (!sched_fits(n_tiles, s.n_items)) return s;
  int* hist = reinterpret_cast<int*>(scratch);     // [256], bin = kSchedMaxCost - key
  uint8_t* tcost = scratch + 1024;                 // [n_tiles]
  uint8_t* tlink = tcost + kSchedMaxTiles;         // [n_tiles]
  uint8_t* bin = tlink + kSchedMaxTiles;           // [n_tiles]
  uint16_t* order = reinterpret_cast<uint16_t*>(bin + kSchedMaxTiles);  // [n_tiles]
  for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
  for (int t = threadIdx.x; t < n_tiles; t += blockDim.x) {
    tcost[t] = static_cast<uint8_t>(min(max(cost(t), 0), kSchedMaxCost));
    tlink[t] = (t + 1 < n_tiles && link(t)) ? 1 : 0;
  }
  __syncthreads();
  // the first tile of each group finds the group's largest cost and gives
  // every tile of the group that key
  for (int t = threadIdx.x; t < n_tiles; t += blockDim.x) {
    if (t > 0 && tlink[t - 1]) continue;
    int e = t, mx = tcost[t];
    while (tlink[e]) mx = max(mx, static_cast<int>(tcost[++e]));
    for (int u = t; u <= e; ++u) bin[u] = static_cast<uint8_t>(kSchedMaxCost - mx);
    atomicAdd(&hist[kSchedMaxCost - mx], e - t + 1);
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    // exclusive scan of the bins: each lane holds eight consecutive bins
    int v[8], sum = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[k] = hist[8 * lane + k];
      sum += v[k];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - sum;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      hist[8 * lane + k] = run;
      run += v[k];
    }
    __syncwarp();
    // stable placement, 32 tiles a pass from the last tile down: lanes with
    // equal keys take consecutive places after the bin's running offset
    for (int c0 = 0; c0 < n_tiles; c0 += 32) {
      const int t = n_tiles - 1 - (c0 + lane);
      const bool valid = t >= 0;
      const int k = valid ? static_cast<int>(bin[t]) : 256 + lane;
      const uint32_t peers = __match_any_sync(0xffffffffu, k);
      const int leader = __ffs(peers) - 1;
      int base = (valid && lane == leader) ? hist[k] : 0;
      base = __shfl_sync(0xffffffffu, base, leader);
      if (valid) order[base + __popc(peers & ((1u << lane) - 1u))] = static_cast<uint16_t>(t);
      __syncwarp();
      if (valid && lane == leader) hist[k] = base + __popc(peers);
      __syncwarp();
    }
    sched_fill_list(list, order, s.n_items, items_per_tile, lane);
  }
  __syncthreads();
  s.listed = true;
  return s;
}

// Packed documents: the tiles of one document are spread over the packing's
// order, and tiles that share a document's K/V run close together when the
// order is kept; sorting all tiles by cost scatters them (the mean CTA time
// grew 10 %). Here the tiles are sorted by cost within consecutive windows of
// `window` tiles (eight rounds of items), so each window's K/V stays in L2
// while its items are balanced. O(n_tiles * window) comparisons in all.
template <class CostFn>
__device__ ItemSched sched_build_windowed(uint16_t* list, uint8_t* scratch, int n_tiles,
                                          int items_per_tile, int window, CostFn cost) {
  ItemSched s;
  s.listed = false;
  s.n_items = n_tiles * items_per_tile;
  if (!sched_fits(n_tiles, s.n_items) || window < 2) return s;
  uint8_t* tcost = scratch;                                              // [n_tiles]
  uint16_t* order = reinterpret_cast<uint16_t*>(scratch + kSchedMaxTiles);  // [n_tiles]
  for (int t = threadIdx.x; t < n_tiles; t += blockDim.x)
    tcost[t] = static_cast<uint8_t>(min(max(cost(t), 0), kSchedMaxCost));
  __syncthreads();
  // rank within the window: larger cost first, ties in tile order
  for (int t = threadIdx.x; t < n_tiles; t += blockDim.x) {
    const int w0 = (t / window) * window;
    const int w1 = min(w0 + window, n_tiles);
    const int c = tcost[t];
    int rank = w0;
    for (int u = w0; u < w1; ++u) {
      const int cu = tcost[u];
      rank += (cu > c || (cu == c && u < t)) ? 1 : 0;
    }
    order[rank] = static_cast<uint16_t>(t);
  }
  __syncthreads();
  if (threadIdx.x < 32) sched_fill_list(list, order, s.n_items, items_per_tile, threadIdx.x);
  __syncthreads();
  s.listed = true;
  return s;
}

}  // namespace prefill_detail

namespace prefill_host {

inline bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
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
inline bool encode_packed_map(CUtensorMap* map, const void* base, int heads, int n_tokens) {
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

}  // namespace prefill_host
}  // namespace pkv
