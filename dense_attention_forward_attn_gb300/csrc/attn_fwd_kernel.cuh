// attn_fwd_kernel.cuh -- the dense, non-causal, BF16, head_dim-128 attention
// forward for sm_103a: O = softmax(scale * Q K^T) V and the natural-log LSE.
//
// Design (from "B200 Attention Kernel from Scratch to Near-SOTA in 60 Diagrams",
// re-targeted to GB300):
//   * Chapter 1 / 5: a work item is (batch*head, a pair of 128-row Q tiles); the
//     KV loop over 128-row K/V tiles runs inside the CTA; each Q tile keeps its
//     own S/P and O in tensor memory (TMEM: S0 | S1 | O0 | O1 = 512 columns).
//   * Chapter 2 / 10: P is written back into TMEM as packed BF16 pairs over the
//     upper half of its S region and feeds the P*V tcgen05.mma as the A operand.
//   * Chapter 3: Q/K/V are staged by TMA with 128-byte swizzle; Q and K are
//     K-major operands, V is the MN-major B operand of P*V.
//   * Chapter 4 / 5 / 12: warp roles -- two softmax warpgroups (one per Q tile),
//     one correction warpgroup (conditional O rescale), one TMA warp and one
//     MMA-issuing warp; handoffs use mbarriers only.  As in the pages, the
//     correction warpgroup also runs the item epilogue (O read out of TMEM,
//     scaled by 1 / row sum, O and LSE stored), so the softmax warpgroups go on
//     with the next item meanwhile; the general mode and the two parts of an
//     item split between CTAs leave it to the stage's softmax warpgroup.
//   * Chapter 6: a ring of KV_STAGES shared slots, each holding one K or one V
//     tile; token t and t+KV_STAGES share a slot; a K token is released after
//     the last Q tile's Q*K^T, a V token after the last Q tile's P*V.
//   * Chapter 7: the MMA order per tile is P_qV(i) then Q_qK(i+1); the stream
//     continues across work items (Chapter 14), so the next item's first Q*K^T
//     is issued as soon as its Q tile and first K tile are resident.
//   * Chapter 8: base-2 exponentials with the scale folded into log2(e), the row
//     max taken on raw scores, ex2.approx.ftz.
//   * Chapter 9 (optional, ATTN_FLAG_SOFT_EXP2; a second instantiation of the
//     kernel): 4 of every 16 P columns take a polynomial exp2 on the FMA and
//     integer pipes instead of MUFU.  On GB300 the default all-MUFU path is
//     faster (MUFU does 32 exp2 per cycle per SM), so it is off by default.
//   * Chapter 11: the kept row max is replaced only when a tile's max exceeds it
//     by at least 8 (base-2 units); otherwise P is taken against the stale max.
//   * Chapter 13 splits P*V to start it before all of P is written; here P*V is
//     issued whole once P is complete and the MMA-issuing warp waits once for P
//     (and V, polled together) instead of twice: each mbarrier wait costs it ~130
//     cycles (measured +2 to +5% end to end).
//   * Chapter 14: persistent CTAs, one per SM, static stride over work items;
//     barriers are initialised once and their phases carried across items.
// LSE = (kept max + log2(row sum)) * ln 2 ("Attention for sm90, Line by Line",
// the exp2 question: the residual is stored in natural-log units).
//
// Every mbarrier wait is bounded in time: on expiry the CTA records a status
// bit in a device word, stops issuing work, waits for its own copies and MMAs in
// flight, frees TMEM and exits.
#pragma once
#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"

#ifndef ATTN_KV_STAGES
#define ATTN_KV_STAGES 3
#endif
#ifndef ATTN_L2_PREFETCH
#define ATTN_L2_PREFETCH 2   // K/V tiles prefetched into L2 ahead of the ring's loads
#endif
// 1: one elected lane per warp arrives on the consumer barriers (counts per warp);
// 0: every thread arrives (counts per thread).
#ifndef ATTN_ARRIVE_PER_WARP
#define ATTN_ARRIVE_PER_WARP 1
#endif


namespace attn {

constexpr int kBlockM = 128;   // rows of a Q tile
constexpr int kBlockN = 128;   // rows of a K/V tile
constexpr int kHeadDim = 128;
constexpr int kKvStages = ATTN_KV_STAGES;
constexpr int kThreads = 512;
constexpr uint32_t kTileBytes = kBlockM * kHeadDim * 2;   // 32 KiB
constexpr uint32_t kSlabBytes = kTileBytes / 2;           // 128 rows x 64 columns (128 B rows)
constexpr float kRebaseThresholdLog2 = 8.0f;
constexpr uint32_t kArrivePerWG = ATTN_ARRIVE_PER_WARP ? 4u : 128u;   // arrivals per warpgroup

// Warp roles.
constexpr int kCorrWarp0 = 8;
constexpr int kLoadWarp = 12;
constexpr int kMmaWarp = 13;

// Register split (setmaxnreg): 2 softmax WGs + correction WG + misc WG.
// (kRegSoftmax * 2 + kRegCorr + kRegMisc) * 128 threads must equal
// 65536 = kThreads * 128 (the registers the block is launched with).  The softmax warps hold a
// full 128-column score row; the correction and TMA/MMA roles work in 16-column chunks.
#ifndef ATTN_REG_SOFTMAX
#define ATTN_REG_SOFTMAX 200
#define ATTN_REG_CORR 56
#define ATTN_REG_MISC 56
#endif
constexpr uint32_t kRegSoftmax = ATTN_REG_SOFTMAX;
constexpr uint32_t kRegCorr = ATTN_REG_CORR;
constexpr uint32_t kRegMisc = ATTN_REG_MISC;
static_assert((kRegSoftmax * 2 + kRegCorr + kRegMisc) * 128 == 65536, "register split");

// TMEM columns.
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_s(int q) { return q ? 128u : 0u; }
__host__ __device__ constexpr uint32_t col_o(int q) { return q ? 384u : 256u; }
constexpr uint32_t kColP = 64;   // packed P sits over S columns 64..127 of its stage
// The CTA allocates all 512 columns, so its allocation starts at lane 0, column 0.  MMA
// operands use this constant (checked after the allocation) so the issuing code keeps them in
// warp-uniform registers.
constexpr uint32_t kTmemBase = 0;

// Kernel modes (template argument kMode): which cases an instantiation carries code for.
//   kModeFull:    dense launches with nothing masked or ragged (Sq a multiple of 256, Sk of 128,
//                 a non-zero scale, a 32-byte-aligned output): every work item has two Q tiles
//                 over the same KV tiles.  Built with the split schedule only (a launch without
//                 split items runs it with an empty split part).
//   kModeCausal:  the same launches with the causal mask: masking on the diagonal tile only,
//                 stages of unequal length.
//   kModeGeneral: everything (ragged lengths, zero scale, one-Q-tile items, 16-byte output
//                 stores, the failure-path test hook).
// Code that a launch never runs still costs this kernel (instruction fetch), so each launch
// takes the leanest mode that covers it.
constexpr int kModeFull = 0, kModeCausal = 1, kModeGeneral = 2;

// Device status bits (bounded waits that expired, by role).
constexpr unsigned kStatusTimeoutLoad = 1u << 0;
constexpr unsigned kStatusTimeoutMma = 1u << 1;
constexpr unsigned kStatusTimeoutSoftmax = 1u << 2;
constexpr unsigned kStatusTimeoutCorrection = 1u << 3;
constexpr unsigned kStatusTimeoutDrain = 1u << 4;
constexpr unsigned kStatusTmemBase = 1u << 5;   // allocation did not start at column 0
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per wait
constexpr uint64_t kDrainLimitNs = 200000000ull;   // 0.2 s for own in-flight work

struct alignas(8) SmemCtl {
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[kKvStages], kv_empty[kKvStages];
  uint64_t s_full[2];      // MMA -> softmax: S_q(i) in TMEM
  uint64_t p_full[2];      // softmax (P in TMEM) + correction (O rescaled or untouched) -> MMA
  uint64_t stats_full[2];  // softmax -> correction: per-row rescale factor published
  uint64_t o_full[2];      // MMA -> epilogue: last P*V of the item done (O final in TMEM)
  uint64_t fin_full[2][2]; // softmax -> correction: an item's final row statistics, per fin
                           // slot (a stage's softmax can finish two short items before the
                           // correction reads the first: one barrier per slot keeps each
                           // barrier at most one phase ahead of its waiter)
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort_flag;
  int sk_range[2];              // split schedule: this CTA's (item, KV tile) units [a, b)
  float alpha[2][2][kBlockM];   // [stage][tile parity][row]
  float2 fin[2][2][kBlockM];    // [stage][item parity][row]: 1 / row sum, LSE
};

constexpr uint32_t kCtlOffset = (2 + kKvStages) * kTileBytes;
constexpr uint32_t kSmemBytes = kCtlOffset + sizeof(SmemCtl) + 1024;   // +1 KiB for alignment

struct Params {
  void* o;          // BF16 output, [B,H,Sq,128] or [B,Sq,H,128] (strides below)
  float* lse;       // fp32 [B,H,Sq] or null
  int heads;        // H
  int bshd;         // 1: Q/K/V/O are [B,S,H,D]; 0: [B,H,S,D]
  int64_t o_row_stride;   // elements between consecutive query rows of one head
  int64_t o_head_stride;  // elements between heads
  int64_t o_batch_stride; // elements between batches
  int sq;
  int q_tiles;      // ceil(Sq / 128)
  int kv_tiles;     // ceil(Sk / 128)
  int kv_valid_last;  // valid key rows in the last KV tile, 1..128
  int pairs_per_head;
  int num_items;
  int bh;           // B * H
  int causal;       // query i attends keys j <= i (top-left aligned)
  float scale_log2; // scale * log2(e)
  int o_align32;     // o is 32-byte aligned (256-bit stores)
  int test_withhold;  // test hook: CTA 0's TMA warp never loads its first K tile, so the MMA
                      // warp's bounded wait on it expires (exercises the failure path)
  // Split schedule (the kernel's kSplit instantiation): items before sk_item0 (a multiple of the
  // grid) run whole by static stride; the remaining sk_items are cut by KV range so that every
  // CTA gets the same number of (item, KV tile) units.  An item whose KV range is shared by two
  // CTAs leaves a partial result of each part in the workspace; the second to finish combines.
  int sk_item0;
  int sk_items;
  float* ws_o;                  // [slot][part][stage][32 chunks][128 rows][4] fp32: O / l
  float* ws_l;                  // [slot][part][stage][128 rows] fp32: kept max + log2 l
  unsigned long long* ws_flag;  // [slot][stage][warp]: seq of the call whose part arrived
  unsigned long long seq;       // unique per call: flags from earlier calls never match it
};

struct WorkItem {
  int bh;       // flattened batch*head
  int qt0;      // first Q tile of the pair
  int n[2];     // KV tiles attended by Q tile qt0 + q (0: the pair has no second Q tile)
};

// Work item -> (bh, Q-tile pair, KV tiles per Q tile).  Dense: consecutive items walk the Q
// pairs of one head (its K/V stays hot in L2).  Causal: the work of a pair grows with its
// position, so items are numbered heaviest first (last pair of every head, then the one before).
__host__ __device__ inline WorkItem decode_item(int item, int pairs_per_head, int q_tiles,
                                                int kv_tiles, int bh_count, bool causal) {
  WorkItem w;
  int pair;
  if (causal) {
    pair = pairs_per_head - 1 - item / bh_count;
    w.bh = item - (item / bh_count) * bh_count;
  } else {
    w.bh = item / pairs_per_head;
    pair = item - w.bh * pairs_per_head;
  }
  w.qt0 = 2 * pair;
  const int t1 = w.qt0 + 1;
  const int c0 = w.qt0 + 1 < kv_tiles ? w.qt0 + 1 : kv_tiles;
  const int c1 = t1 + 1 < kv_tiles ? t1 + 1 : kv_tiles;
  w.n[0] = causal ? c0 : kv_tiles;
  w.n[1] = t1 < q_tiles ? (causal ? c1 : kv_tiles) : 0;
  return w;
}

__device__ __forceinline__ WorkItem decode_item(int item, const Params& p) {
  return decode_item(item, p.pairs_per_head, p.q_tiles, p.kv_tiles, p.bh, p.causal != 0);
}

// The item a persistent CTA runs in its round-th turn, or -1 when it has none left.  Dense:
// static stride (work_id += gridDim.x).  Causal: every other round runs in reverse CTA order,
// so the heaviest-first numbering spreads evenly over the CTAs.
__host__ __device__ inline int item_of(int round, int cta, int grid, int num_items, bool causal) {
  const int k = round * grid + ((causal && (round & 1)) ? grid - 1 - cta : cta);
  return k < num_items ? k : -1;
}

// Split schedule: CTA `cta` owns units [U*cta/grid, U*(cta+1)/grid) of the U = sk_items * n
// (item, KV tile) units of the split part, item-major.  Every CTA owns at least n units
// (sk_items > grid), so an item is shared by at most two CTAs: the head part (KV tiles [0, x))
// ends the range of CTA s, the tail part (KV tiles [x, n)) starts the range of CTA s + 1, and s
// is the split's slot.  Segment k of a CTA's range: item (local to the split part), first KV
// tile and KV tile count; false when the range has fewer segments.
// The host enables the split only where U * grid fits in 31 bits.
__host__ __device__ inline int split_range_begin(int cta, int grid, int sk_items, int n) {
  return static_cast<int>(static_cast<int64_t>(sk_items) * n * cta / grid);
}
// Segment k of the range [a, b) (from split_range_begin of this CTA and the next).
__host__ __device__ inline bool split_segment_of_range(int k, int a, int b, int n, int& item_local,
                                                       int& j0, int& cnt) {
  const int it = a / n + k;
  const int start = k == 0 ? a : it * n;
  if (start >= b) return false;
  const int end = b < (it + 1) * n ? b : (it + 1) * n;
  item_local = it;
  j0 = start - it * n;
  cnt = end - start;
  return true;
}
__host__ __device__ inline bool split_segment(int k, int cta, int grid, int sk_items, int n,
                                              int& item_local, int& j0, int& cnt) {
  return split_segment_of_range(k, split_range_begin(cta, grid, sk_items, n),
                                split_range_begin(cta + 1, grid, sk_items, n), n, item_local, j0,
                                cnt);
}

// One turn of a persistent CTA: a whole work item, or one part of an item split by KV range.
struct Seg {
  WorkItem w;   // n[q]: KV tiles of this segment for Q tile qt0 + q
  int j0;       // first KV tile of the segment
  int slot;     // -1: the whole item; else the index of the split
  int part;     // 0: the item's KV tiles [0, x); 1: its KV tiles [x, n)
};

// sk_range: this CTA's unit range [a, b) of the split part (set once per CTA, in shared memory).
template <bool kSplit>
__device__ __forceinline__ bool seg_of(int r, const Params& p, const int* sk_range, Seg& s) {
  const int cta = static_cast<int>(blockIdx.x), grid = static_cast<int>(gridDim.x);
  s.j0 = 0;
  s.slot = -1;
  s.part = 0;
  if (!kSplit || r * grid < p.sk_item0) {
    const int item = item_of(r, cta, grid, p.num_items, p.causal != 0);
    if (item < 0) return false;
    s.w = decode_item(item, p);
    return true;
  }
  int il, j0, cnt;
  if (!split_segment_of_range(r - p.sk_item0 / grid, sk_range[0], sk_range[1], p.kv_tiles, il, j0,
                              cnt))
    return false;
  s.w = decode_item(p.sk_item0 + il, p);
  s.w.n[0] = cnt;
  if (s.w.n[1] > 0) s.w.n[1] = cnt;
  s.j0 = j0;
  if (cnt < p.kv_tiles) {
    s.part = j0 > 0 ? 1 : 0;
    s.slot = j0 > 0 ? cta - 1 : cta;
  }
  return true;
}

// tcgen05 shared-memory matrix descriptor, 128-byte swizzle.
//   bits  0-13  start address >> 4      bits 16-29  leading byte offset >> 4
//   bits 32-45  stride byte offset >> 4 bits 46-48  fixed 0b001
//   bits 49-51  base offset (0: tiles are 1024-byte aligned)
//   bits 61-63  swizzle mode (2 = 128-byte)
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, .kind::f16 with BF16 A/B and FP32 accumulate.
//   bits 4-5 D format (1 = F32), 7-9 A format (1 = BF16), 10-12 B format (1 = BF16),
//   bit 15 A major (0 = K), bit 16 B major (1 = MN), bits 17-22 N >> 3, bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t make_idesc_bf16(uint32_t m, uint32_t n, uint32_t b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major << 16) | ((n >> 3) << 17) |
         ((m >> 4) << 24);
}

__device__ unsigned int g_attn_status = 0;

struct Ctx {
  SmemCtl* ctl;
  uint32_t smem_base;   // 1024-aligned shared address of Q0
  uint32_t tmem;        // TMEM base address
  uint32_t warp;
  uint32_t lane;

  __device__ uint32_t bar(const uint64_t& b) const { return ptx::smem_u32(&b); }
  __device__ uint32_t sq(int q) const { return smem_base + q * kTileBytes; }
  __device__ uint32_t skv(int s) const { return smem_base + (2 + s) * kTileBytes; }

  // Arrival of this warp's share on a barrier counted per warpgroup (kArrivePerWG).
  // Callers order their own shared-memory / tcgen05 writes before the call.
  __device__ void arrive(const uint64_t& b) const {
#if ATTN_ARRIVE_PER_WARP
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar(b));
#else
    ptx::mbar_arrive(bar(b));
#endif
  }

  // Warp-uniform bounded wait; all 32 lanes call it.  false = timed out or aborted.
  __device__ bool wait(const uint64_t& b, uint32_t parity, unsigned role_bit) const {
    const uint32_t addr = bar(b);
    if (__builtin_expect(__all_sync(0xffffffffu, ptx::mbar_try_wait(addr, parity)), 1)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
      if (__all_sync(0xffffffffu, ptx::mbar_try_wait(addr, parity))) return true;
      const bool stop = ctl->abort_flag != 0 || (ptx::globaltimer_ns() - t0) > kWaitLimitNs;
      if (__any_sync(0xffffffffu, stop)) {
        if (lane == 0) {
          ctl->abort_flag = 1;
          atomicOr(&g_attn_status, role_bit);
        }
        __syncwarp();
        return false;
      }
    }
  }

  // Two barriers at once: both try_waits are in flight together, so their latencies overlap.
  __device__ bool wait2(const uint64_t& b1, uint32_t par1, const uint64_t& b2, uint32_t par2,
                        unsigned role_bit) const {
    const uint32_t a1 = bar(b1), a2 = bar(b2);
    {
      const uint32_t r1 = ptx::mbar_try_wait(a1, par1);
      const uint32_t r2 = ptx::mbar_try_wait(a2, par2);
      if (__builtin_expect(__all_sync(0xffffffffu, r1 & r2), 1)) return true;
    }
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
      const uint32_t r1 = ptx::mbar_try_wait(a1, par1);
      const uint32_t r2 = ptx::mbar_try_wait(a2, par2);
      if (__all_sync(0xffffffffu, r1 & r2)) return true;
      const bool stop = ctl->abort_flag != 0 || (ptx::globaltimer_ns() - t0) > kWaitLimitNs;
      if (__any_sync(0xffffffffu, stop)) {
        if (lane == 0) {
          ctl->abort_flag = 1;
          atomicOr(&g_attn_status, role_bit);
        }
        __syncwarp();
        return false;
      }
    }
  }

  // Bounded wait on this warp's own in-flight work, ignoring the abort flag.
  __device__ void drain_wait(const uint64_t& b, uint32_t parity) const {
    const uint32_t addr = bar(b);
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!__all_sync(0xffffffffu, ptx::mbar_try_wait(addr, parity))) {
      if (__any_sync(0xffffffffu, (ptx::globaltimer_ns() - t0) > kDrainLimitNs)) {
        if (lane == 0) atomicOr(&g_attn_status, kStatusTimeoutDrain);
        return;
      }
    }
  }
};

// ------------------------------------------------------------------ TMA warp
// kBshd: the layout is a template parameter, so each instantiation's TMA warp holds only its own
// tensor-map rank (a run-time layout branch in the box loads measured up to 3% slower).
template <bool kSplit, bool kBshd, int kMode>
__device__ __forceinline__ void load_role(const Ctx& c, const Params& p, const CUtensorMap* tm_q,
                                          const CUtensorMap* tm_k, const CUtensorMap* tm_v) {
  SmemCtl* ctl = c.ctl;
  int slot = 0;
  uint32_t phase = 0;          // phase of the kv ring round being filled
  uint32_t kv_used = 0;        // bit s: slot s received a load
  uint32_t kv_last_par = 0;    // bit s: phase parity of the last load into slot s
  uint32_t q_cnt[2] = {0, 0};  // Q loads issued per stage
  bool ok = true;

  // Q/K/V tensor maps: 3-D (D, S, B*H) for [B,H,S,D] inputs, 4-D (D, H, S, B) for [B,S,H,D].
  // A box is 64 columns x 128 rows of one head either way (the same swizzled SMEM tile).
  auto load_box = [&](uint32_t dst, const CUtensorMap* tm, uint32_t fb, int col, int row, int bh) {
    if (kBshd) {
      const int b = bh / p.heads, h = bh - b * p.heads;
      ptx::tma_load_4d(dst, tm, fb, col, h, row, b);
    } else {
      ptx::tma_load_3d(dst, tm, fb, col, row, bh);
    }
  };
  // Q tiles, read once, are marked first to evict from L2 so they do not push K/V lines out
  // (re-read by every item of a head).  Causal mode, where the heaviest-first order keeps every
  // head's K/V in use for the whole launch (128 MiB at S=4K, B=4, H=16): +1.0% at causal S=4K,
  // +0.6% at S=16K; full-tile mode, with O stored the same way: +0.0 / +0.6 / +0.6% at
  // S=4K/8K/16K.
  auto load_q_box = [&](uint32_t dst, uint32_t fb, int col, int row, int bh) {
    if (kMode == kModeGeneral) {
      load_box(dst, tm_q, fb, col, row, bh);
    } else if (kBshd) {
      const int b = bh / p.heads, h = bh - b * p.heads;
      ptx::tma_load_4d_hint(dst, tm_q, fb, col, h, row, b, ptx::l2_policy_evict_first());
    } else {
      ptx::tma_load_3d_hint(dst, tm_q, fb, col, row, bh, ptx::l2_policy_evict_first());
    }
  };
  // L2 prefetch of a K or V tile ATTN_L2_PREFETCH tiles ahead of its load: the first CTA to
  // read a tile of a head otherwise waits for DRAM, and so do the CTAs reading it with it.
  auto prefetch = [&](const CUtensorMap* tm, int bh, int row) {
    if (c.lane != 0) return;
    if (kBshd) {
      const int b = bh / p.heads, h = bh - b * p.heads;
      ptx::tma_prefetch_4d(tm, 0, h, row, b);
      ptx::tma_prefetch_4d(tm, 64, h, row, b);
    } else {
      ptx::tma_prefetch_3d(tm, 0, row, bh);
      ptx::tma_prefetch_3d(tm, 64, row, bh);
    }
  };
  // (the test hook exists in the general mode only; the host sends its launches there)
  bool withhold = kMode == kModeGeneral && p.test_withhold != 0 && blockIdx.x == 0;
  auto load_kv = [&](const CUtensorMap* tm, int bh, int row) -> bool {
    if (!c.wait(ctl->kv_empty[slot], phase ^ 1u, kStatusTimeoutLoad)) return false;
    if (__builtin_expect(withhold, 0)) {   // the slot is skipped: nothing is loaded into it, nothing to drain
      withhold = false;
      if (++slot == kKvStages) { slot = 0; phase ^= 1u; }
      return true;
    }
    if (c.lane == 0) {
      const uint32_t fb = c.bar(ctl->kv_full[slot]);
      ptx::mbar_arrive_expect_tx(fb, kTileBytes);
      load_box(c.skv(slot), tm, fb, 0, row, bh);
      load_box(c.skv(slot) + kSlabBytes, tm, fb, 64, row, bh);
    }
    __syncwarp();
    kv_used |= 1u << slot;
    kv_last_par = (kv_last_par & ~(1u << slot)) | (phase << slot);
    if (++slot == kKvStages) { slot = 0; phase ^= 1u; }
    return true;
  };
  auto load_q = [&](int q, int bh, int row) -> bool {
    if (!c.wait(ctl->q_empty[q], (q_cnt[q] & 1u) ^ 1u, kStatusTimeoutLoad)) return false;
    if (c.lane == 0) {
      const uint32_t fb = c.bar(ctl->q_full[q]);
      ptx::mbar_arrive_expect_tx(fb, kTileBytes);
      load_q_box(c.sq(q), fb, 0, row, bh);
      load_q_box(c.sq(q) + kSlabBytes, fb, 64, row, bh);
    }
    __syncwarp();
    ++q_cnt[q];
    return true;
  };

  for (int r = 0; ok; ++r) {
    Seg sg;
    if (!seg_of<kSplit>(r, p, ctl->sk_range, sg)) break;
    const WorkItem& w = sg.w;
    const int row0 = w.qt0 * kBlockM;
    const int ntiles = w.n[1] > 0 ? w.n[1] : w.n[0];   // n[1] >= n[0] whenever it is non-zero
    const int kv0 = sg.j0 * kBlockN;                    // first key row of the segment
#if ATTN_L2_PREFETCH > 0
    for (int j = 0; j < ATTN_L2_PREFETCH && j < ntiles; ++j) {
      prefetch(tm_k, w.bh, kv0 + j * kBlockN);
      prefetch(tm_v, w.bh, kv0 + j * kBlockN);
    }
#endif
    ok = load_q(0, w.bh, row0) && load_kv(tm_k, w.bh, kv0);
    if (ok && (kMode != kModeGeneral || w.n[1] > 0)) ok = load_q(1, w.bh, row0 + kBlockM);
    if (ok) ok = load_kv(tm_v, w.bh, kv0);
    for (int j = 1; ok && j < ntiles; ++j) {
#if ATTN_L2_PREFETCH > 0
      if (j + ATTN_L2_PREFETCH - 1 < ntiles) {
        prefetch(tm_k, w.bh, kv0 + (j + ATTN_L2_PREFETCH - 1) * kBlockN);
        prefetch(tm_v, w.bh, kv0 + (j + ATTN_L2_PREFETCH - 1) * kBlockN);
      }
#endif
      ok = load_kv(tm_k, w.bh, kv0 + j * kBlockN) && load_kv(tm_v, w.bh, kv0 + j * kBlockN);
    }
  }
  if (!ok) {
    // Stop issuing; wait for the copies this warp already started.
    for (int s = 0; s < kKvStages; ++s)
      if ((kv_used >> s) & 1u) c.drain_wait(ctl->kv_full[s], (kv_last_par >> s) & 1u);
    for (int q = 0; q < 2; ++q)
      if (q_cnt[q]) c.drain_wait(ctl->q_full[q], (q_cnt[q] - 1) & 1u);
  }
}

// ------------------------------------------------------------------ MMA warp
template <int Q>
__device__ __forceinline__ void issue_qk(const Ctx& c, int kslot) {
  constexpr uint32_t idesc = make_idesc_bf16(128, 128, 0);
  const uint64_t a0 = smem_desc_sw128(c.sq(Q), 16, 1024);
  const uint64_t b0 = smem_desc_sw128(c.skv(kslot), 16, 1024);
#pragma unroll
  for (int kk = 0; kk < kHeadDim / 16; ++kk) {
    // K-step kk: slab kk/4 (64 columns), 32-byte column offset inside the 128-byte swizzle row.
    const uint32_t off16 = ((kk >> 2) * kSlabBytes + (kk & 3) * 32) >> 4;
    ptx::mma_ss(kTmemBase + col_s(Q), a0 + off16, b0 + off16, idesc, kk > 0);
  }
}

// P_q * V: A = packed P in TMEM, B = V tile (MN-major, 128B swizzle), 8 K-steps of 16 keys.
template <int Q>
__device__ __forceinline__ void issue_pv(const Ctx& c, int vslot, bool overwrite_first) {
  constexpr uint32_t idesc = make_idesc_bf16(128, 128, 1);
  const uint64_t b0 = smem_desc_sw128(c.skv(vslot), kSlabBytes, 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    // 16 V rows per K-step: 16 * 128 bytes inside each 64-column slab.
    ptx::mma_ts(kTmemBase + col_o(Q), kTmemBase + col_s(Q) + kColP + kk * 8,
                b0 + ((kk * 16 * 128) >> 4), idesc, (kk == 0 && overwrite_first) ? 0u : 1u);
  }
}

template <bool kSplit, int kMode>
__device__ __forceinline__ void mma_role(const Ctx& c, const Params& p) {
  SmemCtl* ctl = c.ctl;
  const bool leader = ptx::elect_one();
  int slot = 0;
  uint32_t phase = 0;
  uint32_t q_cnt[2] = {0, 0};
  uint32_t pv_phase[2] = {0, 0};
  bool ok = true;

  auto next_kv = [&](int& s_out) -> bool {
    s_out = slot;
    const bool r = c.wait(ctl->kv_full[slot], phase, kStatusTimeoutMma);
    if (++slot == kKvStages) { slot = 0; phase ^= 1u; }
    return r;
  };
  // Q_qK(j): Q_q of the current item against the K tile in kslot.
  auto qk = [&](int q, int kslot, bool new_item, bool last_qk, bool release_k) -> bool {
    if (new_item) {
      if (!c.wait(ctl->q_full[q], q_cnt[q] & 1u, kStatusTimeoutMma)) return false;
      ++q_cnt[q];
    }
    ptx::tc_fence_after();
    if (leader) {
      if (q == 0) issue_qk<0>(c, kslot); else issue_qk<1>(c, kslot);
      ptx::mma_commit(c.bar(ctl->s_full[q]));
      if (last_qk) ptx::mma_commit(c.bar(ctl->q_empty[q]));
      if (release_k) ptx::mma_commit(c.bar(ctl->kv_empty[kslot]));
    }
    __syncwarp();
    return true;
  };
  // P_q V with V in vslot.  v_phase >= 0: V's token is waited for here too, in the same poll as P
  // (a wait on an mbarrier costs this warp about as much as two MMA issues, and the MMA warp's
  // own instruction time bounds the pipeline, so it waits as rarely as it can).
  auto pv = [&](int q, int vslot, bool first_tile, int v_phase) -> bool {
    if (v_phase >= 0) {
      if (!c.wait2(ctl->kv_full[vslot], static_cast<uint32_t>(v_phase), ctl->p_full[q],
                   pv_phase[q], kStatusTimeoutMma))
        return false;
    } else if (!c.wait(ctl->p_full[q], pv_phase[q], kStatusTimeoutMma)) {
      return false;
    }
    ptx::tc_fence_after();
    if (leader) {
      if (q == 0) issue_pv<0>(c, vslot, first_tile); else issue_pv<1>(c, vslot, first_tile);
    }
    __syncwarp();
    pv_phase[q] ^= 1u;
    return true;
  };

  // K/V tokens are consumed in the order the TMA warp loads them (K_0, V_0, K_1, V_1, ... per
  // item).  Per KV tile j: P_0 V(j), Q_0 K(j+1), P_1 V(j), Q_1 K(j+1) (Chapter 7 order).  A
  // stage whose stream ends on the item's last tile issues the next item's first Q K right after
  // its last P V; a stage that ends earlier (stage 0 of a causal pair) defers it to the end of
  // the item, after the last token of the item has been consumed.
  int r = 0;
  Seg sg;
  if (seg_of<kSplit>(0, p, ctl->sk_range, sg)) {
    WorkItem w = sg.w;
    int kslot;
    ok = next_kv(kslot) && qk(0, kslot, true, w.n[0] == 1, w.n[1] == 0);
    if (ok && w.n[1] > 0) ok = qk(1, kslot, true, w.n[1] == 1, true);
    while (ok) {
      const int ntiles = w.n[1] > 0 ? w.n[1] : w.n[0];
      // The full-tile mode's items all have two Q tiles over the same KV tiles (dense, an even
      // number of full Q tiles; a split segment gives both the same KV range): n0 = n1.
      const int n0 = kMode == kModeFull ? ntiles : w.n[0];
      const int n1 = kMode == kModeFull ? ntiles : w.n[1];
      Seg nsg;
      const bool has_next = seg_of<kSplit>(r + 1, p, ctl->sk_range, nsg);
      const WorkItem nw = has_next ? nsg.w : w;
      int next_kslot = -1;
      // First Q K of stage q for the next item (its K_0 is acquired once for both stages).
      auto issue_next = [&](int q) -> bool {
        if (!has_next || nw.n[q] == 0) return true;
        if (next_kslot < 0 && !next_kv(next_kslot)) return false;
        return qk(q, next_kslot, true, nw.n[q] == 1, q == 1 || nw.n[1] == 0);
      };
      bool next0_done = false;
      if constexpr (kMode != kModeGeneral) {
        // n1 = n0 + d, d in {0, 1}: d = 1 for most causal pairs, 0 in the full-tile mode.  The
        // tiles both stages share run a loop without per-stage tests; stage 0's last tile and
        // stage 1's extra one follow (the same MMAs and commits in the same order as the general
        // loop below; the MMA warp's instructions per tile bound this pipeline: +1.4% at causal
        // S=4K, +2.4% at causal S=16K, +2.6% for the split schedule at S=16K, bitwise the same).
        const int d = n1 - n0;
        for (int j = 0; ok && j < n0 - 1; ++j) {
          const int vslot = slot;
          const int v_phase = static_cast<int>(phase);
          if (++slot == kKvStages) { slot = 0; phase ^= 1u; }
          int kn = -1;
          if (!(ok = pv(0, vslot, j == 0, v_phase))) break;
          if (!(ok = next_kv(kn))) break;
          if (!(ok = qk(0, kn, false, j + 1 == n0 - 1, false))) break;
          if (!(ok = pv(1, vslot, j == 0, -1))) break;
          if (leader) ptx::mma_commit(c.bar(ctl->kv_empty[vslot]));
          __syncwarp();
          if (!(ok = qk(1, kn, false, j + 1 == n1 - 1, true))) break;
        }
        if (ok) {   // j = n0 - 1: stage 0's last tile
          const int vslot = slot;
          const int v_phase = static_cast<int>(phase);
          if (++slot == kKvStages) { slot = 0; phase ^= 1u; }
          ok = pv(0, vslot, n0 == 1, v_phase);
          if (ok) {
            if (leader) ptx::mma_commit(c.bar(ctl->o_full[0]));
            __syncwarp();
            if (d == 0) {
              ok = issue_next(0);
              next0_done = true;
            }
          }
          if (ok) ok = pv(1, vslot, n0 == 1, -1);
          if (ok) {
            if (leader) {
              if (d == 0) ptx::mma_commit(c.bar(ctl->o_full[1]));
              ptx::mma_commit(c.bar(ctl->kv_empty[vslot]));
            }
            __syncwarp();
            if (d == 1) {
              int kn = -1;
              ok = next_kv(kn) && qk(1, kn, false, true, true);
            }
          }
        }
        if (ok && d == 1) {   // j = n0: stage 1's last tile
          const int vslot = slot;
          const int v_phase = static_cast<int>(phase);
          if (++slot == kKvStages) { slot = 0; phase ^= 1u; }
          ok = pv(1, vslot, false, v_phase);
          if (ok) {
            if (leader) {
              ptx::mma_commit(c.bar(ctl->o_full[1]));
              ptx::mma_commit(c.bar(ctl->kv_empty[vslot]));
            }
            __syncwarp();
          }
        }
      } else
      for (int j = 0; ok && j < ntiles; ++j) {
        // V(j): its token is taken from the ring here and waited for by the first P V on it.
        const int vslot = slot;
        int v_phase = static_cast<int>(phase);
        if (++slot == kKvStages) { slot = 0; phase ^= 1u; }
        int kslot_next = -1;
        // stage 0: P0 V(j), then Q0 K(j+1)
        if (j < n0) {
          if (!(ok = pv(0, vslot, j == 0, v_phase))) break;
          v_phase = -1;
          if (leader) {
            if (j == n0 - 1) ptx::mma_commit(c.bar(ctl->o_full[0]));
            if (j >= n1) ptx::mma_commit(c.bar(ctl->kv_empty[vslot]));
          }
          __syncwarp();
          if (j + 1 < n0) {
            if (!(ok = next_kv(kslot_next))) break;
            if (!(ok = qk(0, kslot_next, false, j + 1 == n0 - 1, j + 1 >= n1))) break;
          } else if (j == ntiles - 1) {
            if (!(ok = issue_next(0))) break;
            next0_done = true;
          }
        }
        // stage 1: P1 V(j), then Q1 K(j+1)
        if (j < n1) {
          if (!(ok = pv(1, vslot, j == 0, v_phase))) break;
          v_phase = -1;
          if (leader) {
            if (j == n1 - 1) ptx::mma_commit(c.bar(ctl->o_full[1]));
            ptx::mma_commit(c.bar(ctl->kv_empty[vslot]));
          }
          __syncwarp();
          if (j + 1 < n1) {
            if (kslot_next < 0 && !(ok = next_kv(kslot_next))) break;
            if (!(ok = qk(1, kslot_next, false, j + 1 == n1 - 1, true))) break;
          }
        }
      }
      if (!ok) break;
      if (!next0_done && !(ok = issue_next(0))) break;
      if (!(ok = issue_next(1))) break;
      if (!has_next) break;
      w = nw;
      ++r;
    }
  }
  // Wait for every MMA this thread issued before TMEM can be released.
  if (leader) ptx::mma_commit(c.bar(ctl->drain));
  __syncwarp();
  c.drain_wait(ctl->drain, 0);
}

// ------------------------------------------------------------------ softmax warpgroups
// Raw scores of columns >= valid become -inf (they then never hold the row max).
// Masked columns (>= valid) get the raw score -inf: they never set the row max, and their P is
// exp2(-inf) = 0 (the multiplier is always positive, so -inf stays -inf).  keep = 0 (zero scale)
// also turns every kept score into 0, so each of them gets P = exp2(0) = 1.
__device__ __forceinline__ void mask_scores(uint32_t (&sr)[4][32], int valid, uint32_t keep) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc)
#pragma unroll
    for (int i = 0; i < 32; ++i)
      sr[cc][i] = cc * 32 + i >= valid ? 0xff800000u : (sr[cc][i] & keep);
}

// P of one KV tile: exp2(s * scale_log2 - m_kept), two columns per packed FMA, packed BF16 into
// TMEM over the upper half of this stage's S columns, published once all 128 are written
// (p_full).  Masked columns arrive as -inf and come out as 0.  Returns the row sum of the tile's
// fp32 P.
// 2^x for two values on the FMA and integer pipes, no MUFU ("B200 Attention Kernel from Scratch to
// Near-SOTA in 60 Diagrams", Chapter 9 and its appendix on the approximation): x = n + f with
// n = floor(x), f in [0, 1); 2^f by the cubic minimax fit of 2^f on [0, 1] with p(0) = 1 (relative
// error 8.6e-5; coefficients from soft_exp2_fit.py); n is added to the exponent field.  Below
// -126 the result is 0, as the flushing hardware path gives (masked scores are -inf).
constexpr float kExp2C1 = 0.69511676f, kExp2C2 = 0.227645f, kExp2C3 = 0.07706704f;
__device__ __forceinline__ float2 soft_exp2x2(float2 x) {
  constexpr float kRound = 12582912.0f;   // 1.5 * 2^23: x + kRound, rounded down, is kRound + n
  const bool lo_x = x.x < -126.0f, lo_y = x.y < -126.0f;
  x.x = fmaxf(x.x, -127.0f);   // keeps n in range (and -inf finite) before the result is dropped
  x.y = fmaxf(x.y, -127.0f);
  const float2 rr = make_float2(kRound, kRound);
  const float2 t = ptx::fadd2_rm(x, rr);
  const float2 f = ptx::fsub2(x, ptx::fsub2(t, rr));
  float2 y = ptx::ffma2(make_float2(kExp2C3, kExp2C3), f, make_float2(kExp2C2, kExp2C2));
  y = ptx::ffma2(y, f, make_float2(kExp2C1, kExp2C1));
  y = ptx::ffma2(y, f, make_float2(1.0f, 1.0f));
  const int bias = __float_as_int(kRound);
  y.x = __int_as_float(__float_as_int(y.x) + ((__float_as_int(t.x) - bias) << 23));
  y.y = __int_as_float(__float_as_int(y.y) + ((__float_as_int(t.y) - bias) << 23));
  if (lo_x) y.x = 0.0f;
  if (lo_y) y.y = 0.0f;
  return y;
}

template <bool kSoftExp2>
__device__ __forceinline__ float produce_p(const Ctx& c, int q, const uint32_t (&sr)[4][32],
                                           float scale_log2, float m_kept, uint32_t taddr_s) {
  SmemCtl* ctl = c.ctl;
  const float2 c2 = make_float2(scale_log2, scale_log2);
  const float2 nm2 = make_float2(-m_kept, -m_kept);
  float2 sum2[4];
#pragma unroll
  for (int cc = 3; cc >= 0; --cc) {
    uint32_t pk[16];
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float2 x = ptx::ffma2(make_float2(__uint_as_float(sr[cc][2 * i]), __uint_as_float(sr[cc][2 * i + 1])),
                            c2, nm2);
      if (kSoftExp2 && (i & 7) >= 6) {   // columns 12..15 of every 16 (Chapter 9's split)
        x = soft_exp2x2(x);
      } else {
        x.x = ptx::ex2_ftz(x.x);
        x.y = ptx::ex2_ftz(x.y);
      }
      if (i & 1) acc1 = ptx::fadd2(acc1, x); else acc0 = ptx::fadd2(acc0, x);
      pk[i] = ptx::pack_bf16x2(x.x, x.y);
    }
    sum2[cc] = ptx::fadd2(acc0, acc1);
    ptx::tmem_st_32x32b_x16(taddr_s + kColP + 16 * cc, pk);
  }
  ptx::tmem_wait_st();
  ptx::tc_fence_before();
  c.arrive(ctl->p_full[q]);
  const float2 t2 = ptx::fadd2(ptx::fadd2(sum2[3], sum2[2]), ptx::fadd2(sum2[1], sum2[0]));
  return t2.x + t2.y;
}

// Max of the 128 raw scores of this thread's row (bit patterns from tcgen05.ld).
__device__ __forceinline__ float row_max_128(const uint32_t (&sr)[4][32]) {
  auto f = [&](int i) { return __uint_as_float(sr[i >> 5][i & 31]); };
  float a[43];
#pragma unroll
  for (int i = 0; i < 42; ++i) a[i] = ptx::fmax3(f(3 * i), f(3 * i + 1), f(3 * i + 2));
  a[42] = fmaxf(f(126), f(127));
  float b[15];
#pragma unroll
  for (int i = 0; i < 14; ++i) b[i] = ptx::fmax3(a[3 * i], a[3 * i + 1], a[3 * i + 2]);
  b[14] = a[42];
  float d[5];
#pragma unroll
  for (int i = 0; i < 5; ++i) d[i] = ptx::fmax3(b[3 * i], b[3 * i + 1], b[3 * i + 2]);
  return fmaxf(ptx::fmax3(d[0], d[1], d[2]), fmaxf(d[3], d[4]));
}

// Item epilogue of stage q in the general mode, run by the stage's own softmax warpgroup: O_q
// (final once the item's last P*V is done, o_full) is read from TMEM, scaled by 1 / (row sum of
// the BF16 weights) and
// packed to BF16 in registers;
// once read, O_q's columns are free for the next item's first P*V, which waits for the next
// P this warpgroup publishes.  The stores to global memory follow from the registers.
__device__ __forceinline__ bool epilogue_read(const Ctx& c, int q, uint32_t o_parity, float inv_l,
                                              uint32_t (&pk)[64]) {
  if (!c.wait(c.ctl->o_full[q], o_parity, kStatusTimeoutSoftmax)) return false;
  ptx::tc_fence_after();
  const uint32_t taddr_o = c.tmem + ((32u * (c.warp & 3u)) << 16) + col_o(q);
#pragma unroll
  for (int h = 0; h < 2; ++h) {   // 64 columns per TMEM wait
    uint32_t r[2][32];
    ptx::tmem_ld_32x32b_x64(taddr_o + 64 * h, r[0], r[1]);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
      for (int i = 0; i < 16; ++i)
        pk[32 * h + 16 * c2 + i] = ptx::pack_bf16x2(__uint_as_float(r[c2][2 * i]) * inv_l,
                                                    __uint_as_float(r[c2][2 * i + 1]) * inv_l);
  }
  ptx::tc_fence_before();
  return true;
}

// General mode: O row and LSE of this thread's query row of stage q of item w (rows past a ragged
// end of Q are computed but not stored).  The row (256 bytes) goes out in 32-byte stores when the
// output is 32-byte aligned (half the store instructions of 16-byte ones: measured +1.2% at S=4K
// and +2.8% causal when this epilogue served every mode), else in 16-byte stores.
// LSE = (kept max + log2 l) * ln 2, l the row sum of the fp32 P.
__device__ __forceinline__ void epilogue_store(const Params& p, int q, const WorkItem& w, int row,
                                               float m, float l, const uint32_t (&pk)[64]) {
  const int grow = (w.qt0 + q) * kBlockM + row;
  if (grow >= p.sq) return;
  const int b = w.bh / p.heads, h = w.bh - b * p.heads;
  uint8_t* out = static_cast<uint8_t*>(p.o) +
                 (b * p.o_batch_stride + h * p.o_head_stride + grow * p.o_row_stride) * 2;
  if (__builtin_expect(p.o_align32, 1)) {   // 32-byte stores where allowed
#pragma unroll
    for (int i = 0; i < 8; ++i) ptx::st_global_v8(out + 32 * i, pk + 8 * i);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      ptx::st_global_v4(out + 16 * i, pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
  }
  if (p.lse != nullptr)
    p.lse[static_cast<size_t>(w.bh) * p.sq + grow] = (m + log2f(l)) * 0.69314718055994530942f;
}

// Item epilogue of stage q for one part of an item split between two CTAs (this warp's 32 rows).
// The warp first looks at its flag: if the partner part's warp has already left the call's
// sequence number there, its O / l (fp32) and base-2 LSE are in the workspace and this warp
// combines at once.  Otherwise it writes its own part there and swaps the sequence number into
// the flag; if that swap returns the number, the partner wrote in the meantime and this warp
// combines, else the partner will.  Exactly one of the two warps combines, and neither waits.
// The combining warp clears the flag again.
// The combination is O = w0 O0/l0 + w1 O1/l1 with w_i = 2^(L_i - L), L = log2(2^L0 + 2^L1),
// each product and the sum rounded separately, so it is the same whichever warp computes it.
// Not inlined: it runs at most twice per CTA, and inlined into the softmax role it slowed the
// whole-item rounds by 0.5-1% (larger loop code).  It takes the few parameters it reads by value
// (SplitOut): marking the kernel's parameter block __grid_constant__ so that its address could be
// passed instead made the [B,S,H,D] forward 6-8% slower in both instantiations (measured).
struct SplitOut {
  float* ws_o;
  float* ws_l;
  unsigned long long* ws_flag;
  unsigned long long seq;
  void* o;
  float* lse;
  int64_t o_row_stride, o_head_stride, o_batch_stride;
  int sq;
  int heads;
};

__device__ __forceinline__ SplitOut split_out(const Params& p) {
  return SplitOut{p.ws_o, p.ws_l, p.ws_flag, p.seq, p.o, p.lse, p.o_row_stride, p.o_head_stride,
                  p.o_batch_stride, p.sq, p.heads};
}

__device__ __noinline__ bool epilogue_split(const Ctx& c, const SplitOut p, int q, const Seg& sg,
                                               int row, float m, float l, float l_bf16,
                                               uint32_t o_parity) {
  if (!c.wait(c.ctl->o_full[q], o_parity, kStatusTimeoutSoftmax)) return false;
  ptx::tc_fence_after();
  const uint32_t taddr_o = c.tmem + ((32u * (c.warp & 3u)) << 16) + col_o(q);
  const float inv_l = 1.0f / l_bf16;   // O / l with the row sum of the weights P*V used
  const float L_own = m + log2f(l);     // the part's log2-sum-exp, from the fp32 row sum
  constexpr size_t kPartFloats = static_cast<size_t>(kBlockM) * kHeadDim;
  const size_t own = (static_cast<size_t>(sg.slot) * 2 + sg.part) * 2 + q;   // [slot][part][stage]
  const size_t oth = (static_cast<size_t>(sg.slot) * 2 + (1 - sg.part)) * 2 + q;
  unsigned long long* flag = p.ws_flag + (static_cast<size_t>(sg.slot) * 2 + q) * 4 + (c.warp & 3u);
  unsigned long long f = 0;
  if (c.lane == 0) f = ptx::ld_acquire_u64(flag);
  __syncwarp();   // orders lane 0's acquire before the other lanes' reads of the partner's part
  f = __shfl_sync(0xffffffffu, f, 0);
  if (f != p.seq) {
    float* dst = p.ws_o + own * kPartFloats + row * 4;   // chunk i (4 columns) at + i * 128 * 4
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t r[32];
      ptx::tmem_ld_32x32b_x32(taddr_o + 32 * cc, r);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 8; ++i)
        ptx::st_global_v4(dst + (cc * 8 + i) * kBlockM * 4,
                          __float_as_uint(__uint_as_float(r[4 * i]) * inv_l),
                          __float_as_uint(__uint_as_float(r[4 * i + 1]) * inv_l),
                          __float_as_uint(__uint_as_float(r[4 * i + 2]) * inv_l),
                          __float_as_uint(__uint_as_float(r[4 * i + 3]) * inv_l));
    }
    p.ws_l[own * kBlockM + row] = L_own;
    __threadfence();
    __syncwarp();
    if (c.lane == 0) {
      f = atomicExch(flag, p.seq);
      __threadfence();
    }
    __syncwarp();
    f = __shfl_sync(0xffffffffu, f, 0);
    if (f != p.seq) {   // the partner combines
      ptx::tc_fence_before();
      return true;
    }
  }
  __threadfence();
  // Both parts have arrived and nothing else touches this flag in this launch: clear it, so a later
  // launch with the same sequence number (a replayed CUDA graph) does not take it for its partner.
  if (c.lane == 0) *flag = 0ull;
  // Combine: this part from TMEM (O / l recomputed exactly as stored), the other from the workspace.
  const float L_oth = __ldcg(p.ws_l + oth * kBlockM + row);
  const float L0 = sg.part == 0 ? L_own : L_oth, L1 = sg.part == 0 ? L_oth : L_own;
  const float L = fmaxf(L0, L1);
  const float e0 = ptx::ex2_ftz(L0 - L), e1 = ptx::ex2_ftz(L1 - L);
  const float sum = e0 + e1;
  const float w0 = e0 / sum, w1 = e1 / sum;
  const float w_own = sg.part == 0 ? w0 : w1, w_oth = sg.part == 0 ? w1 : w0;
  const float4* src = reinterpret_cast<const float4*>(p.ws_o + oth * kPartFloats) + row;
  const int grow = (sg.w.qt0 + q) * kBlockM + row;
  const bool store = grow < p.sq;
  const int b = sg.w.bh / p.heads, h = sg.w.bh - b * p.heads;
  uint8_t* out = static_cast<uint8_t*>(p.o) +
                 (b * p.o_batch_stride + h * p.o_head_stride + grow * p.o_row_stride) * 2;
  float4 nxt[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) nxt[i] = __ldcg(src + i * kBlockM);
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {   // 32 columns per step, the next step's loads in flight
    float4 cur[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
    if (cc < 3) {
#pragma unroll
      for (int i = 0; i < 8; ++i) nxt[i] = __ldcg(src + ((cc + 1) * 8 + i) * kBlockM);
    }
    uint32_t r[32];
    ptx::tmem_ld_32x32b_x32(taddr_o + 32 * cc, r);
    ptx::tmem_wait_ld();
    auto mix = [&](int k, float oth_v) {
      const float own_v = __uint_as_float(r[k]) * inv_l;
      return __fadd_rn(__fmul_rn(own_v, w_own), __fmul_rn(oth_v, w_oth));
    };
    if (store) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {   // 8 columns = 16 bytes of BF16
        const float4 x = cur[2 * i], y = cur[2 * i + 1];
        ptx::st_global_v4(out + 64 * cc + 16 * i,
                          ptx::pack_bf16x2(mix(8 * i, x.x), mix(8 * i + 1, x.y)),
                          ptx::pack_bf16x2(mix(8 * i + 2, x.z), mix(8 * i + 3, x.w)),
                          ptx::pack_bf16x2(mix(8 * i + 4, y.x), mix(8 * i + 5, y.y)),
                          ptx::pack_bf16x2(mix(8 * i + 6, y.z), mix(8 * i + 7, y.w)));
      }
    }
  }
  ptx::tc_fence_before();
  if (store && p.lse != nullptr)
    p.lse[static_cast<size_t>(sg.w.bh) * p.sq + grow] = (L + log2f(sum)) * 0.69314718055994530942f;
  return true;
}

template <bool kSoftExp2, bool kSplit, int kMode>
__device__ __forceinline__ void softmax_role(const Ctx& c, const Params& p, int q) {
  SmemCtl* ctl = c.ctl;
  const uint32_t row_base = 32u * (c.warp & 3u);
  const int row = static_cast<int>(row_base + c.lane);
  const uint32_t taddr_s = c.tmem + (row_base << 16) + col_s(q);
  // A zero scale makes every kept score 0 (mask_scores on every tile) and uses multiplier 1, so
  // masked columns still give -inf * 1 = -inf rather than -inf * 0 = NaN.
  const bool zero_scale = kMode == kModeGeneral && p.scale_log2 == 0.f;
  const float scale_log2 = zero_scale ? 1.f : p.scale_log2;
  const uint32_t keep = zero_scale ? 0u : 0xffffffffu;
  uint32_t tphase = 0;
  uint32_t o_parity = 0;     // o_full phase of the previous item
  bool have_prev = false;    // an item whose epilogue is still to do
  Seg sp;
  float m_prev = 0.f, l_prev = 1.f, lr_prev = 1.f;
  uint32_t fin_par = 0;   // ctl->fin slot of the next item the correction warpgroup finishes

  for (int r = 0;; ++r) {
    Seg sg;
    if (!seg_of<kSplit>(r, p, ctl->sk_range, sg)) break;
    const WorkItem& w = sg.w;
    const int ntiles = w.n[q];
    if (kMode == kModeGeneral && ntiles == 0) continue;
    const int qtile = w.qt0 + q;
    // General mode and split parts: the previous item's epilogue, before this item's first P:
    // its O columns are then free when that P is published (the first P*V of an item overwrites
    // O), and the read overlaps this item's first Q*K^T, issued right after the previous item's
    // last P*V.  Otherwise the correction warpgroup runs it.
    if (have_prev) {
      if (kSplit && sp.slot >= 0) {
        if (!epilogue_split(c, split_out(p), q, sp, row, m_prev, l_prev, lr_prev, o_parity)) return;
      } else if constexpr (kMode == kModeGeneral) {
        uint32_t pk[64];
        if (!epilogue_read(c, q, o_parity, 1.0f / lr_prev, pk)) return;
        epilogue_store(p, q, sp.w, row, m_prev, l_prev, pk);
      }
      o_parity ^= 1u;
    }
    float m_kept = 0.f;   // base-2 units; set on the first tile
    float l = 0.f;    // row sum of the fp32 P (for the LSE)
    float dl = 0.f;   // BF16 rounding of the largest P of each tile (see below)
    for (int j = 0; j < ntiles; ++j) {
      if (!c.wait(ctl->s_full[q], tphase, kStatusTimeoutSoftmax)) return;
      ptx::tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) ptx::tmem_ld_32x32b_x32(taddr_s + 32 * cc, sr[cc]);
      ptx::tmem_wait_ld();
      // Masked columns (no weight): past the end of a key sequence that is not a multiple of
      // 128 (zero-filled key rows), and, with the causal mask, past this row on the diagonal
      // tile.  They must not enter the max and get P = 0 below.  The test is warp-uniform.
      const int jg = sg.j0 + j;   // KV tile index within the head
      const bool diag = p.causal != 0 && jg == qtile;
      // Tiles with masked columns: the causal diagonal (kModeCausal), also a ragged last key tile
      // and every tile at zero scale (kModeGeneral); kModeFull has no masking code, whose
      // presence, never taken, cost the dense forward ~2% (same-box A/B, bitwise the same).
      const bool partial =
          kMode == kModeCausal ? diag
          : kMode == kModeGeneral
              ? (zero_scale || diag || (jg == p.kv_tiles - 1 && p.kv_valid_last < kBlockN))
              : false;
      int valid = kBlockN;
      if (kMode == kModeGeneral && jg == p.kv_tiles - 1) valid = p.kv_valid_last;
      if (diag) valid = min(valid, row + 1);
      if (partial) mask_scores(sr, valid, keep);

      // Row max over the raw scores: a 3-input-max tree (depth 5, 65 instructions).
      const float s_max = row_max_128(sr);
      const float m_tile = s_max * scale_log2;
      float alpha = 1.f;
      if (j == 0) {
        m_kept = m_tile;
      } else if (__builtin_expect(m_tile - m_kept >= kRebaseThresholdLog2, 0)) {
        alpha = ptx::ex2_ftz(m_kept - m_tile);
        l *= alpha;
        dl *= alpha;
        m_kept = m_tile;
      }
      ctl->alpha[q][tphase][row] = alpha;
      c.arrive(ctl->stats_full[q]);

      l += produce_p<kSoftExp2>(c, q, sr, scale_log2, m_kept, taddr_s);
      // P*V multiplies the BF16-rounded P, the row sum l adds the fp32 P.  O is divided by
      // l + dl, where dl carries the rounding (BF16 minus fp32) of the tile's largest P, the same
      // value produce_p computed for that column: numerator and denominator then agree on the
      // weight that dominates a peaked row, while the LSE keeps the exact fp32 sum.
      const float p_top = ptx::ex2_ftz(fmaf(s_max, scale_log2, -m_kept));
      dl += __uint_as_float(ptx::pack_bf16x2(0.f, p_top)) - p_top;
      tphase ^= 1u;
    }
    if (kMode != kModeGeneral && !(kSplit && sg.slot >= 0)) {
      // The correction warpgroup writes this item's O and LSE (after its last P*V) while this
      // warpgroup goes on with the next item (a split item's part is finished here, below).
      ctl->fin[q][fin_par][row] =
          make_float2(1.0f / (l + dl), (m_kept + log2f(l)) * 0.69314718055994530942f);
      c.arrive(ctl->fin_full[q][fin_par]);
      fin_par ^= 1u;
    }
    have_prev = true;
    sp = sg;
    m_prev = m_kept;
    l_prev = l;
    lr_prev = l + dl;
  }
  if (have_prev) {
    if (kSplit && sp.slot >= 0) {
      epilogue_split(c, split_out(p), q, sp, row, m_prev, l_prev, lr_prev, o_parity);
    } else if constexpr (kMode == kModeGeneral) {
      uint32_t pk[64];
      if (!epilogue_read(c, q, o_parity, 1.0f / lr_prev, pk)) return;
      epilogue_store(p, q, sp.w, row, m_prev, l_prev, pk);
    }
  }
}

// ------------------------------------------------------------------ correction warpgroup
// Per KV tile and stage: if any row of the warp rebased its max, O_q *= alpha in TMEM; then O_q
// is safe for the next P*V (p_full, together with the softmax's P).  In the full-tile and causal
// modes it also runs the item epilogue of whole items, before the next item's first tile.
template <bool kSplit, int kMode>
__device__ __forceinline__ void correction_role(const Ctx& c, const Params& p) {
  SmemCtl* ctl = c.ctl;
  const uint32_t row_base = 32u * (c.warp & 3u);
  const int row = static_cast<int>(row_base + c.lane);
  uint32_t tphase[2] = {0, 0};
  // Full-tile and causal modes: this warpgroup writes each whole item's O (final after its last
  // P*V, o_full) and LSE from the statistics the softmax warpgroup leaves in ctl->fin, before it
  // lets the next item's first P*V overwrite O (p_full of that item's first tile).  Moving the
  // epilogue here from the softmax warpgroups measured +1.2% at S=4K, +1.0% at S=8K/16K (split
  // schedule), +2.8% / +2.4% at causal S=4K / 16K (same box, bitwise the same).
  uint32_t opar[2] = {0, 0};   // o_full phase of the previous item (every item)
  uint32_t fcnt[2] = {0, 0};   // items finished here per stage: ctl->fin slot fcnt & 1,
                               // that slot's fin_full phase (fcnt >> 1) & 1
  Seg prev;
  bool have_prev = false;
  auto epilogue = [&](int q, const Seg& sgp) -> bool {
    // Every item's o_full phase is waited for, so the parity tracked here never falls behind.
    if (!c.wait(ctl->o_full[q], opar[q], kStatusTimeoutCorrection)) return false;
    opar[q] ^= 1u;
    if (kSplit && sgp.slot >= 0) return true;   // a split item's part: the softmax finishes it
    const WorkItem& w = sgp.w;
    const uint32_t slot = fcnt[q] & 1u;
    if (!c.wait(ctl->fin_full[q][slot], (fcnt[q] >> 1) & 1u, kStatusTimeoutCorrection)) return false;
    ptx::tc_fence_after();
    const float2 f = ctl->fin[q][slot][row];
    const uint32_t taddr_o = c.tmem + (row_base << 16) + col_o(q);
    const int grow = (w.qt0 + q) * kBlockM + row;
    const int b = w.bh / p.heads, h = w.bh - b * p.heads;
    uint8_t* out = static_cast<uint8_t*>(p.o) +
                   (b * p.o_batch_stride + h * p.o_head_stride + grow * p.o_row_stride) * 2;
    const uint64_t pol = ptx::l2_policy_evict_first();
#pragma unroll 1
    for (int cc = 0; cc < 8; ++cc) {
      uint32_t v[16];
      ptx::tmem_ld_32x32b_x16(taddr_o + 16 * cc, v);
      ptx::tmem_wait_ld();
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        pk[i] = ptx::pack_bf16x2(__uint_as_float(v[2 * i]) * f.x, __uint_as_float(v[2 * i + 1]) * f.x);
      ptx::st_global_v8_hint(out + 32 * cc, pk, pol);   // written once: first to evict from L2
    }
    if (p.lse != nullptr) p.lse[static_cast<size_t>(w.bh) * p.sq + grow] = f.y;
    ptx::tc_fence_before();
    ++fcnt[q];
    return true;
  };

  for (int r = 0;; ++r) {
    Seg sg;
    if (!seg_of<kSplit>(r, p, ctl->sk_range, sg)) break;
    const WorkItem& w = sg.w;
    const int ntiles = w.n[1] > 0 ? w.n[1] : w.n[0];
    for (int j = 0; j < ntiles; ++j) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (kMode != kModeFull && j >= w.n[q]) continue;
        if (kMode != kModeGeneral && j == 0 && have_prev && !epilogue(q, prev)) return;
        if (!c.wait(ctl->stats_full[q], tphase[q], kStatusTimeoutCorrection)) return;
        // alpha is 1 on an item's first tile, so the previous item's O, which its softmax
        // warpgroup may still be reading, is not touched here.
        const float a = ctl->alpha[q][tphase[q]][row];
        if (__builtin_expect(__any_sync(0xffffffffu, a != 1.0f), 0)) {
          const uint32_t taddr_o = c.tmem + (row_base << 16) + col_o(q);
          ptx::tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t r[16];
            ptx::tmem_ld_32x32b_x16(taddr_o + 16 * cc, r);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * a);
            ptx::tmem_st_32x32b_x16(taddr_o + 16 * cc, r);
          }
          ptx::tmem_wait_st();
        }
        ptx::tc_fence_before();
        c.arrive(ctl->p_full[q]);
        tphase[q] ^= 1u;
      }
    }
    if (kMode != kModeGeneral) {
      prev = sg;
      have_prev = true;
    }
  }
  if (kMode != kModeGeneral && have_prev) {
    if (epilogue(0, prev)) epilogue(1, prev);
  }
}

// ------------------------------------------------------------------ kernel
template <bool kSoftExp2, bool kSplit, bool kBshd, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  Ctx c;
  c.smem_base = base;
  c.ctl = reinterpret_cast<SmemCtl*>(smem_raw + (base - raw) + kCtlOffset);
  c.warp = threadIdx.x >> 5;
  c.lane = threadIdx.x & 31u;
  SmemCtl* ctl = c.ctl;

  if (threadIdx.x == 0) {
    for (int q = 0; q < 2; ++q) {
      ptx::mbar_init(c.bar(ctl->q_full[q]), 1);
      ptx::mbar_init(c.bar(ctl->q_empty[q]), 1);
      ptx::mbar_init(c.bar(ctl->s_full[q]), 1);
      ptx::mbar_init(c.bar(ctl->p_full[q]), 2 * kArrivePerWG);   // softmax + correction WGs
      ptx::mbar_init(c.bar(ctl->stats_full[q]), kArrivePerWG);
      ptx::mbar_init(c.bar(ctl->o_full[q]), 1);
      ptx::mbar_init(c.bar(ctl->fin_full[q][0]), kArrivePerWG);
      ptx::mbar_init(c.bar(ctl->fin_full[q][1]), kArrivePerWG);
    }
    for (int s = 0; s < kKvStages; ++s) {
      ptx::mbar_init(c.bar(ctl->kv_full[s]), 1);
      ptx::mbar_init(c.bar(ctl->kv_empty[s]), 1);
    }
    ptx::mbar_init(c.bar(ctl->drain), 1);
    ctl->abort_flag = 0;
    if (kSplit) {
      ctl->sk_range[0] = split_range_begin(blockIdx.x, gridDim.x, p.sk_items, p.kv_tiles);
      ctl->sk_range[1] = split_range_begin(blockIdx.x + 1, gridDim.x, p.sk_items, p.kv_tiles);
    }
    ptx::fence_mbar_init();
  }
  if (c.warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&ctl->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  if (c.warp == kLoadWarp && c.lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_alloc_base = ctl->tmem_base;
  c.tmem = kTmemBase;
  if (tmem_alloc_base != kTmemBase) {
    if (threadIdx.x == 0) atomicOr(&g_attn_status, kStatusTmemBase);
  } else if (c.warp < kCorrWarp0) {
    ptx::setmaxnreg_inc<kRegSoftmax>();
    softmax_role<kSoftExp2, kSplit, kMode>(c, p, static_cast<int>(c.warp >> 2));
  } else if (c.warp < kLoadWarp) {
    ptx::setmaxnreg_dec<kRegCorr>();
    correction_role<kSplit, kMode>(c, p);
  } else {
    ptx::setmaxnreg_dec<kRegMisc>();
    if (c.warp == kLoadWarp) load_role<kSplit, kBshd, kMode>(c, p, &tm_q, &tm_k, &tm_v);
    else if (c.warp == kMmaWarp) mma_role<kSplit, kMode>(c, p);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (c.warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_alloc_base, kTmemCols);
  }
}

}  // namespace attn
