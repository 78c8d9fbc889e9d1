// attn_bwd_kernel.cuh -- backward of the dense head_dim-128 attention for sm_103a, consuming
// the forward's natural-log LSE ("Attention for sm90, Line by Line", the exp2 question: the
// residual is the row max in natural-log units so the backward can rebuild P).
//
// With P = exp(scale * Q K^T - LSE) (masked entries 0), dO = dL/dO and
//     delta_i = sum_d dO_id O_id,   dS = P o (dO V^T - delta),
//     dV = P^T dO,   dK = scale * dS^T Q,   dQ = scale * dS K,
// three kernels run in order on one stream:
//   attn_bwd_delta_kernel  delta (fp32, one warp per query row)
//   attn_bwd_dkdv_kernel   one CTA per 128-row K/V tile: S^T = K Q^T and dP^T = V dO^T into
//                          TMEM, P^T and dS^T (BF16) written back over their upper halves, then
//                          dV += P^T dO and dK += dS^T Q with A from TMEM; loops over Q tiles
//   attn_bwd_dq_kernel     one CTA per pair of 128-row Q tiles: per tile S = Q K^T, then
//                          dP = dO V^T over it, dS (BF16) over dP, dQ += dS K; loops over
//                          K/V tiles, each feeding both tiles
// Every gradient is written by exactly one CTA (no atomics: deterministic).  dQ repeats the
// S and dP products of dK/dV (7 tile products per tile pair instead of 5).
//
// Roles: dK/dV CTA (320 threads): warps 0-7 two elementwise warpgroups (one TMEM lane = one key
// row per thread, each warpgroup half of the query columns), warp 8 TMA, warp 9 tcgen05.mma
// issue and TMEM allocation; dQ CTA (384 threads): one elementwise warpgroup per Q tile, then a
// TMA and an MMA warp.  Tiles are staged by TMA
// with 128-byte swizzle exactly as in the forward kernel; every mbarrier wait is bounded.
#pragma once
#include <cuda.h>
#include <cstdint>

#include "attn_fwd_kernel.cuh"

namespace attn {
namespace bwd {

constexpr int kThreads = 320;   // dK/dV kernel
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
// Streamed tiles in flight.  dK/dV kernel: one ring of 4 slots (Q_i, dO_i alternate).  dQ kernel:
// two K slots and one V slot (K_j lives from S_j to the last dQ += dS_j K_j, V_j only feeds the
// dP_j products).
constexpr int kRing = 4;
constexpr int kDkdvRing = 4;

struct Params {
  const void* lse;     // fp32 [B,H,Sq], natural log (the forward's output)
  float* delta;        // fp32 [B,H,Sq]
  void* out0;          // dQ kernel: dQ; dK/dV kernel: dK        BF16 [B,H,S,128]
  void* out1;          // dK/dV kernel: dV
  int sq, sk;
  int q_tiles, kv_tiles;
  int q_valid_last, kv_valid_last;   // valid rows in the last Q / K/V tile, 1..128
  int bh;
  int heads;           // H
  int bshd;            // 1: Q/K/V/dO and the gradients are [B,S,H,D] (lse, delta stay [B,H,S])
  int causal;
  float scale;         // softmax scale
  float scale_log2;    // scale * log2(e)
};

struct alignas(8) SmemCtl {
  uint64_t fixed_full;          // the CTA's own two resident tiles are in SMEM
  uint64_t ring_full[kRing], ring_empty[kRing];
  uint64_t acc_full;            // MMA -> elementwise: the accumulators are final
  // dK/dV kernel, per Q tile: S^T and dP^T in TMEM (MMA -> elementwise), P^T and dS^T written
  // back (elementwise -> MMA).  Separate barriers let dV += P^T dO start before dS^T exists.
  uint64_t s_full, dp_full, p_ready, ds_ready;
  uint64_t epi_full;            // dK/dV kernel: the elementwise warps staged dK, dV in SMEM
  // dQ kernel over a pair of Q tiles (a, b), per tile t: S_t in TMEM (dq_s_full), S_t read so
  // dP_t may overwrite it (dq_x_read), dP_t in TMEM (dq_dp_full), dS_t written back
  // (dq_ds_ready); dq_do_full: both dO tiles resident.
  uint64_t dq_s_full[2], dq_x_read[2], dq_dp_full[2], dq_ds_ready[2], dq_do_full;
  uint64_t vec_sync;            // elementwise warps exchanged per-column vectors (dK/dV)
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort_flag;
  float lse2[2][kBlockM];       // dK/dV kernel: -LSE * log2(e) of the current Q tile's columns
  float dlt[2][kBlockM];        // dK/dV kernel: delta of the current Q tile's columns
};

// dK/dV kernel: 2 resident + 4 ring tiles, control block, 1 KiB to align the base by hand.
constexpr uint32_t kCtlOffsetDkdv = (2 + kDkdvRing) * kTileBytes;
constexpr uint32_t kSmemBytesDkdv = kCtlOffsetDkdv + sizeof(SmemCtl) + 1024;
constexpr unsigned kStatusSmemAlign = 1u << 6;   // dynamic shared memory not 1024-aligned

// Bounded waits, as in the forward kernel: all 32 lanes call; false = timed out or aborted.
struct Sync {
  SmemCtl* ctl;
  uint32_t lane;
  __device__ uint32_t bar(const uint64_t& b) const { return ptx::smem_u32(&b); }
  __device__ bool wait(const uint64_t& b, uint32_t parity, unsigned role_bit) const {
    const uint32_t addr = bar(b);
    if (__all_sync(0xffffffffu, ptx::mbar_try_wait(addr, parity))) return true;
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
  __device__ void arrive(const uint64_t& b) const {
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(bar(b));
  }
};

// ------------------------------------------------------------------ delta = rowsum(dO o O)
// delta[row] for rows in [B,H,Sq] order; O and dO are [B,H,Sq,128] or, with bshd, [B,Sq,H,128].
__global__ void __launch_bounds__(256) attn_bwd_delta_kernel(const uint16_t* __restrict__ o,
                                                             const uint16_t* __restrict__ dout,
                                                             float* __restrict__ delta,
                                                             int64_t rows, int heads, int sq,
                                                             int bshd) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const uint32_t lane = threadIdx.x & 31u;
  if (row >= rows) return;
  int64_t src = row;
  if (bshd) {
    const int64_t bh = row / sq, s = row - bh * sq;
    const int64_t b = bh / heads, h = bh - b * heads;
    src = (b * sq + s) * heads + h;
  }
  const uint2 a = *reinterpret_cast<const uint2*>(o + src * kHeadDim + lane * 4);
  const uint2 b = *reinterpret_cast<const uint2*>(dout + src * kHeadDim + lane * 4);
  auto lo = [](uint32_t x) { return __uint_as_float(x << 16); };
  auto hi = [](uint32_t x) { return __uint_as_float(x & 0xffff0000u); };
  float acc = lo(a.x) * lo(b.x);
  acc = fmaf(hi(a.x), hi(b.x), acc);
  acc = fmaf(lo(a.y), lo(b.y), acc);
  acc = fmaf(hi(a.y), hi(b.y), acc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) delta[row] = acc;
}

// ------------------------------------------------------------------ shared pieces
// D[tmem cols d] (+)= A[smem, K-major SW128] * B[smem, K-major SW128]^T, 128x128x128.
__device__ __forceinline__ void mma_kmajor(uint32_t d, uint32_t a_smem, uint32_t b_smem) {
  constexpr uint32_t idesc = make_idesc_bf16(128, 128, 0);
  const uint64_t a0 = smem_desc_sw128(a_smem, 16, 1024);
  const uint64_t b0 = smem_desc_sw128(b_smem, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < kHeadDim / 16; ++kk) {
    const uint32_t off16 = ((kk >> 2) * kSlabBytes + (kk & 3) * 32) >> 4;
    ptx::mma_ss(d, a0 + off16, b0 + off16, idesc, kk > 0);
  }
}

// D[tmem cols d] (+)= A[tmem cols a, packed BF16 128x128] * B[smem 128 rows x 128, MN-major].
__device__ __forceinline__ void mma_tmem_a(uint32_t d, uint32_t a, uint32_t b_smem,
                                           bool accumulate) {
  constexpr uint32_t idesc = make_idesc_bf16(128, 128, 1);
  const uint64_t b0 = smem_desc_sw128(b_smem, kSlabBytes, 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    ptx::mma_ts(d, a + kk * 8, b0 + ((kk * 16 * 128) >> 4), idesc,
                (accumulate || kk > 0) ? 1u : 0u);
}

// Load two 64-column boxes (one 128-row tile) of head bh: from the 3-D map (128, S, B*H) of a
// [B,H,S,128] tensor (heads4d == 0) or the 4-D map (128, H, S, B) of a [B,S,H,128] tensor
// (heads4d == H).
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* tm, uint32_t bar,
                                          int row, int bh, int heads4d) {
  if (heads4d) {
    const int b = bh / heads4d, h = bh - b * heads4d;
    ptx::tma_load_4d(dst, tm, bar, 0, h, row, b);
    ptx::tma_load_4d(dst + kSlabBytes, tm, bar, 64, h, row, b);
  } else {
    ptx::tma_load_3d(dst, tm, bar, 0, row, bh);
    ptx::tma_load_3d(dst + kSlabBytes, tm, bar, 64, row, bh);
  }
}

// Streamed Q/dO tiles of the dK/dV kernel are prefetched into L2 this many tiles ahead of their
// loads (the K/V stream of the dQ kernel gains nothing from it).
constexpr int kDkdvPrefetch = 2;

// L2 prefetch of one 128-row tile (both 64-column boxes) of head bh.
__device__ __forceinline__ void prefetch_tile(const CUtensorMap* tm, int row, int bh, int heads4d) {
  if (heads4d) {
    const int b = bh / heads4d, h = bh - b * heads4d;
    ptx::tma_prefetch_4d(tm, 0, h, row, b);
    ptx::tma_prefetch_4d(tm, 64, h, row, b);
  } else {
    ptx::tma_prefetch_3d(tm, 0, row, bh);
    ptx::tma_prefetch_3d(tm, 64, row, bh);
  }
}

// Byte offset of row `row` of head bh in a BF16 [B,H,S,128] or (kBshd) [B,S,H,128] tensor.
template <bool kBshd>
__device__ __forceinline__ size_t row_offset(const Params& p, int bh, int row, int seq) {
  if (kBshd) {
    const int b = bh / p.heads, h = bh - b * p.heads;
    return ((static_cast<size_t>(b) * seq + row) * p.heads + h) * (kHeadDim * 2);
  }
  return (static_cast<size_t>(bh) * seq + row) * (kHeadDim * 2);
}

// Write 16 fp32 accumulator columns as BF16 (times `mul`) to a global row.
__device__ __forceinline__ void store_cols16(uint8_t* out, const uint32_t (&r)[16], float mul) {
  uint32_t pk[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    pk[i] = ptx::pack_bf16x2(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
  ptx::st_global_v4(out, pk[0], pk[1], pk[2], pk[3]);
  ptx::st_global_v4(out + 16, pk[4], pk[5], pk[6], pk[7]);
}

__device__ __forceinline__ void zero_row(uint8_t* out) {
#pragma unroll
  for (int i = 0; i < 16; ++i) ptx::st_global_v4(out + 16 * i, 0u, 0u, 0u, 0u);
}

struct Layout {
  SmemCtl* ctl;
  int heads4d;     // H for [B,S,H,D] tensors (4-D tensor maps), 0 for [B,H,S,D]
  uint32_t base;   // 1024-aligned shared address of the first resident tile
  __device__ uint32_t fixed(int i) const { return base + i * kTileBytes; }
  __device__ uint32_t ring(int s) const { return base + (2 + s) * kTileBytes; }
};

__device__ __forceinline__ Layout setup(uint8_t* smem_raw, uint32_t ctl_offset, const Params& p) {
  const uint32_t raw = ptx::smem_u32(smem_raw);
  Layout L;
  L.heads4d = p.bshd ? p.heads : 0;
  L.base = (raw + 1023u) & ~1023u;
  L.ctl = reinterpret_cast<SmemCtl*>(smem_raw + (L.base - raw) + ctl_offset);
  return L;
}

__device__ __forceinline__ void init_barriers(SmemCtl* ctl, const Sync& s) {
  ptx::mbar_init(s.bar(ctl->fixed_full), 1);
  for (int i = 0; i < kRing; ++i) {
    ptx::mbar_init(s.bar(ctl->ring_full[i]), 1);
    ptx::mbar_init(s.bar(ctl->ring_empty[i]), 1);
  }
  ptx::mbar_init(s.bar(ctl->acc_full), 1);
  ptx::mbar_init(s.bar(ctl->s_full), 1);
  ptx::mbar_init(s.bar(ctl->dp_full), 1);
  ptx::mbar_init(s.bar(ctl->p_ready), 8);
  ptx::mbar_init(s.bar(ctl->ds_ready), 8);
  ptx::mbar_init(s.bar(ctl->vec_sync), 8);
  ptx::mbar_init(s.bar(ctl->epi_full), 8);
  for (int t = 0; t < 2; ++t) {
    ptx::mbar_init(s.bar(ctl->dq_s_full[t]), 1);
    ptx::mbar_init(s.bar(ctl->dq_x_read[t]), 4);
    ptx::mbar_init(s.bar(ctl->dq_dp_full[t]), 1);
    ptx::mbar_init(s.bar(ctl->dq_ds_ready[t]), 4);
  }
  ptx::mbar_init(s.bar(ctl->dq_do_full), 1);
  ptx::mbar_init(s.bar(ctl->drain), 1);
  ctl->abort_flag = 0;
  ptx::fence_mbar_init();
}

// TMA warp: the two resident tiles, then `n` pairs of streamed tiles (first map, second map)
// for tile indices t0 .. t0+n-1, through the ring.
__device__ __forceinline__ void stream_tiles(const Layout& L, const Sync& s, const CUtensorMap* f0,
                                             const CUtensorMap* f1, int frow, const CUtensorMap* r0,
                                             const CUtensorMap* r1, int t0, int n, int bh) {
  SmemCtl* ctl = L.ctl;
  if (s.lane == 0) {
    const uint32_t fb = s.bar(ctl->fixed_full);
    ptx::mbar_arrive_expect_tx(fb, 2 * kTileBytes);
    load_tile(L.fixed(0), f0, fb, frow, bh, L.heads4d);
    load_tile(L.fixed(1), f1, fb, frow, bh, L.heads4d);
  }
  __syncwarp();
  int slot = 0;
  uint32_t phase = 0, used = 0, last_par = 0;
  bool ok = true;
  if (s.lane == 0)
    for (int t = 1; t < kDkdvPrefetch && t < n; ++t) {
      prefetch_tile(r0, (t0 + t) * kBlockM, bh, L.heads4d);
      prefetch_tile(r1, (t0 + t) * kBlockM, bh, L.heads4d);
    }
  for (int t = 0; ok && t < 2 * n; ++t) {
    if ((t & 1) && s.lane == 0 && (t >> 1) + kDkdvPrefetch < n) {
      prefetch_tile(r0, (t0 + (t >> 1) + kDkdvPrefetch) * kBlockM, bh, L.heads4d);
      prefetch_tile(r1, (t0 + (t >> 1) + kDkdvPrefetch) * kBlockM, bh, L.heads4d);
    }
    if (!(ok = s.wait(ctl->ring_empty[slot], phase ^ 1u, kStatusTimeoutLoad))) break;
    if (s.lane == 0) {
      const uint32_t fb = s.bar(ctl->ring_full[slot]);
      ptx::mbar_arrive_expect_tx(fb, kTileBytes);
      load_tile(L.ring(slot), (t & 1) ? r1 : r0, fb, (t0 + (t >> 1)) * kBlockM, bh, L.heads4d);
    }
    __syncwarp();
    used |= 1u << slot;
    last_par = (last_par & ~(1u << slot)) | (phase << slot);
    if (++slot == kDkdvRing) { slot = 0; phase ^= 1u; }
  }
  if (!ok) {
    for (int i = 0; i < kDkdvRing; ++i)
      if ((used >> i) & 1u) s.drain_wait(ctl->ring_full[i], (last_par >> i) & 1u);
  }
  s.drain_wait(ctl->fixed_full, 0);
}

// ------------------------------------------------------------------ dQ kernel
// One CTA per pair of 128-row Q tiles (a = 2p, b = 2p + 1) of one head.  Each streamed K/V tile
// feeds six products (S, dP and dQ += dS K for both tiles) instead of three, which halves the
// streamed bytes per product, and the tensor pipe runs one tile's products while the other
// tile's elementwise warps work (the two-stage overlap of the forward kernel).
// TMEM: X_a [0,128) and X_b [128,256) hold S, then dP over it once the elementwise warps have read
// S, then packed BF16 dS over its lower 64 columns; dQ_a [256,384), dQ_b [384,512).
// SMEM: Q_a, dO_a, Q_b, dO_b resident; a ring of two K tiles and one V tile.
// Warps 0-3 elementwise for tile a, 4-7 for tile b, 8 TMA, 9 tcgen05.mma issue, 10-11 idle (the
// register split below works on whole warpgroups).
constexpr int kDqThreads = 384;
constexpr int kDqLoadWarp = 8;
constexpr int kDqMmaWarp = 9;
// Register split (setmaxnreg): launched with 168 registers per thread (65536 / 384, rounded down
// to the allocation unit; the host checks the compiled count), the two elementwise warpgroups
// take 224 (a full 128-column row of P plus a 32-column chunk of dP), the third gives back to 56:
// (2 * 224 + 56) * 128 == 168 * 384.
constexpr uint32_t kDqRegLaunch = 168, kDqRegEw = 224, kDqRegMisc = 56;
static_assert((2 * kDqRegEw + kDqRegMisc) * 128 == kDqRegLaunch * kDqThreads, "register split");
constexpr int kDqKRing = 2;                        // ring slots 0..1: K tiles; slot 2: the V tile
constexpr uint32_t kColDQ = 256;
constexpr uint32_t kCtlOffsetDq = (4 + kDqKRing + 1) * kTileBytes;
constexpr uint32_t kSmemBytesDq = kCtlOffsetDq + sizeof(SmemCtl);
static_assert(kSmemBytesDq <= 227 * 1024, "dQ kernel shared memory exceeds a CTA's 227 KiB");

// Work of CTA blockIdx.x: head bh, first Q tile qa, K/V tiles n[t] each tile t of the pair sees
// (0 for a tile past the end).  Causal: heaviest pairs first.
__device__ __forceinline__ void dq_item(const Params& p, int& bh, int& qa, int (&n)[2]) {
  const int pairs = (p.q_tiles + 1) >> 1;
  int pr;
  if (p.causal) {
    pr = pairs - 1 - static_cast<int>(blockIdx.x) / p.bh;
    bh = static_cast<int>(blockIdx.x) % p.bh;
  } else {
    bh = static_cast<int>(blockIdx.x) / pairs;
    pr = static_cast<int>(blockIdx.x) % pairs;
  }
  qa = 2 * pr;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qt = qa + t;
    n[t] = qt >= p.q_tiles ? 0 : (p.causal ? min(qt + 1, p.kv_tiles) : p.kv_tiles);
  }
}

// Ring slot r of the paired kernel (after the four resident tiles).
__device__ __forceinline__ uint32_t dq_ring(const Layout& L, int r) { return L.ring(2 + r); }

// TMA warp: Q_a, Q_b, K_0, dO_a, dO_b, V_0, then K_j, V_j for j = 1..nkv-1.
__device__ __forceinline__ void dq_loads(const Layout& L, const Sync& s, const CUtensorMap* tm_q,
                                          const CUtensorMap* tm_do, const CUtensorMap* tm_k,
                                          const CUtensorMap* tm_v, int qa, int ntiles, int nkv,
                                          int bh) {
  SmemCtl* ctl = L.ctl;
  auto fixed_pair = [&](const uint64_t& b, const CUtensorMap* tm, int first) {
    if (s.lane == 0) {
      const uint32_t fb = s.bar(b);
      ptx::mbar_arrive_expect_tx(fb, ntiles * kTileBytes);
      for (int t = 0; t < ntiles; ++t)
        load_tile(L.fixed(2 * t + first), tm, fb, (qa + t) * kBlockM, bh, L.heads4d);
    }
    __syncwarp();
  };
  fixed_pair(ctl->fixed_full, tm_q, 0);
  int ks = 0;
  uint32_t kph = 0, vph = 0, used = 0, last_par = 0;
  bool ok = true;
  auto load = [&](int slot, uint32_t ph, const CUtensorMap* tm, int row) -> bool {
    if (!s.wait(ctl->ring_empty[slot], ph ^ 1u, kStatusTimeoutLoad)) return false;
    if (s.lane == 0) {
      const uint32_t fb = s.bar(ctl->ring_full[slot]);
      ptx::mbar_arrive_expect_tx(fb, kTileBytes);
      load_tile(dq_ring(L, slot), tm, fb, row, bh, L.heads4d);
    }
    __syncwarp();
    used |= 1u << slot;
    last_par = (last_par & ~(1u << slot)) | (ph << slot);
    return true;
  };
  for (int j = 0; ok && j < nkv; ++j) {
    if (!(ok = load(ks, kph, tm_k, j * kBlockN))) break;
    if (++ks == kDqKRing) { ks = 0; kph ^= 1u; }
    if (j == 0) fixed_pair(ctl->dq_do_full, tm_do, 1);
    if (!(ok = load(kDqKRing, vph, tm_v, j * kBlockN))) break;
    vph ^= 1u;
  }
  if (!ok) {
    for (int i = 0; i <= kDqKRing; ++i)
      if ((used >> i) & 1u) s.drain_wait(ctl->ring_full[i], (last_par >> i) & 1u);
  }
  s.drain_wait(ctl->fixed_full, 0);
  if (nkv > 0) s.drain_wait(ctl->dq_do_full, 0);
}

// P of one S row (128 columns) for the dQ kernel: exp2(S * scale_log2 - LSE * log2 e), with
// kSel, 0 at columns >= valid.
template <bool kSel>
__device__ __forceinline__ void dq_p(const uint32_t (&sr)[4][32], float2 sl2, float2 nl, int valid,
                                     float2 (&pf)[4][16]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 e = ptx::ffma2(
          make_float2(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])), sl2, nl);
      pf[c][i].x = (!kSel || 32 * c + 2 * i < valid) ? ptx::ex2_ftz(e.x) : 0.f;
      pf[c][i].y = (!kSel || 32 * c + 2 * i + 1 < valid) ? ptx::ex2_ftz(e.y) : 0.f;
    }
  }
}

// kMask: the launch may have masked keys (a ragged last K/V tile or the causal mask); the
// instantiation for launches without any has no masking code.
template <bool kMask, bool kBshd>
__global__ void __launch_bounds__(kDqThreads, 1)
attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((ptx::smem_u32(smem_raw) & 1023u) != 0) {   // no room for realignment: skip the CTA
    if (threadIdx.x == 0) atomicOr(&g_attn_status, kStatusSmemAlign);
    return;
  }
  Layout L = setup(smem_raw, kCtlOffsetDq, p);
  L.heads4d = kBshd ? p.heads : 0;   // the layout is known at compile time: one tensor-map rank
  SmemCtl* ctl = L.ctl;
  const uint32_t warp = threadIdx.x >> 5;
  Sync s{ctl, threadIdx.x & 31u};
  int bh, qa, n[2];
  dq_item(p, bh, qa, n);
  const int nkv = n[0] > n[1] ? n[0] : n[1];

  if (threadIdx.x == 0) init_barriers(ctl, s);
  if (warp == kDqMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&ctl->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_alloc_base = ctl->tmem_base;
  const bool tmem_ok = tmem_alloc_base == kTmemBase;
  if (!tmem_ok && threadIdx.x == 0) atomicOr(&g_attn_status, kStatusTmemBase);

  if (tmem_ok && warp >= 8) ptx::setmaxnreg_dec<kDqRegMisc>();
  if (tmem_ok && warp == kDqLoadWarp) {
    dq_loads(L, s, &tm_q, &tm_do, &tm_k, &tm_v, qa, n[1] > 0 ? 2 : 1, nkv, bh);
  } else if (tmem_ok && warp == kDqMmaWarp) {
    // Per K/V tile j the tensor pipe runs dP_a(j), dP_b(j), dQ_a(j), S_a(j+1), dQ_b(j), S_b(j+1):
    // S_t(j+1) reuses X_t once dQ_t(j) has read dS_t(j) (tcgen05.mma from one thread run in
    // order), and a tile past its last K/V tile (causal) drops out.
    const bool leader = ptx::elect_one();
    bool ok = s.wait(ctl->fixed_full, 0, kStatusTimeoutMma);
    int ks = 0;
    uint32_t kph = 0, vph = 0;
    auto next_k = [&](int& out) -> bool {
      out = ks;
      const bool r = s.wait(ctl->ring_full[ks], kph, kStatusTimeoutMma);
      if (++ks == kDqKRing) { ks = 0; kph ^= 1u; }
      return r;
    };
    auto issue_s = [&](int t, int kslot) {
      ptx::tc_fence_after();
      if (leader) {
        mma_kmajor(kTmemBase + 128u * t, L.fixed(2 * t), dq_ring(L, kslot));   // S_t = Q_t K^T
        ptx::mma_commit(s.bar(ctl->dq_s_full[t]));
      }
      __syncwarp();
    };
    int kcur = 0;
    ok = ok && next_k(kcur);
    if (ok) {
      for (int t = 0; t < 2; ++t)
        if (n[t] > 0) issue_s(t, kcur);
    }
    ok = ok && s.wait(ctl->dq_do_full, 0, kStatusTimeoutMma);
    for (int j = 0; ok && j < nkv; ++j) {
      if (!(ok = s.wait(ctl->ring_full[kDqKRing], vph, kStatusTimeoutMma))) break;
      vph ^= 1u;
      for (int t = 0; ok && t < 2; ++t) {
        if (j >= n[t]) continue;
        if (!(ok = s.wait(ctl->dq_x_read[t], j & 1u, kStatusTimeoutMma))) break;
        ptx::tc_fence_after();
        if (leader) {
          mma_kmajor(kTmemBase + 128u * t, L.fixed(2 * t + 1), dq_ring(L, kDqKRing));  // dP_t = dO_t V^T
          ptx::mma_commit(s.bar(ctl->dq_dp_full[t]));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (leader) ptx::mma_commit(s.bar(ctl->ring_empty[kDqKRing]));
      __syncwarp();
      int knext = -1;
      for (int t = 0; ok && t < 2; ++t) {
        if (j >= n[t]) continue;
        if (!(ok = s.wait(ctl->dq_ds_ready[t], j & 1u, kStatusTimeoutMma))) break;
        ptx::tc_fence_after();
        if (leader) {
          mma_tmem_a(kTmemBase + kColDQ + 128u * t, kTmemBase + 128u * t, dq_ring(L, kcur), j > 0);  // dQ_t += dS_t K
          if (t == 1 || j >= n[1]) ptx::mma_commit(s.bar(ctl->ring_empty[kcur]));
        }
        __syncwarp();
        if (j + 1 < n[t]) {
          if (knext < 0 && !(ok = next_k(knext))) break;
          issue_s(t, knext);
        }
      }
      kcur = knext;
    }
    if (leader) {
      if (ok) ptx::mma_commit(s.bar(ctl->acc_full));
      ptx::mma_commit(s.bar(ctl->drain));
    }
    __syncwarp();
    s.drain_wait(ctl->drain, 0);
  } else if (tmem_ok && warp < 8) {
    ptx::setmaxnreg_inc<kDqRegEw>();
    const int t = static_cast<int>(warp >> 2);
    const uint32_t row_base = 32u * (warp & 3u);
    const int r = static_cast<int>(row_base + s.lane);
    const int qt = qa + t;
    const int qrow = qt * kBlockM + r;
    const bool row_ok = n[t] > 0 && qrow < p.sq;
    const size_t gi = static_cast<size_t>(bh) * p.sq + qrow;
    const float lse2 = row_ok ? static_cast<const float*>(p.lse)[gi] * 1.4426950408889634f : 0.f;
    const float dlt = row_ok ? p.delta[gi] : 0.f;
    const uint32_t x = kTmemBase + (row_base << 16) + 128u * t;
    bool ok = true;
    for (int j = 0; ok && j < n[t]; ++j) {
      if (!(ok = s.wait(ctl->dq_s_full[t], j & 1u, kStatusTimeoutSoftmax))) break;
      ptx::tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld_32x32b_x32(x + 32 * c, sr[c]);
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      s.arrive(ctl->dq_x_read[t]);   // dP_t may now overwrite S_t
      // P = exp2(S * scale_log2 - LSE * log2 e), 0 past `valid`; kept in fp32 for dS.  Only the
      // tiles with masked keys (the ragged last one, the causal diagonal) take the selects.
      float2 pf[4][16];
      const float2 sl2 = make_float2(p.scale_log2, p.scale_log2), nl = make_float2(-lse2, -lse2);
      const bool masked_tile = kMask && ((j == p.kv_tiles - 1 && p.kv_valid_last < kBlockN) ||
                                         (p.causal && j == qt));
      if (masked_tile) {
        int valid = j == p.kv_tiles - 1 ? p.kv_valid_last : kBlockN;
        if (p.causal && j == qt) valid = min(valid, r + 1);
        dq_p<true>(sr, sl2, nl, valid, pf);
      } else {
        dq_p<false>(sr, sl2, nl, kBlockN, pf);
      }
      // dS = P o (dP - delta), packed BF16 into columns 16c..16c+15 once dP columns
      // 32c..32c+31 are in registers: every column written has been read.  The load of the
      // next 32 dP columns is in flight while a chunk is computed and stored.
      if (!(ok = s.wait(ctl->dq_dp_full[t], j & 1u, kStatusTimeoutSoftmax))) break;
      ptx::tc_fence_after();
      const float2 nd = make_float2(-dlt, -dlt);
      uint32_t dr[2][32];
      ptx::tmem_ld_32x32b_x32(x, dr[0]);
      ptx::tmem_wait_ld_regs(dr[0]);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (c < 3) ptx::tmem_ld_32x32b_x32(x + 32 * (c + 1), dr[(c + 1) & 1]);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 d = ptx::fadd2(make_float2(__uint_as_float(dr[c & 1][2 * i]),
                                                  __uint_as_float(dr[c & 1][2 * i + 1])), nd);
          const float2 v = ptx::fmul2(pf[c][i], d);
          pk[i] = ptx::pack_bf16x2(v.x, v.y);
        }
        ptx::tmem_st_32x32b_x16(x + 16 * c, pk);
        if (c < 3) ptx::tmem_wait_ld_regs(dr[(c + 1) & 1]);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      s.arrive(ctl->dq_ds_ready[t]);
    }
    if (ok && n[t] > 0 && s.wait(ctl->acc_full, 0, kStatusTimeoutSoftmax)) {
      ptx::tc_fence_after();
      uint8_t* out = static_cast<uint8_t*>(p.out0) + row_offset<kBshd>(p, bh, qrow, p.sq);
      const uint32_t acc_col = kTmemBase + (row_base << 16) + kColDQ + 128u * t;
#pragma unroll 2
      for (int c = 0; c < 8; ++c) {
        uint32_t acc[16];
        ptx::tmem_ld_32x32b_x16(acc_col + 16 * c, acc);
        ptx::tmem_wait_ld();
        if (row_ok) store_cols16(out + 32 * c, acc, p.scale);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kDqMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_alloc_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ dK/dV kernel
// TMEM: S^T [0,128) with packed BF16 P^T over 32..95, dP^T [128,256) with packed BF16 dS^T over
// 160..223, dK [256,384), dV [384,512).  The packed columns of query columns [64g, 64g+64) sit
// inside S^T (dP^T) columns [64g, 64g+64), the ones elementwise warpgroup g reads.
constexpr uint32_t kColST = 0, kColDPT = 128, kColDK = 256, kColDV = 384;
constexpr uint32_t kColPT = 32;   // packed operand offset inside S^T and dP^T

__device__ __forceinline__ void dkdv_item(const Params& p, int& bh, int& kt, int& q0, int& nq) {
  if (p.causal) {   // heaviest K/V tiles (earliest keys) first
    kt = static_cast<int>(blockIdx.x) / p.bh;
    bh = static_cast<int>(blockIdx.x) % p.bh;
    q0 = kt;        // Q tiles kt.. see keys of K/V tile kt (top-left alignment)
    nq = kt < p.q_tiles ? p.q_tiles - kt : 0;
  } else {
    bh = static_cast<int>(blockIdx.x) / p.kv_tiles;
    kt = static_cast<int>(blockIdx.x) % p.kv_tiles;
    q0 = 0;
    nq = p.q_tiles;
  }
}

// P^T of 64 columns (query columns c0..c0+63 of key row r) for the dK/dV kernel: exp2(S^T *
// scale_log2 - LSE_col * log2 e); with kDiag, 0 at query columns c < r (the causal diagonal).
template <bool kDiag>
__device__ __forceinline__ void dkdv_p(const uint32_t (&xr)[2][32], const float* va, float2 sl2,
                                       int c0, int r, float2 (&pf)[2][16]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int i2 = 0; i2 < 16; ++i2) {
      const int col = c0 + 32 * h + 2 * i2;
      const float2 a = *reinterpret_cast<const float2*>(va + 32 * h + 2 * i2);
      const float2 e = ptx::ffma2(make_float2(__uint_as_float(xr[h][2 * i2]),
                                              __uint_as_float(xr[h][2 * i2 + 1])), sl2, a);
      float p0 = ptx::ex2_ftz(e.x);
      float p1 = ptx::ex2_ftz(e.y);
      if (kDiag) {
        p0 = col < r ? 0.f : p0;
        p1 = col + 1 < r ? 0.f : p1;
      }
      pf[h][i2] = make_float2(p0, p1);
    }
  }
}

// kMask: the launch uses the causal mask (the only per-element masking this kernel does).
template <bool kMask, bool kBshd>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                     const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Layout L = setup(smem_raw, kCtlOffsetDkdv, p);
  L.heads4d = kBshd ? p.heads : 0;   // the layout is known at compile time: one tensor-map rank
  SmemCtl* ctl = L.ctl;
  const uint32_t warp = threadIdx.x >> 5;
  Sync s{ctl, threadIdx.x & 31u};
  int bh, kt, q0, nq;
  dkdv_item(p, bh, kt, q0, nq);

  if (threadIdx.x == 0) init_barriers(ctl, s);
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&ctl->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_alloc_base = ctl->tmem_base;
  const bool tmem_ok = tmem_alloc_base == kTmemBase;
  if (!tmem_ok && threadIdx.x == 0) atomicOr(&g_attn_status, kStatusTmemBase);

  if (tmem_ok && warp == kLoadWarp && nq > 0) {
    // resident: K, V of this tile; streamed: Q_i, dO_i
    stream_tiles(L, s, &tm_k, &tm_v, kt * kBlockN, &tm_q, &tm_do, q0, nq, bh);
  } else if (tmem_ok && warp == kMmaWarp && nq > 0) {
    // Per Q tile i the tensor pipe runs dV(i), S(i+1), dK(i), dP(i+1): S^T(i+1) overwrites
    // P^T(i) only after dV(i) has been issued, dP^T(i+1) overwrites dS^T(i) only after dK(i),
    // and the elementwise work on tile i+1 overlaps the products of tile i.
    const bool leader = ptx::elect_one();
    bool ok = s.wait(ctl->fixed_full, 0, kStatusTimeoutMma);
    int slot = 0;
    uint32_t phase = 0;
    auto next_slot = [&](int& out) -> bool {
      out = slot;
      const bool r = s.wait(ctl->ring_full[slot], phase, kStatusTimeoutMma);
      if (++slot == kDkdvRing) { slot = 0; phase ^= 1u; }
      return r;
    };
    int qs = 0, ds = 0;
    ok = ok && next_slot(qs) && next_slot(ds);
    if (ok) {
      ptx::tc_fence_after();
      if (leader) {
        mma_kmajor(kTmemBase + kColST, L.fixed(0), L.ring(qs));    // S^T = K Q^T
        ptx::mma_commit(s.bar(ctl->s_full));
        mma_kmajor(kTmemBase + kColDPT, L.fixed(1), L.ring(ds));   // dP^T = V dO^T
        ptx::mma_commit(s.bar(ctl->dp_full));
      }
      __syncwarp();
    }
    for (int i = 0; ok && i < nq; ++i) {
      const bool more = i + 1 < nq;
      if (!(ok = s.wait(ctl->p_ready, i & 1u, kStatusTimeoutMma))) break;
      ptx::tc_fence_after();
      if (leader) {
        mma_tmem_a(kTmemBase + kColDV, kTmemBase + kColST + kColPT, L.ring(ds), i > 0);   // dV += P^T dO
        ptx::mma_commit(s.bar(ctl->ring_empty[ds]));
      }
      __syncwarp();
      int qn = 0, dn = 0;
      if (more) {
        if (!(ok = next_slot(qn))) break;
        ptx::tc_fence_after();
        if (leader) {
          mma_kmajor(kTmemBase + kColST, L.fixed(0), L.ring(qn));
          ptx::mma_commit(s.bar(ctl->s_full));
        }
        __syncwarp();
      }
      if (!(ok = s.wait(ctl->ds_ready, i & 1u, kStatusTimeoutMma))) break;
      ptx::tc_fence_after();
      if (leader) {
        mma_tmem_a(kTmemBase + kColDK, kTmemBase + kColDPT + kColPT, L.ring(qs), i > 0);  // dK += dS^T Q
        ptx::mma_commit(s.bar(ctl->ring_empty[qs]));
        if (!more) ptx::mma_commit(s.bar(ctl->acc_full));
      }
      __syncwarp();
      if (more) {
        if (!(ok = next_slot(dn))) break;
        ptx::tc_fence_after();
        if (leader) {
          mma_kmajor(kTmemBase + kColDPT, L.fixed(1), L.ring(dn));
          ptx::mma_commit(s.bar(ctl->dp_full));
        }
        __syncwarp();
      }
      qs = qn;
      ds = dn;
    }
    if (leader) ptx::mma_commit(s.bar(ctl->drain));
    __syncwarp();
    s.drain_wait(ctl->drain, 0);
  } else if (tmem_ok && warp < 8) {
    // Two elementwise warpgroups: warpgroup g works query columns [64g, 64g+64) of every key row
    // (one TMEM lane per thread), so a pass is 64 columns per thread.
    const int g = static_cast<int>(warp >> 2);
    const uint32_t row_base = 32u * (warp & 3u);
    const int r = static_cast<int>(row_base + s.lane);   // key row within the tile
    const int krow = kt * kBlockN + r;
    const uint32_t lane_off = row_base << 16;
    const int c0 = 64 * g;                               // this thread's first query column
    const float* lse = static_cast<const float*>(p.lse) + static_cast<size_t>(bh) * p.sq;
    const float* dl = p.delta + static_cast<size_t>(bh) * p.sq;
    // Column vectors of Q tile i, one value per thread: warpgroup 0 stages -LSE*log2 e of query
    // column r, warpgroup 1 its delta; masked query columns (past Sq) get -LSE = -inf, so P = 0.
    // The next tile's value is loaded a tile ahead from an in-range address and first used when
    // it is staged, so the load's latency never stalls the warp.
    const float* src = g == 0 ? lse : dl;
    auto fetch = [&](int i) -> float {
      const int qi = (q0 + i) * kBlockM + r;
      return src[qi < p.sq ? qi : p.sq - 1];
    };
    auto stage = [&](int i, float raw) -> float {
      const int qi = (q0 + i) * kBlockM + r;
      if (g == 0) return qi < p.sq ? -(raw * 1.4426950408889634f) : __int_as_float(0xff800000);
      return qi < p.sq ? raw : 0.f;
    };
    float* vec = g == 0 ? &ctl->lse2[0][0] : &ctl->dlt[0][0];
    bool ok = true;
    float nv = 0.f;
    if (nq > 0) {
      vec[r] = stage(0, fetch(0));
      s.arrive(ctl->vec_sync);
    }
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    const uint32_t st_cols = kTmemBase + lane_off + kColST, dpt_cols = kTmemBase + lane_off + kColDPT;
    for (int i = 0; ok && i < nq; ++i) {
      const int par = i & 1;
      if (i + 1 < nq) nv = fetch(i + 1);   // next tile's vector, in flight meanwhile
      if (!(ok = s.wait(ctl->vec_sync, par, kStatusTimeoutSoftmax))) break;
      if (!(ok = s.wait(ctl->s_full, par, kStatusTimeoutSoftmax))) break;
      ptx::tc_fence_after();
      const bool diag = kMask && p.causal && q0 + i == kt;   // query column c < key row r is masked
      const float* va = ctl->lse2[par] + c0;
      const float* vd = ctl->dlt[par] + c0;
      // P^T = exp2(S^T * scale_log2 + (-LSE_col * log2 e)), kept in fp32 for dS^T.  The packed
      // BF16 P^T of columns c0.. lands on columns kColPT + c0/2.., inside this thread's own 64
      // columns, written once all of them are in registers.
      uint32_t xr[2][32];
      ptx::tmem_ld_32x32b_x32(st_cols + c0, xr[0]);
      ptx::tmem_ld_32x32b_x32(st_cols + c0 + 32, xr[1]);
      ptx::tmem_wait_ld_regs(xr[0]);
      ptx::tmem_wait_ld_regs(xr[1]);
      float2 pf[2][16];
      if (diag) dkdv_p<true>(xr, va, sl2, c0, r, pf);   // only the causal diagonal tile selects
      else dkdv_p<false>(xr, va, sl2, c0, r, pf);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pp[16];
#pragma unroll
        for (int i2 = 0; i2 < 16; ++i2) pp[i2] = ptx::pack_bf16x2(pf[h][i2].x, pf[h][i2].y);
        ptx::tmem_st_32x32b_x16(st_cols + kColPT + c0 / 2 + 16 * h, pp);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      s.arrive(ctl->p_ready);
      // dS^T = P^T o (dP^T - delta_col), packed into the dP^T columns the same way.
      if (!(ok = s.wait(ctl->dp_full, par, kStatusTimeoutSoftmax))) break;
      ptx::tc_fence_after();
      ptx::tmem_ld_32x32b_x32(dpt_cols + c0, xr[0]);
      ptx::tmem_ld_32x32b_x32(dpt_cols + c0 + 32, xr[1]);
      ptx::tmem_wait_ld_regs(xr[0]);
      ptx::tmem_wait_ld_regs(xr[1]);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pd[16];
#pragma unroll
        for (int i2 = 0; i2 < 16; ++i2) {
          const float2 d = *reinterpret_cast<const float2*>(vd + 32 * h + 2 * i2);
          const float2 v = ptx::fmul2(pf[h][i2],
                                      ptx::fsub2(make_float2(__uint_as_float(xr[h][2 * i2]),
                                                             __uint_as_float(xr[h][2 * i2 + 1])), d));
          pd[i2] = ptx::pack_bf16x2(v.x, v.y);
        }
        ptx::tmem_st_32x32b_x16(dpt_cols + kColPT + c0 / 2 + 16 * h, pd);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      s.arrive(ctl->ds_ready);
      if (i + 1 < nq) {
        // the other buffer was last read at tile i-1, whose dS^T the MMA warp has consumed
        vec[(par ^ 1) * kBlockM + r] = stage(i + 1, nv);
        s.arrive(ctl->vec_sync);
      }
    }
    const bool row_ok = krow < p.sk;
    const size_t gk = row_offset<kBshd>(p, bh, krow, p.sk);
    if (nq == 0) {
      // keys no query attends (causal, Sk > Sq): zero gradients (dK by warpgroup 0, dV by 1)
      if (row_ok) zero_row(static_cast<uint8_t*>(g == 0 ? p.out0 : p.out1) + gk);
    } else if (ok && s.wait(ctl->acc_full, 0, kStatusTimeoutSoftmax)) {
      // Every product is done, so the Q/dO ring is free: dK (ring slot 0) and dV (slot 1) are
      // staged there as BF16 in the TMA layout (two 64-column slabs, 128-byte swizzle; warpgroup
      // g fills slab g) and stored with four tensor copies (rows past Sk are clipped by the
      // tensor maps).
      ptx::tc_fence_after();
      const uint32_t swz = static_cast<uint32_t>(r) & 7u;
#pragma unroll 2
      for (int c = 4 * g; c < 4 * g + 4; ++c) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          uint32_t acc[16];
          ptx::tmem_ld_32x32b_x16(kTmemBase + lane_off + (t ? kColDV : kColDK) + 16 * c, acc);
          ptx::tmem_wait_ld();
          const float mul = t ? 1.0f : p.scale;
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            pk[i] = ptx::pack_bf16x2(__uint_as_float(acc[2 * i]) * mul,
                                     __uint_as_float(acc[2 * i + 1]) * mul);
          const uint32_t line = L.ring(t) + (c >> 2) * kSlabBytes + static_cast<uint32_t>(r) * 128u;
          const uint32_t u = 2u * (c & 3);
          ptx::st_shared_v4(line + ((u ^ swz) << 4), pk[0], pk[1], pk[2], pk[3]);
          ptx::st_shared_v4(line + (((u + 1u) ^ swz) << 4), pk[4], pk[5], pk[6], pk[7]);
        }
      }
      ptx::fence_proxy_async_smem();
      s.arrive(ctl->epi_full);
      if (warp == 0) {
        const bool staged = s.wait(ctl->epi_full, 0, kStatusTimeoutSoftmax);
        if (staged && s.lane == 0) {
          const int row0 = kt * kBlockN;
          for (int t = 0; t < 2; ++t) {
            const CUtensorMap* tm = t ? &tm_dv : &tm_dk;
            for (int sl = 0; sl < 2; ++sl) {
              const uint32_t src = L.ring(t) + sl * kSlabBytes;
              if (L.heads4d) {
                const int b = bh / L.heads4d, h = bh - b * L.heads4d;
                ptx::tma_store_4d(tm, src, 64 * sl, h, row0, b);
              } else {
                ptx::tma_store_3d(tm, src, 64 * sl, row0, bh);
              }
            }
          }
          ptx::bulk_commit_group();
          ptx::bulk_wait_all();
        }
        __syncwarp();
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_alloc_base, kTmemCols);
  }
}

}  // namespace bwd
}  // namespace attn
