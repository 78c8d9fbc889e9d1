// attn_fwd.cu -- host side of the C ABI declared in include/attn_fwd.h:
// argument checks, TMA tensor-map encoding, persistent-grid sizing, launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <chrono>
#include <mutex>
#include <random>

#include "../../include/attn_fwd.h"
#include "attn_fwd_kernel.cuh"
#include "attn_bwd_kernel.cuh"
#include "attn_host.cuh"

namespace {

struct DeviceInfo {
  bool ready = false;
  int cc_major = 0, cc_minor = 0;
  int num_sms = 0;
  int smem_optin = 0;
  bool attr_set = false;
  bool bwd_attr_set = false;
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int device_info(int dev, DeviceInfo* out) {
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    d.ready = true;
  }
  if (d.cc_major != 10 || d.cc_minor != 3) return ATTN_ERR_ARCH;
  if (d.smem_optin < static_cast<int>(attn::kSmemBytes)) return ATTN_ERR_ARCH;
  // The kernels that split registers between warpgroups (setmaxnreg) need the block to be
  // launched with exactly the per-thread count the split adds up to: with fewer, an increase
  // could never be granted.  The compiled counts are checked once per device.
  auto regs_are = [](const void* fn, int want) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return false;
    return fa.numRegs == want;
  };
  if (!d.attr_set) {
    const void* fwd_kernels[] = {
        reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, false, false, attn::kModeCausal>),
        reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, false, false, attn::kModeGeneral>),
        reinterpret_cast<const void*>(attn::attn_fwd_kernel<true, false, false, attn::kModeGeneral>),
        reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, true, false, attn::kModeFull>),
        reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, true, false, attn::kModeGeneral>),
        reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, false, true, attn::kModeCausal>),
        reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, false, true, attn::kModeGeneral>),
        reinterpret_cast<const void*>(attn::attn_fwd_kernel<true, false, true, attn::kModeGeneral>),
        reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, true, true, attn::kModeFull>),
        reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, true, true, attn::kModeGeneral>)};
    for (const void* fn : fwd_kernels) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(attn::kSmemBytes)) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
      }
      if (!regs_are(fn, 65536 / attn::kThreads)) {
        cudaGetLastError();
        return ATTN_ERR_UNSUPPORTED;
      }
    }
    d.attr_set = true;
  }
  if (!d.bwd_attr_set) {
    const void* dq_kernels[] = {
        reinterpret_cast<const void*>(attn::bwd::attn_bwd_dq_kernel<true, false>),
        reinterpret_cast<const void*>(attn::bwd::attn_bwd_dq_kernel<false, false>),
        reinterpret_cast<const void*>(attn::bwd::attn_bwd_dq_kernel<true, true>),
        reinterpret_cast<const void*>(attn::bwd::attn_bwd_dq_kernel<false, true>)};
    const void* dkdv_kernels[] = {
        reinterpret_cast<const void*>(attn::bwd::attn_bwd_dkdv_kernel<true, false>),
        reinterpret_cast<const void*>(attn::bwd::attn_bwd_dkdv_kernel<false, false>),
        reinterpret_cast<const void*>(attn::bwd::attn_bwd_dkdv_kernel<true, true>),
        reinterpret_cast<const void*>(attn::bwd::attn_bwd_dkdv_kernel<false, true>)};
    for (const void* fn : dq_kernels) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(attn::bwd::kSmemBytesDq)) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
      }
      if (!regs_are(fn, static_cast<int>(attn::bwd::kDqRegLaunch))) {
        cudaGetLastError();
        return ATTN_ERR_UNSUPPORTED;
      }
    }
    for (const void* fn : dkdv_kernels) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(attn::bwd::kSmemBytesDkdv)) != cudaSuccess) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
      }
    }
    d.bwd_attr_set = true;
  }
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = d;
  return ATTN_OK;
}

// A BF16 [B,H,S,128] tensor as the 3-D TMA tensor (128, S, B*H), or a [B,S,H,128] tensor as the
// 4-D tensor (128, H, S, B).  Box: 64 columns x 128 sequence rows of one head, 128-byte swizzle,
// L2 promotion 256 B.  Rows past the sequence end of a head read as zeros.
int encode_qkv(CUtensorMap* map, const void* base, int64_t B, int64_t H, int64_t S, bool bshd) {
  const cuuint64_t D = attn::kHeadDim, e = 2;
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4];
  cuuint32_t rank;
  if (bshd) {
    rank = 4;
    dims[0] = D; dims[1] = H; dims[2] = S; dims[3] = B;
    strides[0] = D * e; strides[1] = H * D * e; strides[2] = S * H * D * e;
    box[0] = 64; box[1] = 1; box[2] = 128; box[3] = 1;
  } else {
    rank = 3;
    dims[0] = D; dims[1] = S; dims[2] = B * H;
    strides[0] = D * e; strides[1] = S * D * e;
    box[0] = 64; box[1] = 128; box[2] = 1;
  }
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na && nb && x < y + nb && y < x + na;
}

// Shape checks shared by attn_fwd and attn_fwd_plan.
int check_shape(int B, int H, int Sq, int Sk, int D) {
  if (B < 0 || H < 0 || Sq < 0 || Sk < 0 || D <= 0) return ATTN_ERR_INVALID_ARG;
  if (D != attn::kHeadDim) return ATTN_ERR_UNSUPPORTED;
  const int64_t bh = static_cast<int64_t>(B) * H;
  if (bh == 0 || Sq == 0) return ATTN_OK;   // empty problem
  if (Sk == 0) return ATTN_ERR_INVALID_ARG;
  const int64_t items = bh * ((ceil_div(Sq, attn::kBlockM) + 1) / 2);
  if (bh > INT32_MAX || items > INT32_MAX) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// The split schedule of attn_fwd_ws for a problem of `items` work items of `kv_tiles` KV tiles
// each on `grid` persistent CTAs.  Whole rounds run as before; when the last round would be
// partly idle, the last two rounds' items (between grid and 2*grid of them) are instead cut by
// KV range so every CTA gets the same number of (item, KV tile) units.  Used only where that
// shortens the longest CTA by at least kSplitMinGainTiles KV tiles.  Every extra segment of a CTA
// costs ~2 us of pipeline fill and drain, the combining epilogue ~3 us, and with all CTAs given
// equal work the slowest SM sets the end.  Measured on GB300 (split against whole items, same box,
// with the split instantiation's lean MMA loop): S=8K at 16 heads (16 tiles shorter) +2.9%, S=16K
// at 16 heads (33 tiles) +3.2%, S=12K at 24 heads (40) +2.8%; S=4K at 16 heads (8 tiles) 0.0%,
// and +0.9% once whole items' epilogue moved to the correction warpgroup ([B,S,H,D]: +1.7%).
// Dense, non-causal, exp2 on MUFU only.
struct SplitPlan {
  bool on = false;
  int sk_item0 = 0, sk_items = 0;
  size_t off_flag = 0, off_l = 0, off_o = 0, bytes = 0;
};

SplitPlan split_plan(int64_t items, int grid, int kv_tiles, int flags) {
  SplitPlan sp;
  if (flags & (ATTN_FLAG_CAUSAL | ATTN_FLAG_SOFT_EXP2 | ATTN_FLAG_TEST_WITHHOLD)) return sp;
  if (grid < 2 || items <= grid || items % grid == 0 || kv_tiles < 2) return sp;
  const int64_t sk_item0 = (items / grid - 1) * grid;
  const int64_t sk_items = items - sk_item0;   // in (grid, 2 grid)
  const int64_t units = sk_items * kv_tiles;
  if (units * grid > INT32_MAX) return sp;   // the kernel's unit arithmetic is 32-bit
  const int64_t longest = (units + grid - 1) / grid;
  constexpr int64_t kSplitMinGainTiles = 8;
  if (2 * static_cast<int64_t>(kv_tiles) - longest < kSplitMinGainTiles) return sp;
  sp.on = true;
  sp.sk_item0 = static_cast<int>(sk_item0);
  sp.sk_items = static_cast<int>(sk_items);
  const size_t slots = static_cast<size_t>(grid - 1);
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  sp.off_flag = 0;
  sp.off_l = up(slots * 2 * 4 * sizeof(unsigned long long));
  sp.off_o = sp.off_l + up(slots * 2 * 2 * attn::kBlockM * sizeof(float));
  sp.bytes = sp.off_o + slots * 2 * 2 * attn::kBlockM * attn::kHeadDim * sizeof(float);
  return sp;
}

// Per-call sequence numbers for the split schedule's flags: a random 32-bit salt per process in
// the high half, so numbers left in a workspace by another process or an earlier call differ.
unsigned long long next_seq() {
  static std::atomic<unsigned long long> counter{0};
  static const unsigned long long salt = [] {
    unsigned long long r;
    try {
      std::random_device rd;
      r = rd();
    } catch (...) {   // no entropy source: the clock and this object's address instead
      r = static_cast<unsigned long long>(
              std::chrono::high_resolution_clock::now().time_since_epoch().count()) ^
          reinterpret_cast<uintptr_t>(&counter);
    }
    return ((r & 0xffffffffull) | 1ull) << 32;
  }();
  return salt + counter.fetch_add(1, std::memory_order_relaxed);
}

int launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int Sq, int Sk, int D, float scale, int flags, void* workspace,
               size_t workspace_bytes, bool use_ws, void* stream);

}  // namespace

extern "C" {

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported shape or parameter";
    case ATTN_ERR_ARCH: return "device is not a compute capability 10.3 (GB300) GPU";
    case ATTN_ERR_CUDA: return "CUDA runtime or driver call failed";
    case ATTN_ERR_TOO_LARGE:
      return "problem exceeds the fixed scratch of the allocation-free entry point";
    default: return "unknown status";
  }
}

int attn_fwd_plan(int B, int H, int Sq, int Sk, int D, int flags, int num_sms, attn_plan* plan) {
  if (plan == nullptr) return ATTN_ERR_INVALID_ARG;
  if (flags & ~ATTN_FLAGS_ALL) return ATTN_ERR_INVALID_ARG;
  const int rc = check_shape(B, H, Sq, Sk, D);
  if (rc != ATTN_OK) return rc;
  if (num_sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
  }
  std::memset(plan, 0, sizeof(*plan));
  const int64_t bh = static_cast<int64_t>(B) * H;
  plan->q_tiles = ceil_div(Sq, attn::kBlockM);
  plan->kv_tiles = ceil_div(Sk, attn::kBlockN);
  plan->work_items = (Sq == 0) ? 0 : bh * ((plan->q_tiles + 1) / 2);
  plan->grid = static_cast<int>(plan->work_items < num_sms ? plan->work_items : num_sms);
  plan->threads = attn::kThreads;
  plan->kv_stages = attn::kKvStages;
  plan->smem_bytes = static_cast<int>(attn::kSmemBytes);
  plan->tmem_cols = static_cast<int>(attn::kTmemCols);
  return ATTN_OK;
}

int attn_fwd_work_item(int64_t item, int B, int H, int Sq, int Sk, int flags, int* bh,
                       int* q_tile0, int* kv_tiles0, int* kv_tiles1) {
  if (bh == nullptr || q_tile0 == nullptr || kv_tiles0 == nullptr || kv_tiles1 == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (flags & ~ATTN_FLAGS_ALL) return ATTN_ERR_INVALID_ARG;
  const int rc = check_shape(B, H, Sq, Sk, attn::kHeadDim);
  if (rc != ATTN_OK) return rc;
  const int q_tiles = ceil_div(Sq, attn::kBlockM);
  const int pairs = (q_tiles + 1) / 2;
  const int64_t items = static_cast<int64_t>(B) * H * pairs;
  if (item < 0 || item >= items) return ATTN_ERR_INVALID_ARG;
  const attn::WorkItem w =
      attn::decode_item(static_cast<int>(item), pairs, q_tiles, ceil_div(Sk, attn::kBlockN),
                        B * H, (flags & ATTN_FLAG_CAUSAL) != 0);
  *bh = w.bh;
  *q_tile0 = w.qt0;
  *kv_tiles0 = w.n[0];
  *kv_tiles1 = w.n[1];
  return ATTN_OK;
}

int attn_fwd_schedule(int cta, int round, int grid, int64_t work_items, int flags) {
  if (cta < 0 || round < 0 || grid <= 0 || cta >= grid || work_items < 0 || work_items > INT32_MAX)
    return -1;
  return attn::item_of(round, cta, grid, static_cast<int>(work_items),
                       (flags & ATTN_FLAG_CAUSAL) != 0);
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int Sq, int Sk, int D, float scale, void* stream) {
  return attn_fwd_ex(q, k, v, o, lse, B, H, Sq, Sk, D, scale, 0, stream);
}

int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Sq, int Sk, int D, float scale, int flags, void* stream) {
  return launch_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, scale, flags, nullptr, 0, false, stream);
}

int attn_fwd_workspace(int B, int H, int Sq, int Sk, int D, int flags, size_t* bytes) {
  if (bytes == nullptr) return ATTN_ERR_INVALID_ARG;
  if (flags & ~ATTN_FLAGS_ALL) return ATTN_ERR_INVALID_ARG;
  const int rc = check_shape(B, H, Sq, Sk, D);
  if (rc != ATTN_OK) return rc;
  *bytes = 0;
  const int64_t bh = static_cast<int64_t>(B) * H;
  if (bh == 0 || Sq == 0) return ATTN_OK;
  int dev = 0, num_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  const int64_t items = bh * ((ceil_div(Sq, attn::kBlockM) + 1) / 2);
  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  *bytes = split_plan(items, grid, ceil_div(Sk, attn::kBlockN), flags).bytes;
  return ATTN_OK;
}

int attn_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Sq, int Sk, int D, float scale, int flags, void* workspace,
                size_t workspace_bytes, void* stream) {
  return launch_fwd(q, k, v, o, lse, B, H, Sq, Sk, D, scale, flags, workspace, workspace_bytes,
                    true, stream);
}

int attn_fwd_segment(int cta, int round, int grid, int64_t work_items, int kv_tiles, int flags,
                     int* item, int* kv_tile0, int* kv_count, int* slot, int* part) {
  if (!item || !kv_tile0 || !kv_count || !slot || !part) return ATTN_ERR_INVALID_ARG;
  if (cta < 0 || round < 0 || grid <= 0 || cta >= grid || work_items < 0 ||
      work_items > INT32_MAX || kv_tiles <= 0 || (flags & ~ATTN_FLAGS_ALL))
    return ATTN_ERR_INVALID_ARG;
  const SplitPlan sp = split_plan(work_items, grid, kv_tiles, flags);
  *slot = -1;
  *part = 0;
  if (!sp.on || static_cast<int64_t>(round) * grid < sp.sk_item0) {
    const int it = attn::item_of(round, cta, grid, static_cast<int>(work_items),
                                 (flags & ATTN_FLAG_CAUSAL) != 0);
    if (it < 0) return 0;
    *item = it;
    *kv_tile0 = 0;
    *kv_count = -1;   // the whole item (its KV tiles per Q tile: attn_fwd_work_item)
    return 1;
  }
  int il, j0, cnt;
  if (!attn::split_segment(round - sp.sk_item0 / grid, cta, grid, sp.sk_items, kv_tiles, il, j0,
                           cnt))
    return 0;
  *item = sp.sk_item0 + il;
  *kv_tile0 = j0;
  *kv_count = cnt;
  if (cnt < kv_tiles) {
    *part = j0 > 0 ? 1 : 0;
    *slot = j0 > 0 ? cta - 1 : cta;
  }
  return 1;
}

}  // extern "C"

namespace {

int launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int Sq, int Sk, int D, float scale, int flags, void* workspace,
               size_t workspace_bytes, bool use_ws, void* stream) {
  if (flags & ~ATTN_FLAGS_ALL) return ATTN_ERR_INVALID_ARG;
  int rc = check_shape(B, H, Sq, Sk, D);
  if (rc != ATTN_OK) return rc;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (scale < 0.f) return ATTN_ERR_UNSUPPORTED;
  const int64_t bh = static_cast<int64_t>(B) * H;
  if (bh == 0 || Sq == 0) return ATTN_OK;
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  auto mis16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (mis16(q) || mis16(k) || mis16(v) || mis16(o)) return ATTN_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  const size_t nq = static_cast<size_t>(bh) * Sq * D * 2, nk = static_cast<size_t>(bh) * Sk * D * 2;
  const size_t nl = lse ? static_cast<size_t>(bh) * Sq * 4 : 0;
  if (overlaps(o, nq, q, nq) || overlaps(o, nq, k, nk) || overlaps(o, nq, v, nk) ||
      overlaps(lse, nl, q, nq) || overlaps(lse, nl, k, nk) || overlaps(lse, nl, v, nk) ||
      overlaps(lse, nl, o, nq))
    return ATTN_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  DeviceInfo info;
  rc = device_info(dev, &info);
  if (rc != ATTN_OK) return rc;

  alignas(64) CUtensorMap tm_q, tm_k, tm_v;
  const bool bshd = (flags & ATTN_FLAG_BSHD) != 0;
  if (encode_qkv(&tm_q, q, B, H, Sq, bshd) != ATTN_OK ||
      encode_qkv(&tm_k, k, B, H, Sk, bshd) != ATTN_OK ||
      encode_qkv(&tm_v, v, B, H, Sk, bshd) != ATTN_OK)
    return ATTN_ERR_CUDA;

  attn::Params p;
  p.o = o;
  p.lse = lse;
  p.sq = Sq;
  p.heads = H;
  p.bshd = bshd ? 1 : 0;
  const int64_t Dl = attn::kHeadDim;
  p.o_row_stride = bshd ? H * Dl : Dl;
  p.o_head_stride = bshd ? Dl : static_cast<int64_t>(Sq) * Dl;
  p.o_batch_stride = static_cast<int64_t>(H) * Sq * Dl;
  p.q_tiles = ceil_div(Sq, attn::kBlockM);
  p.kv_tiles = ceil_div(Sk, attn::kBlockN);
  p.kv_valid_last = Sk - (p.kv_tiles - 1) * attn::kBlockN;
  p.pairs_per_head = (p.q_tiles + 1) / 2;
  p.num_items = static_cast<int>(bh * p.pairs_per_head);
  p.bh = static_cast<int>(bh);
  p.causal = (flags & ATTN_FLAG_CAUSAL) ? 1 : 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  p.test_withhold = (flags & ATTN_FLAG_TEST_WITHHOLD) ? 1 : 0;
  p.o_align32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0 ? 1 : 0;
  const int grid = p.num_items < info.num_sms ? p.num_items : info.num_sms;
  p.sk_item0 = p.num_items;
  p.sk_items = 0;
  p.ws_o = p.ws_l = nullptr;
  p.ws_flag = nullptr;
  p.seq = 0;
  const SplitPlan sp = use_ws ? split_plan(p.num_items, grid, p.kv_tiles, flags) : SplitPlan();
  if (sp.on) {
    if (workspace == nullptr || workspace_bytes < sp.bytes ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
      return ATTN_ERR_INVALID_ARG;
    const size_t nw = sp.bytes;
    if (overlaps(workspace, nw, q, nq) || overlaps(workspace, nw, k, nk) ||
        overlaps(workspace, nw, v, nk) || overlaps(workspace, nw, o, nq) ||
        overlaps(workspace, nw, lse, nl))
      return ATTN_ERR_INVALID_ARG;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.sk_item0 = sp.sk_item0;
    p.sk_items = sp.sk_items;
    p.ws_flag = reinterpret_cast<unsigned long long*>(ws + sp.off_flag);
    p.ws_l = reinterpret_cast<float*>(ws + sp.off_l);
    p.ws_o = reinterpret_cast<float*>(ws + sp.off_o);
    p.seq = next_seq();
  }

  // Instantiations: <software exp2, split schedule, [B,S,H,D], mode>.  The software exp2 is built
  // in the general mode only and never with the split schedule, the causal mode never splits, and
  // the full-tile mode is built only with the split schedule: launches without split items run it
  // with an empty split part (sk_item0 = all items), which measured as fast as the whole-item
  // instantiation at S=4K and 0.8-1.2% faster at S=8K-16K (its MMA loop has no per-stage tests).
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const bool soft = (flags & ATTN_FLAG_SOFT_EXP2) != 0;
  const bool general = soft || p.kv_valid_last != attn::kBlockN || p.scale_log2 == 0.f ||
                       Sq % (2 * attn::kBlockM) != 0 || !p.o_align32 || p.test_withhold;
#define ATTN_LAUNCH(S, P, L, M) \
  attn::attn_fwd_kernel<S, P, L, M><<<grid, attn::kThreads, attn::kSmemBytes, cs>>>(tm_q, tm_k, tm_v, p)
  if (bshd) {
    if (soft) ATTN_LAUNCH(true, false, true, attn::kModeGeneral);
    else if (sp.on && general) ATTN_LAUNCH(false, true, true, attn::kModeGeneral);
    else if (general) ATTN_LAUNCH(false, false, true, attn::kModeGeneral);
    else if (p.causal) ATTN_LAUNCH(false, false, true, attn::kModeCausal);
    else ATTN_LAUNCH(false, true, true, attn::kModeFull);
  } else {
    if (soft) ATTN_LAUNCH(true, false, false, attn::kModeGeneral);
    else if (sp.on && general) ATTN_LAUNCH(false, true, false, attn::kModeGeneral);
    else if (general) ATTN_LAUNCH(false, false, false, attn::kModeGeneral);
    else if (p.causal) ATTN_LAUNCH(false, false, false, attn::kModeCausal);
    else ATTN_LAUNCH(false, true, false, attn::kModeFull);
  }
#undef ATTN_LAUNCH
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_device_status(unsigned int* word, int clear) {
  if (word == nullptr) return ATTN_ERR_INVALID_ARG;
  if (cudaMemcpyFromSymbol(word, attn::g_attn_status, sizeof(unsigned int)) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(attn::g_attn_status, &zero, sizeof(unsigned int)) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
  }
  return ATTN_OK;
}

// ------------------------------------------------------------------ host-buffer forward
namespace {
attn::host::Pipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu;

int host_shape(int B, int H, int Sq, int Sk, int D, int flags) {
  if (flags & ~ATTN_FLAGS_ALL) return ATTN_ERR_INVALID_ARG;
  return check_shape(B, H, Sq, Sk, D);
}

// Lazily create the two copy streams and the events of this device (under g_pipe_mu).
int pipe_for(int dev, attn::host::Pipe** out) {
  attn::host::Pipe& P = g_pipe[dev];
  if (!P.ready) {
    bool ok = cudaStreamCreateWithFlags(&P.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&P.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&P.start, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < attn::host::kMaxChunks; ++i)
      ok = cudaEventCreateWithFlags(&P.ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&P.ev_k[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&P.ev_out[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    P.ready = true;
  }
  *out = &P;
  return ATTN_OK;
}
}  // namespace

int attn_fwd_host_workspace(int B, int H, int Sq, int Sk, int D, int flags, size_t* bytes) {
  if (bytes == nullptr) return ATTN_ERR_INVALID_ARG;
  const int rc = host_shape(B, H, Sq, Sk, D, flags);
  if (rc != ATTN_OK) return rc;
  *bytes = attn::host::layout(static_cast<int64_t>(B) * H, Sq, Sk, D).total;
  return ATTN_OK;
}

int attn_fwd_host_chunking(int B, int H, int Sq, int Sk, int flags, int num_sms,
                           int64_t* units_per_chunk, int64_t* chunks) {
  if (units_per_chunk == nullptr || chunks == nullptr || num_sms <= 0) return ATTN_ERR_INVALID_ARG;
  const int rc = host_shape(B, H, Sq, Sk, attn::kHeadDim, flags);
  if (rc != ATTN_OK) return rc;
  const bool bshd = (flags & ATTN_FLAG_BSHD) != 0;
  const int64_t pairs = (ceil_div(Sq, attn::kBlockM) + 1) / 2;
  const int64_t units = bshd ? B : static_cast<int64_t>(B) * H;
  const int64_t per_unit = bshd ? static_cast<int64_t>(H) * pairs : pairs;
  const int64_t items = units * per_unit;
  const int64_t grid = items < num_sms ? items : num_sms;
  if (units == 0) {
    *units_per_chunk = *chunks = 0;
    return ATTN_OK;
  }
  *units_per_chunk = attn::host::host_chunk_units(units, per_unit, grid, attn::host::kMaxChunks);
  *chunks = (units + *units_per_chunk - 1) / *units_per_chunk;
  return ATTN_OK;
}

int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                  int Sq, int Sk, int D, float scale, int flags, void* workspace,
                  size_t workspace_bytes, void* stream) {
  int rc = host_shape(B, H, Sq, Sk, D, flags);
  if (rc != ATTN_OK) return rc;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (scale < 0.f) return ATTN_ERR_UNSUPPORTED;
  const int64_t bh = static_cast<int64_t>(B) * H;
  if (bh == 0 || Sq == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !workspace) return ATTN_ERR_INVALID_ARG;
  const attn::host::Layout L = attn::host::layout(bh, Sq, Sk, D);
  if (workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return ATTN_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  DeviceInfo info;
  rc = device_info(dev, &info);
  if (rc != ATTN_OK) return rc;
  int64_t per_chunk = 0, nchunks = 0;
  rc = attn_fwd_host_chunking(B, H, Sq, Sk, flags, info.num_sms, &per_chunk, &nchunks);
  if (rc != ATTN_OK) return rc;

  const bool bshd = (flags & ATTN_FLAG_BSHD) != 0;
  // bytes of one unit (a head, or a batch entry) of each tensor
  const size_t uq = static_cast<size_t>(Sq) * D * 2 * (bshd ? H : 1);
  const size_t uk = static_cast<size_t>(Sk) * D * 2 * (bshd ? H : 1);
  const size_t ul = static_cast<size_t>(Sq) * 4 * (bshd ? H : 1);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);

  std::lock_guard<std::mutex> lk(g_pipe_mu);
  attn::host::Pipe* P = nullptr;
  rc = pipe_for(dev, &P);
  if (rc != ATTN_OK) return rc;
  auto fail = [] {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  };
  // The copies start after everything already queued on the caller's stream (which may still
  // read the workspace, or write these host buffers).
  if (cudaEventRecord(P->start, cs) != cudaSuccess ||
      cudaStreamWaitEvent(P->in, P->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(P->out, P->start, 0) != cudaSuccess)
    return fail();
  const int64_t units = bshd ? B : bh;
  for (int64_t c = 0, u0 = 0; c < nchunks; ++c) {
    const int64_t nu = units - u0 < per_chunk ? units - u0 : per_chunk;
    uint8_t* dq = ws + L.q + u0 * uq;
    uint8_t* dk = ws + L.k + u0 * uk;
    uint8_t* dv = ws + L.v + u0 * uk;
    uint8_t* dO = ws + L.o + u0 * uq;
    float* dl = lse ? reinterpret_cast<float*>(ws + L.lse + u0 * ul) : nullptr;
    const uint8_t* hq = static_cast<const uint8_t*>(q) + u0 * uq;
    const uint8_t* hk = static_cast<const uint8_t*>(k) + u0 * uk;
    const uint8_t* hv = static_cast<const uint8_t*>(v) + u0 * uk;
    if (cudaMemcpyAsync(dq, hq, nu * uq, cudaMemcpyHostToDevice, P->in) != cudaSuccess ||
        cudaMemcpyAsync(dk, hk, nu * uk, cudaMemcpyHostToDevice, P->in) != cudaSuccess ||
        cudaMemcpyAsync(dv, hv, nu * uk, cudaMemcpyHostToDevice, P->in) != cudaSuccess ||
        cudaEventRecord(P->ev_in[c], P->in) != cudaSuccess ||
        cudaStreamWaitEvent(cs, P->ev_in[c], 0) != cudaSuccess)
      return fail();
    const int sub_b = bshd ? static_cast<int>(nu) : 1;
    const int sub_h = bshd ? H : static_cast<int>(nu);
    rc = attn_fwd_ex(dq, dk, dv, dO, dl, sub_b, sub_h, Sq, Sk, D, scale, flags, stream);
    if (rc != ATTN_OK) return rc;
    if (cudaEventRecord(P->ev_k[c], cs) != cudaSuccess ||
        cudaStreamWaitEvent(P->out, P->ev_k[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<uint8_t*>(o) + u0 * uq, dO, nu * uq, cudaMemcpyDeviceToHost,
                        P->out) != cudaSuccess)
      return fail();
    if (lse && cudaMemcpyAsync(reinterpret_cast<uint8_t*>(lse) + u0 * ul, dl, nu * ul,
                               cudaMemcpyDeviceToHost, P->out) != cudaSuccess)
      return fail();
    if (cudaEventRecord(P->ev_out[c], P->out) != cudaSuccess) return fail();
    u0 += nu;
  }
  // The caller's stream completes only after the last copy back (the out stream is in order).
  if (cudaStreamWaitEvent(cs, P->ev_out[nchunks - 1], 0) != cudaSuccess) return fail();
  return ATTN_OK;
}

}  // extern "C"

// The backward's two gradient kernels are independent once delta is written; the dQ kernel runs
// on a side stream of the library so its CTAs can take the SMs that the dK/dV kernel's last,
// partly filled wave leaves idle (and the other way round), instead of each kernel ending on its
// own partial wave.  One side stream and a fork/join event pair per device, created on first use.
namespace {
struct BwdFork {
  bool ready = false;
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
BwdFork g_bwd_fork[kMaxDevices];
std::mutex g_bwd_mu;
}  // namespace

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv,
                        float* delta, int B, int H, int Sq, int Sk, int D, float scale, int flags,
                        void* stream) {
  if (flags & ~(ATTN_FLAG_CAUSAL | ATTN_FLAG_BSHD)) return ATTN_ERR_INVALID_ARG;
  int rc = check_shape(B, H, Sq, Sk, D);
  if (rc != ATTN_OK) return rc;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (scale < 0.f) return ATTN_ERR_UNSUPPORTED;
  const int64_t bh = static_cast<int64_t>(B) * H;
  if (bh == 0) return ATTN_OK;
  if (Sq == 0) {
    if (Sk == 0) return ATTN_OK;
    // no queries: every key and value gradient is zero
    if (!dk || !dv) return ATTN_ERR_INVALID_ARG;
    const size_t nk = static_cast<size_t>(bh) * Sk * D * 2;
    if (cudaMemsetAsync(dk, 0, nk, static_cast<cudaStream_t>(stream)) != cudaSuccess ||
        cudaMemsetAsync(dv, 0, nk, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    return ATTN_OK;
  }
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !delta)
    return ATTN_ERR_INVALID_ARG;
  auto mis16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (mis16(q) || mis16(k) || mis16(v) || mis16(o) || mis16(dout) || mis16(dq) || mis16(dk) ||
      mis16(dv))
    return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(delta) & 3u))
    return ATTN_ERR_INVALID_ARG;
  const size_t nq = static_cast<size_t>(bh) * Sq * D * 2, nk = static_cast<size_t>(bh) * Sk * D * 2;
  const size_t nl = static_cast<size_t>(bh) * Sq * 4;
  const void* ins[6] = {q, k, v, o, dout, lse};
  const size_t in_n[6] = {nq, nk, nk, nq, nq, nl};
  void* outs[4] = {dq, dk, dv, delta};
  const size_t out_n[4] = {nq, nk, nk, nl};
  for (int a = 0; a < 4; ++a) {
    for (int b = 0; b < 6; ++b)
      if (overlaps(outs[a], out_n[a], ins[b], in_n[b])) return ATTN_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (overlaps(outs[a], out_n[a], outs[b], out_n[b])) return ATTN_ERR_INVALID_ARG;
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  DeviceInfo info;
  rc = device_info(dev, &info);
  if (rc != ATTN_OK) return rc;

  const bool bshd = (flags & ATTN_FLAG_BSHD) != 0;
  alignas(64) CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_dk, tm_dv;
  if (encode_qkv(&tm_q, q, B, H, Sq, bshd) != ATTN_OK ||
      encode_qkv(&tm_k, k, B, H, Sk, bshd) != ATTN_OK ||
      encode_qkv(&tm_v, v, B, H, Sk, bshd) != ATTN_OK ||
      encode_qkv(&tm_do, dout, B, H, Sq, bshd) != ATTN_OK ||
      encode_qkv(&tm_dk, dk, B, H, Sk, bshd) != ATTN_OK ||
      encode_qkv(&tm_dv, dv, B, H, Sk, bshd) != ATTN_OK)
    return ATTN_ERR_CUDA;

  attn::bwd::Params p;
  p.lse = lse;
  p.delta = delta;
  p.sq = Sq;
  p.sk = Sk;
  p.q_tiles = ceil_div(Sq, attn::kBlockM);
  p.kv_tiles = ceil_div(Sk, attn::kBlockN);
  p.q_valid_last = Sq - (p.q_tiles - 1) * attn::kBlockM;
  p.kv_valid_last = Sk - (p.kv_tiles - 1) * attn::kBlockN;
  p.bh = static_cast<int>(bh);
  p.heads = H;
  p.bshd = bshd ? 1 : 0;
  p.causal = (flags & ATTN_FLAG_CAUSAL) ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);

  const int64_t rows = bh * Sq;
  attn::bwd::attn_bwd_delta_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
      static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), delta, rows, H, Sq,
      p.bshd);
  std::lock_guard<std::mutex> lk(g_bwd_mu);
  BwdFork& F = g_bwd_fork[dev];
  if (!F.ready) {
    if (cudaStreamCreateWithFlags(&F.side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&F.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&F.join, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_CUDA;
    }
    F.ready = true;
  }
  // dQ waits for delta (and for everything queued on the caller's stream before it); the
  // caller's stream waits for dQ before anything it runs next.
  if (cudaEventRecord(F.fork, st) != cudaSuccess || cudaStreamWaitEvent(F.side, F.fork, 0) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  p.out0 = dk;
  p.out1 = dv;
  // The masking code is compiled only into the instantiations for launches that need it (the
  // causal mask; for the dQ kernel also a ragged last K/V tile), the layout into each one's own.
  const bool mask_dq = p.causal != 0 || p.kv_valid_last != attn::kBlockN;
  const unsigned dkdv_grid = static_cast<unsigned>(bh * p.kv_tiles);
  const unsigned dq_grid = static_cast<unsigned>(bh * ((p.q_tiles + 1) / 2));
#define ATTN_DKDV(M, L)                                                                      \
  attn::bwd::attn_bwd_dkdv_kernel<M, L><<<dkdv_grid, attn::bwd::kThreads,                   \
                                          attn::bwd::kSmemBytesDkdv, st>>>(tm_q, tm_k, tm_v, \
                                                                           tm_do, tm_dk, tm_dv, p)
#define ATTN_DQ(M, L)                                                                           \
  attn::bwd::attn_bwd_dq_kernel<M, L><<<dq_grid, attn::bwd::kDqThreads, attn::bwd::kSmemBytesDq, \
                                        F.side>>>(tm_q, tm_k, tm_v, tm_do, p)
  if (p.causal) {
    if (bshd) ATTN_DKDV(true, true); else ATTN_DKDV(true, false);
  } else {
    if (bshd) ATTN_DKDV(false, true); else ATTN_DKDV(false, false);
  }
  p.out0 = dq;
  p.out1 = nullptr;
  if (mask_dq) {
    if (bshd) ATTN_DQ(true, true); else ATTN_DQ(true, false);
  } else {
    if (bshd) ATTN_DQ(false, true); else ATTN_DQ(false, false);
  }
#undef ATTN_DKDV
#undef ATTN_DQ
  const bool launched = cudaGetLastError() == cudaSuccess;
  // Join even after a failed launch, so the caller's stream never runs ahead of a dQ in flight.
  if (cudaEventRecord(F.join, F.side) != cudaSuccess || cudaStreamWaitEvent(st, F.join, 0) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  return launched ? ATTN_OK : ATTN_ERR_CUDA;
}

// ------------------------------------------------------------------ allocation-free backward
// Scratch for attn_bwd_noalloc: the per-query-row delta of the backward lives in this fixed
// device array instead of a buffer the caller allocates.  Every GPU that loads the library holds
// it (4 MiB) until the process exits.  Host code must not use its name as a device address: the
// address is looked up once per device with cudaGetSymbolAddress.
namespace {

constexpr int64_t kNoAllocDeltaMax = int64_t(1) << 20;   // floats: B * H * Sq <= 1,048,576
static __device__ __align__(256) float g_noalloc_delta[kNoAllocDeltaMax];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

}  // namespace

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                int B, int H, int Sq, int Sk, int D, float scale, int flags,
                                void* stream) {
  if (B < 0 || H < 0 || Sq < 0) return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * H * Sq > kNoAllocDeltaMax) return ATTN_ERR_TOO_LARGE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  // The device checks first (architecture, kernel attributes), so a device this library does not
  // run on reports ATTN_ERR_ARCH as attn_bwd does, before the array's address is looked up.
  DeviceInfo info;
  const int rc = device_info(dev, &info);
  if (rc != ATTN_OK) return rc;
  float* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_delta) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return ATTN_ERR_CUDA;
      }
      g_noalloc_ptr[dev] = static_cast<float*>(ptr);
    }
    scratch = g_noalloc_ptr[dev];
  }
  // delta is written in full by the backward's first kernel before it is read, so the array's
  // leftover contents from an earlier call never matter.
  return attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch, B, H, Sq, Sk, D, scale, flags,
                  stream);
}
