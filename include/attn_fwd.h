/*
 * attn_fwd.h -- C ABI of the GB300 (sm_103a) dense attention forward.
 *
 * One operation: the dense, non-causal attention forward with head_dim 128,
 *     O   = softmax(scale * Q K^T) V
 *     LSE = log(sum_j exp(scale * q_i . k_j))        (natural log, per query row)
 * computed tile by tile with the online-softmax state (running row max, row
 * sum, unnormalised O) so the Sq x Sk score matrix never reaches memory.
 *
 * Where the operation is defined:
 *   "B200 Attention Kernel from Scratch to Near-SOTA in 60 Diagrams" -- scope
 *   (dense, head dim 128, non-causal, BF16), Chapter 1 section ii (Q, K, V and
 *   the output share the shape [B, num_heads, seq_len, head_dim]; 128x128
 *   tiles), Chapter 1 section B (the online-softmax update and the final
 *   division by the row sum), Chapter 8 (base-2 exponent with the scale folded
 *   in), Chapter 11 (the kept max is rebased only past a threshold), and the
 *   Appendix "Benchmark Calibration" (contiguous BHLD inputs).
 *   "Attention for sm90, Line by Line", the exp2 question: the residual LSE is
 *   stored in natural-log units.
 *
 * No function here allocates device memory, copies between host and device or
 * synchronises, unless its comment says so.  All entry points are thread-safe.
 */
#ifndef ATTN_FWD_H_
#define ATTN_FWD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = -1, /* null/misaligned pointer, negative size, aliasing, bad scale */
  ATTN_ERR_UNSUPPORTED = -2, /* valid request outside what this build supports (D != 128, ...) */
  ATTN_ERR_ARCH = -3,        /* the current device is not a compute capability 10.3 GPU */
  ATTN_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed (launch, tensor-map encode) */
  ATTN_ERR_TOO_LARGE = -5    /* beyond the fixed scratch size of attn_bwd_noalloc */
} attn_status;

/*
 * attn_fwd -- enqueue one attention forward on `stream`.
 *
 *   q    device, BF16, [B, H, Sq, D] contiguous (row-major, D fastest), read only
 *   k    device, BF16, [B, H, Sk, D] contiguous, read only
 *   v    device, BF16, [B, H, Sk, D] contiguous, read only
 *   o    device, BF16, [B, H, Sq, D] contiguous, written (every element)
 *   lse  device, fp32, [B, H, Sq] contiguous, written; may be NULL (not stored)
 *   B, H, Sq, Sk, D   sizes; supported: D == 128, any Sq >= 0 and Sk >= 1 (the last
 *                     128-row tile of a sequence may be partial)
 *   scale             multiplies Q K^T before the softmax; finite and >= 0
 *                     (the row max is taken on raw scores and then scaled)
 *   stream            a cudaStream_t (NULL = the legacy default stream)
 *
 * Ownership: the caller owns every buffer; the library keeps no pointer after
 * the call returns.  q, k, v, o and lse must be distinct, non-overlapping
 * device allocations of the current device; q, k, v, o 16-byte aligned, lse
 * 4-byte aligned.
 *
 * Errors: arguments are checked on the host before anything is enqueued; any
 * error returns without launching.  B*H == 0 or Sq == 0 is a valid empty
 * problem: ATTN_OK, nothing launched.  Sk == 0 with Sq > 0 is
 * ATTN_ERR_INVALID_ARG (a softmax over no keys).  D != 128 is
 * ATTN_ERR_UNSUPPORTED.  A device that is not compute capability 10.3 gives
 * ATTN_ERR_ARCH.  A failed launch gives ATTN_ERR_CUDA (the sticky-free launch
 * error is cleared).  Non-finite inputs give unspecified outputs.
 *
 * Asynchronous: returns once the kernel is enqueued.  Results are ready when
 * the stream reaches that point.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int Sq, int Sk, int D, float scale, void* stream);

/* Flags of attn_fwd_ex. */
#define ATTN_FLAG_CAUSAL 1 /* query i attends keys j <= i (top-left aligned, i and j from 0) */
#define ATTN_FLAG_BSHD 2   /* q, k, v, o are [B, S, H, D] contiguous (lse stays [B, H, Sq]) */
/* Test hook, attn_fwd_ex only: in CTA 0 the TMA warp never loads its first K tile, so the MMA
 * warp's bounded wait on it expires (2 s); the CTA then stops, records status bits (see
 * attn_device_status) and exits, leaving its outputs unspecified.  For testing the failure path;
 * other CTAs and later calls are unaffected. */
#define ATTN_FLAG_TEST_WITHHOLD 0x100
/* Forward only: 4 of every 16 P columns use a polynomial exp2 on the FMA and integer pipes
 * instead of the MUFU unit ("B200 Attention Kernel from Scratch to Near-SOTA in 60 Diagrams",
 * Chapter 9; relative error of that exp2 <= 1e-4).  Off by default: slower on GB300. */
#define ATTN_FLAG_SOFT_EXP2 4
#define ATTN_FLAGS_ALL \
  (ATTN_FLAG_CAUSAL | ATTN_FLAG_BSHD | ATTN_FLAG_SOFT_EXP2 | ATTN_FLAG_TEST_WITHHOLD)

/*
 * attn_fwd_ex -- attn_fwd with options.  Arguments, ownership, errors and
 * asynchrony as attn_fwd; flags is a bitwise OR of ATTN_FLAG_* (0 = attn_fwd),
 * other bits give ATTN_ERR_INVALID_ARG.
 *
 * ATTN_FLAG_BSHD: q is [B, Sq, H, D], k and v [B, Sk, H, D], o [B, Sq, H, D],
 * all contiguous (the layout FlashAttention-4 is timed on: "B200 Attention
 * Kernel from Scratch to Near-SOTA in 60 Diagrams", Appendix "Benchmark
 * Calibration", the direct-BSHD variant); no conversion copies are made.
 * lse stays [B, H, Sq].  Same alignment and overlap rules.
 *
 * ATTN_FLAG_CAUSAL: the causal mask, key j is used by query i only when
 * j <= i, i.e. the two sequences are aligned at their first positions; every
 * query keeps at least key 0.  "Attention for sm90, Line by Line" (the
 * persistent-flag question) names causal masking and the load imbalance it
 * brings to a persistent schedule; work items are then run heaviest first.
 */
int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Sq, int Sk, int D, float scale, int flags, void* stream);

/*
 * attn_fwd_ws -- attn_fwd_ex with a workspace that lets the persistent grid end
 * evenly.  Chapter 14 of "B200 Attention Kernel from Scratch to Near-SOTA in 60
 * Diagrams" runs work items (a head and a pair of 128-row Q tiles) by static
 * stride over one CTA per SM; when the item count is not a multiple of the grid,
 * the last round leaves SMs idle (S=4K/8K/16K at 16 heads: 1024 items on 152
 * SMs, 7 rounds for 6.74 rounds of work).  Here the items of the last two
 * rounds are cut by KV range so that every CTA processes the same number of
 * (item, 128-key tile) units; an item shared by two CTAs is finished from the
 * two parts' partial results, O_i / l_i and log2-sum-exp L_i, as
 * O = sum_i 2^(L_i - L) O_i / l_i with L = log2 sum_i 2^L_i -- the same
 * rescaling of partial softmax sums that the online recurrence (Chapter 1,
 * section B; Chapter 11) applies tile by tile.  Neither CTA waits for the
 * other: the one that finishes second combines, always in KV order, so results
 * are deterministic.  Output agrees with attn_fwd within rounding (the combined
 * items round O once more in fp32).
 *
 *   q..stream        as attn_fwd_ex
 *   workspace        device memory owned by the caller, 256-byte aligned, at
 *                    least attn_fwd_workspace() bytes (0 bytes: NULL is fine);
 *                    contents on entry are ignored and need no clearing.  Each
 *                    call tags its flags there with a number unique to the call
 *                    and clears every flag it completed, so a launch that reuses
 *                    the number (a replayed CUDA graph) finds them clear; after a
 *                    call that reported an expired wait (attn_device_status),
 *                    zero the workspace before replaying such a launch on it
 *   workspace_bytes  its size
 *
 * The split schedule is used for dense, non-causal calls without
 * ATTN_FLAG_SOFT_EXP2 where it shortens the longest CTA by at least 8
 * KV-tile iterations (each extra segment and the combine cost a few; on a
 * 152-SM GPU: S=4K, S=8K and S=16K at 16 heads and S=12K at 24 heads split,
 * S=2K at 16 heads does not); otherwise this is attn_fwd_ex and the workspace is not
 * touched.  A workspace must not be used by two calls that can run at the same time
 * (different streams): they would overwrite each other's partial results.
 * Errors as attn_fwd_ex, plus ATTN_ERR_INVALID_ARG for a missing, short,
 * misaligned or overlapping workspace when one is needed.
 */
int attn_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Sq, int Sk, int D, float scale, int flags, void* workspace,
                size_t workspace_bytes, void* stream);

/* Bytes of workspace attn_fwd_ws needs for this problem on the current device
 * (0 when it does not split; about 40 MB on a 152-SM GPU when it does). */
int attn_fwd_workspace(int B, int H, int Sq, int Sk, int D, int flags, size_t* bytes);

/* The schedule of attn_fwd_ws on the host, for tests: the segment a persistent
 * CTA runs in its round-th turn for `work_items` items of `kv_tiles` KV tiles on
 * `grid` CTAs.  Returns 1 and fills the outputs, 0 when the CTA has no more
 * segments, ATTN_ERR_INVALID_ARG on bad arguments.  *kv_count == -1: the whole
 * item (as attn_fwd_schedule); otherwise KV tiles [*kv_tile0, *kv_tile0 +
 * *kv_count) of both Q tiles, and when that is not all of them, *slot >= 0 is
 * the split's index and *part is 0 for the part holding KV tile 0, 1 for the
 * other. */
int attn_fwd_segment(int cta, int round, int grid, int64_t work_items, int kv_tiles, int flags,
                     int* item, int* kv_tile0, int* kv_count, int* slot, int* part);

/*
 * attn_fwd_host -- attn_fwd_ex with Q/K/V read from and O/LSE written to HOST
 * memory.  The pages' kernels take device tensors; this entry point is the
 * library's own end-to-end path for inputs that start on the host.
 *
 *   q, k, v     host, BF16, layout per flags as attn_fwd_ex (read)
 *   o           host, BF16, q's shape (written)
 *   lse         host, fp32, [B, H, Sq] (written) or NULL
 *   workspace   device memory owned by the caller, 256-byte aligned, at least
 *               attn_fwd_host_workspace() bytes; holds the device copies of
 *               q, k, v, o, lse; contents on entry are ignored
 *   stream      the caller's stream; the kernels run on it, the copies on two
 *               internal streams of the library that wait for the work already
 *               queued on it, and it waits for the last copy back
 *
 * The problem is split into chunks of whole heads ([B,H,S,D]) or whole batch
 * entries ([B,S,H,D]); each chunk's host-to-device copy, kernel and copy back
 * are ordered by events so chunks overlap one another.  Host buffers should be
 * page-locked (cudaHostAlloc / pinned) for the copies to be asynchronous;
 * pageable memory works but the copies then block the calling thread.  o and lse
 * hold the result once `stream` has completed the call's work.  The workspace
 * must not be used by other work until then.  Sizes, scale, flags and errors
 * as attn_fwd_ex, plus ATTN_ERR_INVALID_ARG for a NULL or short or misaligned
 * workspace.  Calls from several threads are serialised while they enqueue.
 */
int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                  int Sq, int Sk, int D, float scale, int flags, void* workspace,
                  size_t workspace_bytes, void* stream);

/*
 * attn_fwd_host_workspace -- bytes of device workspace attn_fwd_host needs for
 * this problem (written to *bytes).  Host only; errors as attn_fwd_ex's checks.
 */
int attn_fwd_host_workspace(int B, int H, int Sq, int Sk, int D, int flags, size_t* bytes);

/*
 * attn_fwd_host_chunking -- how attn_fwd_host splits the problem for a device of
 * num_sms SMs: chunks of *units_per_chunk heads ([B,H,S,D]) or batch entries
 * ([B,S,H,D]), the last one shorter if they do not divide evenly; *chunks in
 * all, at most 8.  The chunk size is chosen so the chunks' work items fill whole
 * rounds of the persistent grid where possible, with more chunks (more overlap
 * of copies and kernels) breaking ties.  Host only.
 */
int attn_fwd_host_chunking(int B, int H, int Sq, int Sk, int flags, int num_sms,
                           int64_t* units_per_chunk, int64_t* chunks);

/*
 * attn_bwd -- enqueue the backward of attn_fwd(_ex) on `stream`: given the
 * forward's inputs, its output o and natural-log lse, and dout = dL/dO, write
 *     dv = P^T dout,   dk = scale * dS^T q,   dq = scale * dS k,
 *     dS = P o (dout v^T - delta),   delta_i = sum_d dout_id o_id,
 *     P  = exp(scale * q k^T - lse)  (masked entries 0 with ATTN_FLAG_CAUSAL).
 * The LSE the forward stores is this pass's residual ("Attention for sm90,
 * Line by Line", the exp2 question: natural-log units, or the gradients are
 * wrong while the forward is right).
 *
 *   q, o, dout, dq   device, BF16, [B, H, Sq, D] contiguous (dq written), or
 *                    [B, Sq, H, D] with ATTN_FLAG_BSHD
 *   k, v, dk, dv     device, BF16, [B, H, Sk, D] contiguous (dk, dv written), or
 *                    [B, Sk, H, D] with ATTN_FLAG_BSHD
 *   lse              device, fp32, [B, H, Sq], read (attn_fwd's lse), either layout
 *   delta            device, fp32, [B, H, Sq]: scratch owned by the caller, written
 *                    with delta_i and read back by the same call
 *   flags            ATTN_FLAG_CAUSAL (must match the forward) and/or ATTN_FLAG_BSHD;
 *                    any other bit gives ATTN_ERR_INVALID_ARG
 *
 * Sizes, scale, alignment (16 bytes for BF16 tensors, 4 for lse and delta),
 * ownership and error rules as attn_fwd; no output may overlap any input or
 * another output.  Sq == 0 zero-fills dk and dv.  Deterministic: every
 * gradient element is written by exactly one thread, no atomics.
 * Asynchronous: three kernels.  delta, then dk/dv, on `stream`; dq on an
 * internal stream of the library (one per device) that first waits for the
 * work on `stream` up to delta, so the two gradient kernels share the GPU;
 * `stream` then waits for dq.  Everything the call enqueues completes before
 * any later work on `stream` starts, as if all three ran on it.  The internal
 * stream is shared by every call on the device, so dq kernels of calls made
 * on different streams run one after another.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, float* delta, int B, int H,
             int Sq, int Sk, int D, float scale, int flags, void* stream);

/*
 * attn_bwd_noalloc -- attn_bwd for callers that cannot allocate device memory.
 * (No counterpart in the pages; this is a property of the library, not of the
 * method.)  Some callers may not call cudaMalloc around this library: code
 * running under a memory budget or inside an allocator of its own, embedders
 * that own every device allocation, or paths where an allocation would
 * synchronise the device.  attn_bwd needs a [B, H, Sq] fp32 scratch buffer
 * (delta); this entry point takes no such buffer and uses a fixed array
 * compiled into the library instead, so it allocates nothing: no cudaMalloc,
 * cudaFree or allocating library call, on any call (see below for what the
 * first call on a device sets up).
 *
 * Arguments as attn_bwd without `delta`.  Limit: B * H * Sq <= 1,048,576
 * (the array is 4 MiB); larger problems return ATTN_ERR_TOO_LARGE without
 * launching.  Every GPU that loads the library holds the 4 MiB array until the
 * process exits.
 *
 * The first call on a device does the library's one-time set-up for that
 * device, with that device current: it checks the device and sets the kernels'
 * attributes (as the first call of any entry point here does), looks up the
 * array's device address (cudaGetSymbolAddress, which may load the library's
 * device code and place the array), and creates the internal stream and two
 * events the backward uses (as attn_bwd's first call does).  None of these
 * allocate through cudaMalloc, but they are not capturable: make that first call
 * before any stream capture.  All calls share the one array: two calls whose kernels
 * overlap on the GPU (different streams, no ordering between them) race on it
 * and give wrong gradients.  Calls ordered on one stream are safe; the array
 * keeps the last call's contents, which the next call overwrites before reading.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                     const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                     int H, int Sq, int Sk, int D, float scale, int flags, void* stream);

/* Static text for a status code (never NULL). */
const char* attn_status_string(int status);

/*
 * attn_fwd_plan -- the launch attn_fwd would make, computed on the host only
 * (no CUDA call when num_sms > 0; num_sms <= 0 queries the current device).
 * Same argument checks as attn_fwd for the sizes.  Work decomposition:
 * "B200 Attention Kernel from Scratch to Near-SOTA in 60 Diagrams", Chapter 5
 * (two 128-row Q tiles per work item) and Chapter 14 (one persistent CTA per
 * SM, work_id += gridDim.x).
 */
typedef struct attn_plan {
  int64_t work_items;  /* B*H*ceil(ceil(Sq/128)/2): (batch*head, pair of Q tiles) */
  int grid;            /* persistent CTAs = min(num_sms, work_items) */
  int threads;         /* threads per CTA */
  int q_tiles;         /* ceil(Sq / 128) per head */
  int kv_tiles;        /* ceil(Sk / 128): KV-loop iterations per work item */
  int kv_stages;       /* shared-memory K/V ring slots */
  int smem_bytes;      /* dynamic shared memory per CTA */
  int tmem_cols;       /* tensor-memory columns per CTA */
} attn_plan;

int attn_fwd_plan(int B, int H, int Sq, int Sk, int D, int flags, int num_sms, attn_plan* plan);

/*
 * attn_fwd_work_item -- what work item `item` covers, decoded as the kernel
 * does: the flattened batch*head, its first Q tile, and the number of KV tiles
 * each of its two Q tiles attends (kv_tiles1 = 0 when the item has one Q
 * tile).  Host only.
 */
int attn_fwd_work_item(int64_t item, int B, int H, int Sq, int Sk, int flags, int* bh,
                       int* q_tile0, int* kv_tiles0, int* kv_tiles1);

/*
 * attn_fwd_schedule -- the work item persistent CTA `cta` (of `grid`) runs in
 * its round-th turn, or -1 when it has none left; the kernel's own schedule.
 * Host only.
 */
int attn_fwd_schedule(int cta, int round, int grid, int64_t work_items, int flags);

/*
 * attn_device_status -- read (and with clear != 0, reset) the current device's
 * status word.  Bit 0..3: a bounded wait inside the kernel expired (TMA,
 * MMA, softmax, correction role); bit 4: a drain of in-flight work expired;
 * bit 5: the tensor-memory allocation did not start at column 0 (the CTA
 * skipped its work); bit 6: a backward dQ CTA found its dynamic shared memory
 * not 1024-byte aligned (it skipped its work).
 * Zero means no kernel since the last reset hit a wait limit.  Synchronous:
 * copies 4 bytes from the device (waits for prior work on the legacy stream).
 */
int attn_device_status(unsigned int* word, int clear);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_H_ */
