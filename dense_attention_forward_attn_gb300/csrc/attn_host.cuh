// attn_host.cuh -- the host-buffer forward (attn_fwd_host): Q/K/V in host memory, O/LSE written
// back to host memory, with the copies pipelined against the kernel.
//
// The problem is cut into chunks of whole heads ([B,H,S,D]) or whole batch entries ([B,S,H,D]),
// each a contiguous block of every tensor.  Chunk c's host-to-device copy runs on one internal
// stream, its kernel on the caller's stream once that copy is done, and its device-to-host copy
// on a second internal stream once the kernel is done, so copies of one chunk overlap the
// kernel and copies of others.  Chunk sizes are chosen so each chunk's work items fill whole
// rounds of the persistent grid (see host_chunk_units).
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

namespace attn {
namespace host {

constexpr int kMaxChunks = 8;

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Byte offsets of the device copies inside the caller's workspace.
struct Layout {
  size_t q, k, v, o, lse, total;
};

inline Layout layout(int64_t bh, int64_t sq, int64_t sk, int64_t d) {
  Layout L;
  const size_t nq = static_cast<size_t>(bh * sq * d) * 2, nk = static_cast<size_t>(bh * sk * d) * 2;
  L.q = 0;
  L.k = L.q + align256(nq);
  L.v = L.k + align256(nk);
  L.o = L.v + align256(nk);
  L.lse = L.o + align256(nq);
  L.total = L.lse + align256(static_cast<size_t>(bh * sq) * 4);
  return L;
}

// Units (heads or batch entries) per chunk.  Candidates hold r full rounds of the grid
// (r = 1..), at most max_chunks chunks; the one whose chunks need the fewest grid rounds in
// total (best filled waves) wins, ties going to the one with more chunks (more overlap).
inline int64_t host_chunk_units(int64_t units, int64_t items_per_unit, int64_t grid,
                                int64_t max_chunks) {
  if (units <= 1 || items_per_unit <= 0 || grid <= 0) return units > 0 ? units : 1;
  int64_t best = units, best_rounds = -1, best_chunks = 1;
  for (int64_t r = 1; r <= 64; ++r) {
    int64_t c = r * grid / items_per_unit;
    if (c < 1) c = 1;
    if (c > units) c = units;
    const int64_t chunks = (units + c - 1) / c;
    if (chunks <= max_chunks) {
      int64_t rounds = 0;
      for (int64_t u = 0; u < units; u += c) {
        const int64_t n = (units - u < c ? units - u : c) * items_per_unit;
        rounds += (n + grid - 1) / grid;
      }
      if (best_rounds < 0 || rounds < best_rounds ||
          (rounds == best_rounds && chunks > best_chunks)) {
        best = c;
        best_rounds = rounds;
        best_chunks = chunks;
      }
    }
    if (c == units) break;
  }
  return best;
}

struct Pipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t ev_in[kMaxChunks], ev_k[kMaxChunks], ev_out[kMaxChunks];
};

}  // namespace host
}  // namespace attn
