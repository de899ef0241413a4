// Decode-time threshold pruning of a compacted cache (KVzap: Fast, Adaptive,
// and Faithful KV Cache Pruning, §2.3: the w most recent tokens are always
// kept, a token scoring below tau is dropped, and the pruning sits after the
// attention op, in decoding as in prefilling), and the per-row score array it
// reads.
//
// A head's rows are in token order: rows [0, len - w) have been judged, the
// last w rows are the window.  After a decode step has appended one row per
// head, the token that just left the window is row e = len - w - 1; when it
// is not a sink and its score is not >= tau, rows e+1 .. len-1 of every pool
// (K and V rows, or their codes and group parameters) and of the score array
// move down by one row and len shrinks by one.
//
// Mapping: one CTA per head.  A head that keeps its token only stores the new
// token's score.  (The ring form below moves one row per drop instead.)  A head that drops moves w rows of every pool in phases of
// 256 threads x 16 16-byte vectors (one phase for K and V rows of 256 bytes
// at w = 128): every phase is loaded into registers, the CTA synchronises,
// then the phase is stored one row lower.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 16;                     // 16-byte vectors per thread and phase
constexpr int kChunk = kThreads * kVec;      // vectors per phase

struct PrunePools {
  uint4* base[KVC_PRUNE_MAX_POOLS];
  int vpr[KVC_PRUNE_MAX_POOLS];              // 16-byte vectors per row
  int n;
};

__global__ void __launch_bounds__(kThreads, 3)
decode_prune_kernel(PrunePools pools, float* __restrict__ rscore,
                    const int64_t* __restrict__ start, int32_t* __restrict__ len,
                    const float* __restrict__ s_new, int window, int n_sink, float tau,
                    int64_t capacity_rows, int* status) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  const int64_t s0 = start[i];
  const int L = len[i];
  if (L < 1) return;
  if (s0 < 0 || s0 + L > capacity_rows) {
    if (threadIdx.x == 0) report(status, KVC_ERR_RANGE);
    return;
  }
  const float sn = s_new[i];
  const int e = L - window - 1;
  // the exiting token's score, read before any thread writes the array
  const float se = e >= n_sink ? rscore[s0 + e] : 0.f;
  const bool drop = e >= n_sink && !(se >= tau);
  if (!drop) {
    if (threadIdx.x == 0) rscore[s0 + L - 1] = sn;
    return;
  }
  // Rows e+1 .. L-1 (the window) move to e .. L-2 in every pool, and their
  // scores with them; the new token's score goes straight to its new row
  // L-2.  The pools' window rows form one index space of
  // window * sum(vpr) vectors; each phase loads kChunk of them (and up to
  // kThreads scores) into registers, synchronises, and stores them one row
  // lower.  A phase's stores trail its loads by one row, so they never reach
  // what a later phase loads.
  int64_t first[KVC_PRUNE_MAX_POOLS + 1];
  first[0] = 0;
#pragma unroll
  for (int p = 0; p < KVC_PRUNE_MAX_POOLS; ++p)
    first[p + 1] = first[p] + (p < pools.n ? (int64_t)window * pools.vpr[p] : 0);
  const int64_t total = first[KVC_PRUNE_MAX_POOLS];
  const int nscore = window - 1;
  for (int64_t c0 = 0, f0 = 0; c0 < total || f0 < nscore; c0 += kChunk, f0 += kThreads) {
    // vector q of the index space -> its address in row e+1+ of its pool
    auto src_of = [&](int64_t q, int& vpr) {
      uint4* base = pools.base[0];
      int64_t q0 = 0;
      vpr = pools.vpr[0];
#pragma unroll
      for (int k = 1; k < KVC_PRUNE_MAX_POOLS; ++k)
        if (q >= first[k]) { base = pools.base[k]; vpr = pools.vpr[k]; q0 = first[k]; }
      return base + (s0 + e + 1) * vpr + (q - q0);
    };
    uint4 r[kVec];
#pragma unroll
    for (int x = 0; x < kVec; ++x) {
      const int64_t q = c0 + x * kThreads + threadIdx.x;
      int vpr;
      if (q < total) r[x] = *src_of(q, vpr);
    }
    const int64_t f = f0 + threadIdx.x;
    float sf = 0.f;
    if (f < nscore) sf = rscore[s0 + e + 1 + f];
    __syncthreads();
#pragma unroll
    for (int x = 0; x < kVec; ++x) {
      const int64_t q = c0 + x * kThreads + threadIdx.x;
      int vpr;
      if (q < total) {
        uint4* src = src_of(q, vpr);
        *(src - vpr) = r[x];
      }
    }
    if (f < nscore) rscore[s0 + e + f] = sf;
  }
  if (threadIdx.x == 0) {
    rscore[s0 + L - 2] = sn;
    len[i] = L - 1;
  }
}

// Ring form: a head's rows are unordered; its last `window` appended rows (the
// window) are a FIFO held in ring[i * window + s], the entry of step counter t
// in slot t % window (-1: no row).  After the step with counter t_new
// appended row len - 1, slot t_new % window holds the row that leaves the
// window: if it goes, the new row moves into it (every pool and the score)
// -- one row, not the window.  One warp per head; lanes copy the row's
// 16-byte vectors of every pool.
constexpr int kRingWarps = 8;

__global__ void __launch_bounds__(kRingWarps * 32)
decode_prune_ring_kernel(PrunePools pools, float* __restrict__ rscore,
                         const int64_t* __restrict__ start, int32_t* __restrict__ len,
                         int32_t* __restrict__ ring, int64_t t_new,
                         const float* __restrict__ s_new, int n_heads, int window, int n_sink,
                         float tau, int64_t capacity_rows, int* status) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x * kRingWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= n_heads) return;
  const int64_t s0 = start[i];
  const int L = len[i];
  if (L < 1) return;
  if (s0 < 0 || s0 + L > capacity_rows) {
    if (lane == 0) report(status, KVC_ERR_RANGE);
    return;
  }
  const int slot = (int)(t_new % window);
  int32_t* rs = ring + (int64_t)i * window + slot;
  const int nrow = L - 1;                          // the new token's row
  const float sn = s_new[i];
  int e = *rs;                                     // the row leaving the window (-1: none)
  if (e >= nrow) {                                 // not a row of this head's window
    if (lane == 0) report(status, KVC_ERR_RANGE);
    e = -1;
  }
  // the sinks are the head's first rows and never move: a window reaching
  // back to them keeps them
  const bool drop = e >= n_sink && !(rscore[s0 + e] >= tau);
  if (!drop) {
    __syncwarp();
    if (lane == 0) {
      rscore[s0 + nrow] = sn;
      *rs = nrow;
    }
    return;
  }
  for (int p = 0; p < pools.n; ++p) {
    const int vpr = pools.vpr[p];
    const uint4* src = pools.base[p] + (s0 + nrow) * vpr;
    uint4* dst = pools.base[p] + (s0 + e) * vpr;
    for (int x = lane; x < vpr; x += 32) dst[x] = src[x];
  }
  __syncwarp();
  if (lane == 0) {
    rscore[s0 + e] = sn;
    *rs = e;
    len[i] = nrow;
  }
}

// The FIFO of a head whose last `window` rows are its window in append order:
// counter t_next - window + k (k < window) -> row len - window + k in slot
// (t_next - window + k) % window; slots of rows a short head lacks get -1.
__global__ void __launch_bounds__(kThreads)
prune_ring_init_kernel(const int32_t* __restrict__ len, int n_heads, int window, int64_t t_next,
                       int32_t* __restrict__ ring, int* status) {
  pdl_wait();
  pdl_trigger();
  (void)status;
  const int64_t x = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  if (x >= (int64_t)n_heads * window) return;
  const int i = (int)(x / window), k = (int)(x - (int64_t)i * window);
  const int64_t t = t_next - window + k;
  const int64_t row = (int64_t)len[i] - window + k;
  const int slot = (int)(((t % window) + window) % window);
  ring[(int64_t)i * window + slot] = row >= 0 ? (int32_t)row : -1;
}

__global__ void __launch_bounds__(kThreads)
gather_scores_kernel(const float* __restrict__ scores, int T,
                     const int32_t* __restrict__ kept_idx, const int32_t* __restrict__ counts,
                     const int64_t* __restrict__ start, float* __restrict__ rscore,
                     int64_t capacity_rows, int* status) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.y;
  const int j = blockIdx.x * kThreads + threadIdx.x;
  if (j >= T || j >= counts[i]) return;
  const int32_t t = kept_idx[(int64_t)i * T + j];
  const int64_t dst = start[i] + j;
  if (t < 0 || t >= T || dst < 0 || dst >= capacity_rows) {
    report(status, KVC_ERR_RANGE);
    return;
  }
  rscore[dst] = scores[(int64_t)i * T + t];
}

}  // namespace

int decode_prune_launch(void* const* pools, const int* row_bytes, int n_pools, float* rscore,
                        const int64_t* start, int32_t* len, const float* s_new, int n_heads,
                        int window, int n_sink, float tau, int64_t capacity_rows, const Dev& dev,
                        cudaStream_t s) {
  if (n_heads == 0) return KVC_OK;
  PrunePools pp = {};
  pp.n = n_pools;
  for (int p = 0; p < n_pools; ++p) {
    pp.base[p] = static_cast<uint4*>(pools[p]);
    pp.vpr[p] = row_bytes[p] / 16;
  }
  return launch_pdl(decode_prune_kernel, dim3((unsigned)n_heads), dim3(kThreads), 0, s, pp,
                    rscore, start, len, s_new, window, n_sink, tau, capacity_rows, dev.status);
}

int decode_prune_ring_launch(void* const* pools, const int* row_bytes, int n_pools,
                             float* rscore, const int64_t* start, int32_t* len, int32_t* ring,
                             int64_t t_new, const float* s_new, int n_heads, int window,
                             int n_sink, float tau, int64_t capacity_rows, const Dev& dev,
                             cudaStream_t s) {
  if (n_heads == 0) return KVC_OK;
  PrunePools pp = {};
  pp.n = n_pools;
  for (int p = 0; p < n_pools; ++p) {
    pp.base[p] = static_cast<uint4*>(pools[p]);
    pp.vpr[p] = row_bytes[p] / 16;
  }
  const unsigned blocks = (unsigned)((n_heads + kRingWarps - 1) / kRingWarps);
  return launch_pdl(decode_prune_ring_kernel, dim3(blocks), dim3(kRingWarps * 32), 0, s, pp,
                    rscore, start, len, ring, t_new, s_new, n_heads, window, n_sink, tau,
                    capacity_rows, dev.status);
}

int prune_ring_init_launch(const int32_t* len, int n_heads, int window, int64_t t_next,
                           int32_t* ring, const Dev& dev, cudaStream_t s) {
  const int64_t n = (int64_t)n_heads * window;
  if (n == 0) return KVC_OK;
  return launch_pdl(prune_ring_init_kernel, dim3((unsigned)((n + kThreads - 1) / kThreads)),
                    dim3(kThreads), 0, s, len, n_heads, window, t_next, ring, dev.status);
}

int gather_scores_launch(const float* scores, int U, int Hkv, int T, const int32_t* kept_idx,
                         const int32_t* counts, const int64_t* start, float* rscore,
                         int64_t capacity_rows, const Dev& dev, cudaStream_t s) {
  const int n = U * Hkv;
  if (n == 0 || T == 0) return KVC_OK;
  const dim3 grid((unsigned)((T + kThreads - 1) / kThreads), (unsigned)n);
  return launch_pdl(gather_scores_kernel, grid, dim3(kThreads), 0, s, scores, T, kept_idx,
                    counts, start, rscore, capacity_rows, dev.status);
}

}  // namespace kvc
