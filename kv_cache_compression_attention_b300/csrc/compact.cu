// Gather-compaction of the kept K/V rows into a contiguous variable-length
// cache (KVSculpt §1: eviction keeps a subset of the original pairs).
//
// Head i = u*Hkv + g owns rows [start_i, start_i + counts_i + slack) of the
// compacted pools, start_i = offsets_i + i*slack; its row start_i + j is the
// source row kept_idx[i, j] of head i.  Pure byte movement: HBM reads of the
// kept rows only, HBM writes of the same bytes.
//
// Mapping: a persistent grid; each warp takes blocks of 16 consecutive
// output rows.  Lane rho resolves output row r0+rho to (head, source row)
// -- one binary search over the offsets per block, then a forward walk --
// and the warp copies the block's rows with 16-byte non-caching loads and
// streaming stores, several vectors in flight per lane.
#include <atomic>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kThreads = 256;
constexpr int kBlockRows = 16;    // output rows per warp task
constexpr int kUnroll = 8;     // 16-byte vectors in flight per lane and tensor
constexpr int kMaxCachedHeads = 6144;   // offsets kept in shared memory up to this many heads

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__global__ void __launch_bounds__(kThreads)
compact_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v, int vpr_shift, int T,
               int n_heads, const int32_t* __restrict__ kept_idx,
               const int32_t* __restrict__ counts, const int64_t* __restrict__ offsets,
               int slack, uint4* __restrict__ kc, uint4* __restrict__ vc,
               int64_t capacity_rows, int64_t* __restrict__ start, int32_t* __restrict__ len,
               int* status) {
  extern __shared__ int64_t offs_sm[];      // offsets cached when they fit
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  const bool cached = n_heads < kMaxCachedHeads;
  if (cached) {
    for (int i = threadIdx.x; i <= n_heads; i += kThreads) offs_sm[i] = offsets[i];
    __syncthreads();
  }
  const int64_t* offs = cached ? offs_sm : offsets;
  // per-head start / len
  for (int i = blockIdx.x * kThreads + threadIdx.x; i < n_heads; i += gridDim.x * kThreads) {
    start[i] = offs[i] + (int64_t)i * slack;
    len[i] = counts[i];
  }
  // The offsets come from the caller.  A total outside [0, n_heads * T]
  // cannot describe kept rows of this cache: report it and copy nothing
  // (this also bounds the task loop below).
  const int64_t total = offs[n_heads];
  if (total < 0 || total > (int64_t)n_heads * T) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(status, KVC_ERR_RANGE);
    return;
  }
  const int64_t tasks = (total + kBlockRows - 1) / kBlockRows;
  const int64_t warp0 = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
  const int vpr = 1 << vpr_shift;                  // 16-byte vectors per row
  for (int64_t task = warp0; task < tasks; task += nwarps) {
    const int64_t r0 = task * kBlockRows;
    // head of the block's first row: largest i with offsets[i] <= r0
    int lo = 0, hi = n_heads - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (offs[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    // lane rho -> row r0 + rho
    const int64_t r = r0 + lane;
    int64_t src_row = -1, dst_row = -1;
    if (lane < kBlockRows && r < total) {
      int i = lo;
      while (i + 1 < n_heads && offs[i + 1] <= r) ++i;
      // row j of head i: checked against the head's count and T before its
      // index is read (offsets that disagree with the counts are the
      // caller's error and are reported, never followed)
      const int64_t j = r - offs[i];
      const int64_t dst = r + (int64_t)i * slack;
      if (j < 0 || j >= T || dst >= capacity_rows) {
        report(status, KVC_ERR_RANGE);
      } else {
        // the head's count and the index are read together (row j < T of
        // head i lies inside kept_idx whatever the count says); the index
        // is used only if j is below the count
        const int32_t cnt = __ldg(counts + i);
        const int32_t t = __ldg(kept_idx + (int64_t)i * T + j);
        if (j >= cnt || t < 0 || t >= T) {
          report(status, KVC_ERR_RANGE);
        } else {
          src_row = (int64_t)i * T + t;
          dst_row = dst;
        }
      }
    }
    const int nrows = (int)((total - r0) < kBlockRows ? (total - r0) : kBlockRows);
    const int pairs = nrows << vpr_shift;
    for (int p0 = 0; p0 < pairs; p0 += 32 * kUnroll) {
      uint4 kv[kUnroll], vv[kUnroll];
      int64_t dst[kUnroll];
#pragma unroll
      for (int x = 0; x < kUnroll; ++x) {
        const int p = p0 + x * 32 + lane;
        const int row = p >> vpr_shift;
        const int vec = p & (vpr - 1);
        const int64_t s_row = __shfl_sync(0xffffffffu, src_row, row & (kBlockRows - 1));
        const int64_t d_row = __shfl_sync(0xffffffffu, dst_row, row & (kBlockRows - 1));
        dst[x] = -1;
        if (p < pairs && s_row >= 0) {
          kv[x] = ld_stream(k + (s_row << vpr_shift) + vec);
          vv[x] = ld_stream(v + (s_row << vpr_shift) + vec);
          dst[x] = (d_row << vpr_shift) + vec;
        }
      }
#pragma unroll
      for (int x = 0; x < kUnroll; ++x) {
        if (dst[x] >= 0) {
          st_stream(kc + dst[x], kv[x]);
          st_stream(vc + dst[x], vv[x]);
        }
      }
    }
  }
}

}  // namespace

int compact_launch(const void* k, const void* v, int row_bytes, int U, int Hkv, int T,
                   const int32_t* kept_idx, const int32_t* counts, const int64_t* offsets,
                   int slack, void* kc, void* vc, int64_t capacity_rows, int64_t* start,
                   int32_t* len, const Dev& dev, cudaStream_t s) {
  const int vpr = row_bytes / 16;
  if (vpr <= 0 || (vpr & (vpr - 1)) || vpr > 32) return KVC_ERR_UNSUPPORTED;
  int shift = 0;
  while ((1 << shift) < vpr) ++shift;
  const int n_heads = U * Hkv;
  const size_t smem = n_heads < kMaxCachedHeads ? (size_t)(n_heads + 1) * sizeof(int64_t) : 0;
  // resident blocks per SM at the largest shared-memory size (a lower bound
  // for every launch), once per device
  static std::atomic<int> per_sm_memo[64];
  int per_sm = per_sm_memo[dev.device & 63].load();
  if (per_sm == 0) {
    KVC_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, compact_kernel, kThreads, (size_t)kMaxCachedHeads * sizeof(int64_t)));
    if (per_sm < 1) per_sm = 1;
    per_sm_memo[dev.device & 63].store(per_sm);
  }
  const int blocks = dev.sms * per_sm;
  return launch_pdl(compact_kernel, dim3((unsigned)blocks), dim3(kThreads), smem, s,
                    static_cast<const uint4*>(k), static_cast<const uint4*>(v), shift, T,
                    U * Hkv, kept_idx, counts, offsets, slack, static_cast<uint4*>(kc),
                    static_cast<uint4*>(vc), capacity_rows, start, len, dev.status);
}

}  // namespace kvc
