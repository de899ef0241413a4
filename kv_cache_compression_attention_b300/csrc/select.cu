// Budget selection: global top-k across heads, per-head top-k, or a fixed
// threshold, always keeping the protected sinks and recent window.
//
// Sources: KVzap §2.3 (fixed budget "keep exactly x%", or a threshold tau on
// the scores, with the w most recent tokens always kept); KV Cache Transform
// Coding §2A and KVSculpt §2A (sinks and the recent window are not
// compressed); KVSculpt §2D (heads of one layer end up with different
// budgets -- the global pool gives exactly that).
//
// Design (one thread-block cluster per selection pool):
//  * A pool is one unit's Hkv heads (global top-k) or one head (per-head
//    budget, threshold).  The cluster's C CTAs split the pool's tokens into
//    C contiguous ranges; each CTA keeps its range's order-preserving uint32
//    keys in shared memory, head-major (keys[head][token]), so every pass
//    over them is a conflict-free sweep of consecutive words.
//  * Radix select, 4 passes of 8-bit digits, from the most significant
//    digit: every CTA histograms its candidates that match the prefix found
//    so far (into 8 sub-histograms; one atomic per warp when all its
//    candidates share the digit, as in the first pass), adds its
//    histogram into rank 0's with distributed-shared-memory atomics, and
//    after one cluster barrier every CTA reads the totals and picks the same
//    digit.  After the last pass the exact key of the need-th largest
//    candidate (thr) and how many of its equal-key elements to keep are known.
//  * Ties (key == thr) are only ranked when not all of them are kept: a
//    cluster prefix of per-CTA tie counts, then a block scan over tokens of
//    the per-token tie counts, gives the first dropped tie in the tie-break
//    order (token asc, head asc), as an element index e = t * hps + head.
//  * Emission: a counting sweep and a cluster prefix give each CTA its base
//    per head; a block-wide ballot scan over consecutive tokens then writes
//    the ascending token indices of each head.
//  * Offsets (exclusive scan of the counts): a launch with a single pool
//    writes them from rank 0; otherwise a separate single-block kernel scans
//    the counts of all pools (threshold pools have data-dependent totals).
// Every decision is an integer comparison on the fp32 bit patterns, so the
// result is bit-exact and deterministic.
#include <cooperative_groups.h>

#include <map>
#include <mutex>
#include <tuple>

#include "kvc_internal.cuh"

namespace cg = cooperative_groups;

namespace kvc {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxHps = 8;                 // heads per pool kept in registers
constexpr uint32_t kNoThr = 0xffffffffu;   // larger than every real key

struct Args {
  const float* scores;
  int T, hps, mode;
  int64_t need_global;
  float tau;
  const int32_t* head_budget;
  int n_sink, n_recent, nP;
  int32_t* kept;
  int32_t* counts;
  int64_t* offsets;   // written here when the launch has a single pool, else NULL
};

constexpr int kSubHist = 8;              // sub-histograms (4 warps each)
constexpr int kList2 = 4096;             // capacity of the second candidate list

struct Shared {
  uint32_t hist[kSubHist][256];       // this CTA's sub-histograms of the current pass
  uint32_t tot[4][256];               // cluster totals per pass (summed into rank 0)
  uint32_t totl[256];                 // this CTA's copy of the pass totals
  uint32_t warp_tmp[2][kWarps];       // block scans (double-buffered)
  uint32_t warp_tot[2];
  uint32_t hcnt[kWarps][kMaxHps];     // per-warp kept counts per head
  uint32_t emit_tmp[2][kMaxHps][kWarps];  // emission scans (double-buffered)
  uint32_t emit_tot[2][kMaxHps];
  uint32_t xchg_ties;                 // read remotely
  uint32_t xchg_cnt[kMaxHps];         // read remotely
  uint32_t head_base[kMaxHps];
  uint32_t head_total[kMaxHps];
  uint32_t sel_bin, sel_above, sel_count, ecut, tie_base, nlist;
  uint32_t list2[kList2];             // candidates of the last two passes
};

__device__ __forceinline__ bool is_prot(int t, int T, int n_sink, int n_recent) {
  return t < n_sink || t >= T - n_recent;
}

// Exclusive block scan of one value per thread; returns the prefix and sets
// *total.  Two barriers; consecutive calls alternate scratch buffers.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, Shared& sh, int& buf, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += n;
  }
  uint32_t* wt = sh.warp_tmp[buf];
  if (lane == 31) wt[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t x = wt[lane];
    uint32_t y = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, y, off);
      if (lane >= off) y += n;
    }
    wt[lane] = y - x;
    if (lane == 31) sh.warp_tot[buf] = y;
  }
  __syncthreads();
  const uint32_t r = wt[warp] + incl - v;
  *total = sh.warp_tot[buf];
  buf ^= 1;
  return r;
}

__global__ void __launch_bounds__(kThreads, 1)
select_kernel(Args a) {
  cg::cluster_group cl = cg::this_cluster();
  const int C = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const int seg = blockIdx.y;
  const int hps = a.hps;
  const int T = a.T;
  const int head0 = seg * hps;
  const int t0 = (int)((int64_t)rank * T / C);
  const int t1 = (int)((int64_t)(rank + 1) * T / C);
  const int nt = t1 - t0;
  const int nloc = nt * hps;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int sbuf = 0;

  extern __shared__ __align__(16) uint8_t smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + ((sizeof(Shared) + 15) & ~size_t(15)));
  // (the first candidate list follows the keys: nloc more words)

  for (int i = tid; i < 4 * 256; i += kThreads) (&sh.tot[0][0])[i] = 0u;
  for (int i = tid; i < kSubHist * 256; i += kThreads) (&sh.hist[0][0])[i] = 0u;

  // ---- phase A: keys of this CTA's token range, head-major (coalesced
  // global reads, conflict-free shared stores, sixteen loads in flight);
  // item q covers head q / nch, vector slots (q % nch) * 1024 + tid.  When the
  // rows and the range are 16-byte aligned every slot is a float4 of 4 tokens.
  {
    const bool vec = ((T | t0 | nt) & 3) == 0 && (reinterpret_cast<uintptr_t>(a.scores) & 15u) == 0;
    const int per = vec ? 4 : 1;                       // tokens per slot
    const int nslot = nt / per;
    const int nch = (nslot + kThreads - 1) / kThreads;
    const int nq = hps * nch;
    for (int q0 = 0; q0 < nq; q0 += 8) {
      float4 sv[8];
      int hh = q0 / nch, jc = q0 - (q0 / nch) * nch;
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const int js = jc * kThreads + tid;
        if (q0 + x < nq && js < nslot) {
          const float* row = a.scores + (int64_t)(head0 + hh) * T + t0;
          if (vec) sv[x] = __ldg(reinterpret_cast<const float4*>(row) + js);
          else sv[x].x = __ldg(row + js);
        }
        if (++jc == nch) { jc = 0; ++hh; }
      }
      hh = q0 / nch; jc = q0 - hh * nch;
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const int js = jc * kThreads + tid;
        if (q0 + x < nq && js < nslot) {
          const int j = js * per;
          uint32_t* dst = keys + hh * nt + j;
          if (vec) {
            uint4 kk;
            kk.x = is_prot(t0 + j, T, a.n_sink, a.n_recent) ? 0u : score_key(sv[x].x);
            kk.y = is_prot(t0 + j + 1, T, a.n_sink, a.n_recent) ? 0u : score_key(sv[x].y);
            kk.z = is_prot(t0 + j + 2, T, a.n_sink, a.n_recent) ? 0u : score_key(sv[x].z);
            kk.w = is_prot(t0 + j + 3, T, a.n_sink, a.n_recent) ? 0u : score_key(sv[x].w);
            *reinterpret_cast<uint4*>(dst) = kk;
          } else {
            dst[0] = is_prot(t0 + j, T, a.n_sink, a.n_recent) ? 0u : score_key(sv[x].x);
          }
        }
        if (++jc == nch) { jc = 0; ++hh; }
      }
    }
  }
  // every CTA of the cluster is running and its totals are zero before any
  // remote update
  cl.sync();

  // ---- phase B: radix select of the need-th largest candidate key
  int64_t need = 0;
  if (a.mode == KVC_SEL_GLOBAL_TOPK) {
    need = a.need_global;
  } else if (a.mode == KVC_SEL_PER_HEAD) {
    int64_t b = a.head_budget[head0];
    if (b < a.nP) b = a.nP;
    if (b > T) b = T;
    need = b - a.nP;
  }
  uint32_t thr = kNoThr;
  uint32_t ecut = 0;
  if (a.mode == KVC_SEL_THRESHOLD) {
    thr = (a.tau != a.tau) ? kNoThr : score_key(a.tau);
  } else if (need > 0) {
    uint32_t prefix = 0, pmask = 0;
    uint32_t krem = (uint32_t)need;
    uint32_t last_count = 0;
    uint32_t* myhist = sh.hist[warp & (kSubHist - 1)];
    // candidates of the later passes: after pass 0 the keys whose top byte
    // matches are copied to list1; after pass 1 those matching 16 bits go to
    // list2 when they fit (otherwise pass 2 and 3 scan list1 again)
    uint32_t* list1 = keys + nloc;
    uint32_t* list2 = sh.list2;
    const uint32_t* src = keys;
    int nsrc = nloc;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      if (pass > 0) {
        for (int i = tid; i < kSubHist * 256; i += kThreads) (&sh.hist[0][0])[i] = 0u;
        __syncthreads();
      }
      for (int e0 = 0; e0 < nsrc; e0 += kThreads) {
        const int e = e0 + tid;
        bool cand = false;
        uint32_t digit = 0u;
        if (e < nsrc) {
          const uint32_t key = src[e];
          cand = key != 0u && (key & pmask) == prefix;
          digit = (key >> shift) & 255u;
        }
        // one atomic per warp when all its candidates share a digit (the
        // common case in the first pass), else one per candidate
        const uint32_t cmask = __ballot_sync(0xffffffffu, cand);
        if (cmask) {
          const uint32_t d0 = __shfl_sync(0xffffffffu, digit, __ffs(cmask) - 1);
          if (__all_sync(0xffffffffu, !cand || digit == d0)) {
            if (lane == 0) atomicAdd(&myhist[d0], (uint32_t)__popc(cmask));
          } else if (cand) {
            atomicAdd(&myhist[digit], 1u);
          }
        }
      }
      __syncthreads();
      // every CTA adds its histogram into rank 0's totals of this pass
      if (tid < 256) {
        uint32_t h = 0;
#pragma unroll
        for (int x = 0; x < kSubHist; ++x) h += sh.hist[x][tid];
        if (h) atomicAdd(cl.map_shared_rank(&sh.tot[pass][tid], 0), h);
      }
      cl.sync();
      if (tid < 256) sh.totl[tid] = *cl.map_shared_rank(&sh.tot[pass][tid], 0);
      __syncthreads();
      if (warp == 0) {
        uint32_t cnt[8];
        uint32_t lsum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) { cnt[i] = sh.totl[lane * 8 + i]; lsum += cnt[i]; }
        uint32_t suffix = lsum;                  // sum over lanes >= lane
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          uint32_t n = __shfl_down_sync(0xffffffffu, suffix, off);
          if (lane + off < 32) suffix += n;
        }
        uint32_t above = suffix - lsum;          // candidates in higher lanes' bins
#pragma unroll
        for (int i = 7; i >= 0; --i) {
          if (above < krem && krem <= above + cnt[i]) {
            sh.sel_bin = lane * 8 + i;
            sh.sel_above = above;
            sh.sel_count = cnt[i];
          }
          above += cnt[i];
        }
      }
      __syncthreads();
      const uint32_t bin = sh.sel_bin;
      krem -= sh.sel_above;
      last_count = sh.sel_count;
      prefix |= bin << shift;
      pmask |= 255u << shift;
      if (pass < 2) {
        // compact this CTA's candidates of the next pass (warp-aggregated appends)
        uint32_t* dst = (pass == 0) ? list1 : list2;
        const int cap = (pass == 0) ? nloc : kList2;
        if (tid == 0) sh.nlist = 0u;
        __syncthreads();
        for (int e0 = 0; e0 < nsrc; e0 += kThreads) {
          const int e = e0 + tid;
          uint32_t key = 0u;
          bool keep = false;
          if (e < nsrc) {
            key = src[e];
            keep = key != 0u && (key & pmask) == prefix;
          }
          const uint32_t bm = __ballot_sync(0xffffffffu, keep);
          uint32_t base = 0u;
          if (lane == 0 && bm) base = atomicAdd(&sh.nlist, (uint32_t)__popc(bm));
          base = __shfl_sync(0xffffffffu, base, 0);
          const uint32_t at = base + __popc(bm & ((1u << lane) - 1u));
          if (keep && at < (uint32_t)cap) dst[at] = key;
        }
        __syncthreads();
        if (sh.nlist <= (uint32_t)cap) { src = dst; nsrc = (int)sh.nlist; }
        __syncthreads();
      }
    }
    thr = prefix;
    // ---- ties: keep the first krem elements with key == thr in (t, g) order
    if (krem < last_count) {
      uint32_t mine = 0;
      for (int e = tid; e < nloc; e += kThreads) mine += (keys[e] == thr);
      mine = __reduce_add_sync(0xffffffffu, mine);
      if (lane == 0) sh.warp_tmp[0][warp] = mine;
      __syncthreads();
      if (tid == 0) {
        uint32_t s = 0;
        for (int w = 0; w < kWarps; ++w) s += sh.warp_tmp[0][w];
        sh.xchg_ties = s;
      }
      __syncthreads();
      cl.sync();
      if (tid == 0) {
        uint32_t b = 0;
        for (int r = 0; r < rank; ++r) b += *cl.map_shared_rank(&sh.xchg_ties, r);
        sh.tie_base = b;
      }
      __syncthreads();
      const uint32_t base = sh.tie_base;
      const uint32_t local_ties = sh.xchg_ties;
      if (base >= krem) ecut = 0;
      else if (base + local_ties <= krem) ecut = (uint32_t)nloc;
      else {
        // the first dropped tie has local rank `want` in (token, head) order
        const uint32_t want = krem - base;     // 1 <= want < local_ties
        uint32_t carry = 0;
        for (int j0 = 0; j0 < nt; j0 += kThreads) {
          const int j = j0 + tid;
          uint32_t c = 0;
          if (j < nt)
            for (int hh = 0; hh < hps; ++hh) c += (keys[hh * nt + j] == thr);
          uint32_t total;
          const uint32_t excl = carry + block_scan(c, sh, sbuf, &total);
          if (c && excl <= want && want < excl + c) {
            uint32_t k = want - excl;          // 0-based tie index inside token j
            int hh = 0;
            for (; hh < hps; ++hh)
              if (keys[hh * nt + j] == thr) { if (k == 0) break; --k; }
            sh.ecut = (uint32_t)(j * hps + hh);
          }
          carry += total;
          if (carry > want) break;             // uniform across the block
        }
        __syncthreads();
        ecut = sh.ecut;
      }
    } else {
      ecut = (uint32_t)nloc;
    }
  }

  // kept(hh, j): protected, strictly above thr, or a kept tie
  auto kept = [&](int hh, int j) -> bool {
    const uint32_t key = keys[hh * nt + j];
    if (key == 0u) return true;
    if (a.mode == KVC_SEL_THRESHOLD) return key >= thr;
    return key > thr || (key == thr && (uint32_t)(j * hps + hh) < ecut);
  };

  // ---- phase D: per-head counts, cluster prefix, ascending emission
  for (int hh = 0; hh < hps; ++hh) {
    uint32_t c = 0;
    for (int j = tid; j < nt; j += kThreads) c += kept(hh, j);
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) sh.hcnt[warp][hh] = c;
  }
  __syncthreads();
  if (tid < hps) {
    uint32_t s = 0;
    for (int w = 0; w < kWarps; ++w) s += sh.hcnt[w][tid];
    sh.xchg_cnt[tid] = s;
  }
  cl.sync();
  if (tid < hps) {
    uint32_t base = 0, total = 0;
    for (int r = 0; r < C; ++r) {
      const uint32_t v = cl.map_shared_rank(sh.xchg_cnt, r)[tid];
      if (r < rank) base += v;
      total += v;
    }
    sh.head_base[tid] = base;
    if (rank == 0) a.counts[head0 + tid] = (int32_t)total;
    sh.head_total[tid] = total;
  }
  __syncthreads();
  // a launch with a single pool writes the offsets itself (no second kernel)
  if (a.offsets && rank == 0 && tid == 0) {
    int64_t o = 0;
    for (int hh = 0; hh < hps; ++hh) { a.offsets[hh] = o; o += sh.head_total[hh]; }
    a.offsets[hps] = o;
  }
  // one block scan per 1024-token chunk covers every head: flags by ballot,
  // per-warp counts scanned by one warp per head, positions by popcount
  uint32_t carry[kMaxHps];
#pragma unroll
  for (int hh = 0; hh < kMaxHps; ++hh) carry[hh] = (hh < hps) ? sh.head_base[hh] : 0u;
  for (int j0 = 0; j0 < nt; j0 += kThreads) {
    const int j = j0 + tid;
    uint32_t ball[kMaxHps];
    uint32_t (*wt)[kWarps] = sh.emit_tmp[sbuf];
#pragma unroll
    for (int hh = 0; hh < kMaxHps; ++hh) {
      const bool f = hh < hps && j < nt && kept(hh, j);
      ball[hh] = __ballot_sync(0xffffffffu, f);
      if (lane == 0 && hh < hps) wt[hh][warp] = __popc(ball[hh]);
    }
    __syncthreads();
    if (warp < hps) {
      const uint32_t x = wt[warp][lane];
      uint32_t y = x;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, y, off);
        if (lane >= off) y += n;
      }
      wt[warp][lane] = y - x;
      if (lane == 31) sh.emit_tot[sbuf][warp] = y;
    }
    __syncthreads();
    const uint32_t below = (1u << lane) - 1u;
#pragma unroll
    for (int hh = 0; hh < kMaxHps; ++hh) {
      if (hh >= hps) break;
      if (ball[hh] & (1u << lane))
        a.kept[(int64_t)(head0 + hh) * T + carry[hh] + wt[hh][warp] + __popc(ball[hh] & below)] = t0 + j;
      carry[hh] += sh.emit_tot[sbuf][hh];
    }
    sbuf ^= 1;
  }
  // no CTA may leave while a peer can still read its shared memory
  cl.sync();
}

// offsets[i] = sum_{j<i} counts[j], offsets[n] = total (one block).
__global__ void __launch_bounds__(1024)
offsets_kernel(const int32_t* __restrict__ counts, int n, int64_t* __restrict__ offsets) {
  __shared__ int64_t warp_sum[32];
  __shared__ int64_t carry_s;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  for (int i0 = 0; i0 < n; i0 += 1024) {
    const int i = i0 + threadIdx.x;
    const int64_t v = i < n ? (int64_t)counts[i] : 0;
    int64_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int64_t y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int64_t ws = warp_sum[lane];
      int64_t wi = ws;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, wi, off);
        if (lane >= off) wi += y;
      }
      warp_sum[lane] = wi - ws;
    }
    __syncthreads();
    const int64_t carry = carry_s;
    if (i < n) offsets[i] = carry + warp_sum[warp] + incl - v;
    __syncthreads();
    if (threadIdx.x == 1023) carry_s = carry + warp_sum[warp] + incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) offsets[n] = carry_s;
}

// keys of the CTA's range plus the same capacity for the first candidate list
size_t shared_bytes(int keys) { return ((sizeof(Shared) + 15) & ~size_t(15)) + 2ull * keys * 4; }

}  // namespace

int select_launch(const float* scores, int U, int Hkv, int T, int mode, int64_t need_global,
                  float tau, const int32_t* head_budget, int n_sink, int n_recent,
                  int32_t* kept_idx, int32_t* counts, int64_t* offsets, const Dev& dev,
                  cudaStream_t s) {
  const int hps = (mode == KVC_SEL_GLOBAL_TOPK) ? Hkv : 1;
  if (hps > kMaxHps) return KVC_ERR_UNSUPPORTED;
  const int nseg = (mode == KVC_SEL_GLOBAL_TOPK) ? U : U * Hkv;
  const int64_t pool = (int64_t)hps * T;
  const int cap = (int)((dev.max_smem_optin - (int)shared_bytes(0)) / 8);
  // the smallest cluster that keeps <= 16K keys per CTA, else the smallest that fits
  int C = 1;
  while (C < 16 && (pool + C - 1) / C > 16384) C *= 2;
  while (C < 16 && (pool + C - 1) / C > cap) C *= 2;
  if ((pool + C - 1) / C > cap) return KVC_ERR_UNSUPPORTED;
  Args a;
  a.scores = scores; a.T = T; a.hps = hps; a.mode = mode; a.need_global = need_global;
  a.tau = tau; a.head_budget = head_budget; a.n_sink = n_sink; a.n_recent = n_recent;
  a.nP = 0;
  {
    int rs = T - n_recent;
    a.nP = n_sink + (T - rs) - (rs < n_sink ? n_sink - rs : 0);
  }
  a.kept = kept_idx; a.counts = counts;
  a.offsets = (nseg == 1) ? offsets : nullptr;
  static std::mutex mu;
  static bool attr_done[64];
  static std::map<std::tuple<int, int, size_t>, int> active_memo;
  std::lock_guard<std::mutex> lock(mu);
  if (!attr_done[dev.device & 63]) {
    KVC_CUDA_TRY(cudaFuncSetAttribute(select_kernel,
                                      cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
    KVC_CUDA_TRY(cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      dev.max_smem_optin));
    attr_done[dev.device & 63] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  // a cluster must fit one GPC: shrink it (while the keys still fit) until
  // the occupancy query says at least one cluster can be resident (the
  // answer is remembered per device, cluster size and shared memory)
  for (;;) {
    const size_t smem = shared_bytes(((T + C - 1) / C) * hps);
    cfg.gridDim = dim3((unsigned)C, (unsigned)nseg, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int active = 0;
    const auto key = std::make_tuple(dev.device, C, smem);
    auto it = active_memo.find(key);
    if (it != active_memo.end()) {
      active = it->second;
    } else {
      KVC_CUDA_TRY(cudaOccupancyMaxActiveClusters(&active, select_kernel, &cfg));
      active_memo[key] = active;
    }
    if (active > 0) break;
    if (C == 1 || (pool + C / 2 - 1) / (C / 2) > cap) return KVC_ERR_UNSUPPORTED;
    C /= 2;
  }
  KVC_CUDA_TRY(cudaLaunchKernelEx(&cfg, select_kernel, a));
  if (nseg > 1) offsets_kernel<<<1, 1024, 0, s>>>(counts, U * Hkv, offsets);
  return launch_status();
}

}  // namespace kvc
