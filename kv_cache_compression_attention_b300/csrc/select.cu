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
//    C contiguous ranges; each CTA copies its range of every head's score
//    row into shared memory (bulk asynchronous copies when the rows are
//    16-byte aligned), keys[head][token], and turns the scores into
//    order-preserving uint32 keys in place, V = 4 consecutive keys per
//    thread and step when the range allows (1 otherwise).
//  * Radix select, 4 passes of 8-bit digits from the most significant one.
//    Every warp histograms into a private shared-memory histogram (one
//    shared atomic per candidate).  The first pass is counted while the
//    keys are made; the second sweeps the keys once more and appends the
//    candidates that match the first digit to the warp's own list; the
//    third and fourth sweep only that list, compacting it in place.  After
//    each pass every CTA adds its histogram into the bins' owners (bin b
//    lives in CTA b * C / 256) with distributed-shared-memory atomics, and
//    after one cluster barrier every CTA reads the 256 totals and picks the
//    same digit.  When the chosen bin is kept whole, selection stops early:
//    every key at or above the bin's smallest prefix is kept.
//  * Ties (key == thr) are only ranked when not all of them are kept: a
//    cluster prefix of per-CTA tie counts, then a block scan over tokens of
//    the per-token tie counts, gives the first dropped tie in the tie-break
//    order (token asc, head asc), as an element index e = t * hps + head.
//  * Emission: warp w owns a contiguous 1/32 of the range's tokens; per head
//    it writes its kept tokens, ascending, into its own staging segment
//    (ballot + popcount, no block barrier), then one scan over the warps
//    and a cluster prefix of the per-head counts place every segment in the
//    output with coalesced stores.
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
constexpr int kSubRange = 512;             // tokens per emission CTA of the hand-off
constexpr int kMaxSub = 64;                // sub-ranges per CTA range at most

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
  int* status;
  // non-NULL: hand the decision to emit_compact_kernel instead of emitting
  // ([C][2 + hps * hand_sub] words: threshold key, tie cut, kept count per
  // head and 512-token sub-range of the CTA's range)
  uint32_t* hand;
  int hand_sub;
  // select_kernel<V, true> (global top-k, no protected set): head i's
  // candidates are its positions t < lens[i]; the rest are neither
  // candidates nor kept, and the CTAs split only the pool's longest head
  // length, not T
  const int32_t* lens;
};

struct Shared {
  uint32_t whist[kWarps][256];        // per-warp histograms of the current pass
  uint32_t part[4][256];              // partial sums of the warp histograms
  uint32_t tot[4][256];               // per pass: totals of the bins this CTA owns
  uint32_t totl[256];                 // this CTA's copy of the pass totals
  uint32_t warp_tmp[2][kWarps];       // block scans (double-buffered)
  uint32_t warp_tot[2];
  uint32_t wcnt[kMaxHps][kWarps];     // emission: kept tokens per head and warp
  uint32_t wexcl[kMaxHps][kWarps];    // ... their exclusive prefix over warps
  uint32_t xchg_ties;                 // read remotely
  uint32_t xchg_cnt[kMaxHps];         // read remotely
  uint32_t xall[16][kMaxHps];         // every CTA's per-head counts
  uint32_t head_base[kMaxHps];
  uint32_t head_total[kMaxHps];
  uint32_t sel_bin, sel_above, sel_count, ecut, tie_base;
  uint64_t bar;                       // completion of the bulk score copies
};

// Shared-memory layout after Shared: the keys (nt * hps words, rounded up to
// 4), then one region that first holds the warps' candidate lists and later
// the emission staging segments.
struct Layout {
  int nloc, cap_w, per_w, region;
  __host__ __device__ Layout(int nt, int hps, int V) {
    nloc = nt * hps;
    // a warp visits at most ceil(nloc / (1024 V)) groups of 32 V keys
    cap_w = 32 * V * ((nloc + kThreads * V - 1) / (kThreads * V));
    per_w = (nt + kWarps - 1) / kWarps;          // emission tokens per warp
    const int lists = kWarps * cap_w, stage = hps * kWarps * per_w;
    region = lists > stage ? lists : stage;
  }
  __host__ __device__ size_t keys_words() const { return ((size_t)nloc + 3) & ~size_t(3); }
};

// Adds a candidate's digit into the warp's private histogram (lanes with
// equal digits serialise on one address, which costs less than grouping
// them first, or than testing whether the warp's digits agree); returns the
// ballot of candidates.
__device__ __forceinline__ uint32_t hist_add(uint32_t* wh, bool cand, uint32_t digit) {
  const uint32_t cm = __ballot_sync(0xffffffffu, cand);
  if (cand) atomicAdd(&wh[digit], 1u);
  return cm;
}

// V consecutive keys.
template <int V> struct Vec;
template <> struct Vec<1> {
  uint32_t k[1];
  __device__ __forceinline__ void load(const uint32_t* p) { k[0] = *p; }
  __device__ __forceinline__ void store(uint32_t* p) const { *p = k[0]; }
};
template <> struct Vec<4> {
  uint32_t k[4];
  __device__ __forceinline__ void load(const uint32_t* p) {
    const uint4 x = *reinterpret_cast<const uint4*>(p);
    k[0] = x.x; k[1] = x.y; k[2] = x.z; k[3] = x.w;
  }
  __device__ __forceinline__ void store(uint32_t* p) const {
    *reinterpret_cast<uint4*>(p) = make_uint4(k[0], k[1], k[2], k[3]);
  }
};

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

__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_plain() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Offset of the keys in dynamic shared memory; with per-head lengths they
// sit after Shared and the lengths.
template <bool kLens>
__host__ __device__ constexpr size_t keys_offset() {
  return (sizeof(Shared) + (kLens ? kMaxHps * sizeof(int) : 0) + 15) & ~size_t(15);
}

// V = 4 requires every CTA's range to start and end on a multiple of 4
// tokens and 16-byte aligned score rows (then the rows are bulk-copied).
template <int V, bool kLens>
__global__ void __launch_bounds__(kThreads, 1)
select_kernel(Args a) {
  cg::cluster_group cl = cg::this_cluster();
  const int C = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const int seg = blockIdx.y;
  const int hps = a.hps;
  const int T = a.T;
  const int head0 = seg * hps;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  int sbuf = 0;
  // this CTA's token range: of T, or (kLens) of the pool's longest head
  int t0 = 0, t1 = 0;
  if constexpr (!kLens) {
    t0 = (int)((int64_t)rank * T / C);
    t1 = (int)((int64_t)(rank + 1) * T / C);
  }

  extern __shared__ __align__(16) uint8_t smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  int* lenh = reinterpret_cast<int*>(smem_raw + sizeof(Shared));   // kLens: [hps]

  for (int i = tid; i < 4 * 256; i += kThreads) (&sh.tot[0][0])[i] = 0u;
  for (int i = tid; i < kWarps * 256; i += kThreads) (&sh.whist[0][0])[i] = 0u;
  if (tid == 0) {
    mbar_init(&sh.bar, 1);
    fence_barrier_init();
  }
  pdl_trigger();
  __syncthreads();
  // the totals are zero: peers may add into them once this barrier completes
  cluster_arrive_release();
  // the scores (and every output) belong to the previous kernel until here
  pdl_wait();

  int64_t n_cand = 0;
  if constexpr (kLens) {
    // the cluster splits the pool's longest head, in whole 4-token groups
    // when V = 4
    int Te = 0;
    for (int hh = 0; hh < hps; ++hh) {
      const int L = min(T, max(0, a.lens[head0 + hh]));
      Te = max(Te, L);
      n_cand += L;
      if (tid == 0) lenh[hh] = L;
    }
    const int q = V == 4 ? (Te + 3) >> 2 : Te;
    t0 = V * (int)((int64_t)rank * q / C);
    t1 = V * (int)((int64_t)(rank + 1) * q / C);
  }
  const int nt = t1 - t0;
  const Layout lay(nt, hps, V);
  const int nloc = lay.nloc;
  const int nvec = nloc / V;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + keys_offset<kLens>());
  uint32_t* region = keys + lay.keys_words();

  int64_t need = 0;
  if (a.mode == KVC_SEL_GLOBAL_TOPK) {
    need = a.need_global;
    if (kLens && need > n_cand) need = n_cand;   // every candidate kept
  } else if (a.mode == KVC_SEL_PER_HEAD) {
    int64_t b = a.head_budget[head0];
    if (b < a.nP) b = a.nP;
    if (b > T) b = T;
    need = b - a.nP;
  }
  const bool radix = a.mode != KVC_SEL_THRESHOLD && need > 0;
  uint32_t* wh = sh.whist[warp];

  // ---- phase A: the range's scores into shared memory, keys made in place
  // while the first pass's digits (bits 31-24) are counted
  if (V == 4) {
    if (nt > 0) {
      if (tid == 0) {
        mbar_arrive_expect_tx(&sh.bar, (uint32_t)nloc * 4u);
        for (int hh = 0; hh < hps; ++hh)
          bulk_g2s(smem_u32(keys + hh * nt), a.scores + (int64_t)(head0 + hh) * T + t0,
                   (uint32_t)nt * 4u, &sh.bar);
      }
      mbar_wait(&sh.bar, 0, a.status, nullptr);
    }
    for (int q0 = warp * 32; q0 < nvec; q0 += kThreads) {
      const int q = q0 + lane;
      Vec<V> x;
#pragma unroll
      for (int i = 0; i < V; ++i) x.k[i] = 0u;
      const bool ok = q < nvec;
      if (ok) x.load(keys + (size_t)q * V);
#pragma unroll
      for (int i = 0; i < V; ++i) x.k[i] = score_key(__uint_as_float(x.k[i]));
      if (ok) x.store(keys + (size_t)q * V);
      if (radix) {
#pragma unroll
        for (int i = 0; i < V; ++i) hist_add(wh, ok, x.k[i] >> 24);
      }
    }
  } else {
    for (int hh = 0; hh < hps; ++hh) {
      const float* row = a.scores + (int64_t)(head0 + hh) * T + t0;
      uint32_t* kr = keys + hh * nt;
      for (int j0 = warp * 32; j0 < nt; j0 += kThreads) {
        const int j = j0 + lane;
        const bool ok = j < nt;
        const uint32_t key = ok ? score_key(__ldg(row + j)) : 0u;
        if (ok) kr[j] = key;
        if (radix) hist_add(wh, ok, key >> 24);
      }
    }
  }
  __syncthreads();
  // protected tokens of this range: key 0 (not a candidate), taken back out
  // of the first pass's histogram.  The sink range and the part of the
  // recent window past it are disjoint, so no key is visited twice.
  {
    const int s_hi = min(t1, a.n_sink);                        // sinks [t0, s_hi)
    const int r_lo = max(max(t0, T - a.n_recent), a.n_sink);   // recent [r_lo, t1)
    const int ns = max(0, s_hi - t0), nr = max(0, t1 - r_lo);
    const int np = ns + nr;
    for (int i = tid; i < np * hps; i += kThreads) {
      const int hh = i / np, x = i - hh * np;
      const int t = x < ns ? t0 + x : r_lo + (x - ns);
      uint32_t* kp = keys + hh * nt + (t - t0);
      const uint32_t key = *kp;
      *kp = 0u;
      if (radix) atomicSub(&sh.whist[0][key >> 24], 1u);
    }
  }
  if constexpr (kLens) {
    // positions at or past their head's length: key 0 like a protected
    // token (keep() drops them), taken back out of the first histogram
    for (int hh = 0; hh < hps; ++hh) {
      for (int t = max(t0, lenh[hh]) + tid; t < t1; t += kThreads) {
        uint32_t* kp = keys + hh * nt + (t - t0);
        const uint32_t key = *kp;
        if (key) {
          *kp = 0u;
          if (radix) atomicSub(&sh.whist[0][key >> 24], 1u);
        }
      }
    }
  }
  __syncthreads();
  cluster_wait_acquire();

  // ---- phase B: radix select of the need-th largest candidate key
  uint32_t thr = kNoThr;
  uint32_t ecut = 0;
  if (a.mode == KVC_SEL_THRESHOLD) {
    thr = (a.tau != a.tau) ? kNoThr : score_key(a.tau);
  } else if (need > 0) {
    uint32_t prefix = 0, pmask = 0;
    uint32_t krem = (uint32_t)need;
    uint32_t last_count = 0;
    bool whole_bin = false;
    uint32_t* wl = region + warp * lay.cap_w;   // this warp's candidate list
    int nl = 0;                                 // its length (warp-uniform)
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      if (pass == 1) {
        // keys matching the first digit: histogram the second, append to the list
        for (int q0 = warp * 32; q0 < nvec; q0 += kThreads) {
          const int q = q0 + lane;
          Vec<V> x;
          if (q < nvec) x.load(keys + (size_t)q * V);
          else {
#pragma unroll
            for (int i = 0; i < V; ++i) x.k[i] = 0u;
          }
#pragma unroll
          for (int i = 0; i < V; ++i) {
            const bool cand = x.k[i] != 0u && (x.k[i] & pmask) == prefix;
            const uint32_t cm = hist_add(wh, cand, (x.k[i] >> shift) & 255u);
            if (cand) wl[nl + __popc(cm & lt_mask)] = x.k[i];
            nl += __popc(cm);
          }
        }
      } else if (pass > 1) {
        // the warp's list, compacted in place to the candidates of this pass
        // (a lane writes at or below the slot it read; all reads of a group
        // precede its ballot)
        int nn = 0;
        for (int e0 = 0; e0 < nl; e0 += 32) {
          const int e = e0 + lane;
          const uint32_t key = (e < nl) ? wl[e] : 0u;
          const bool cand = key != 0u && (key & pmask) == prefix;
          const uint32_t cm = hist_add(wh, cand, (key >> shift) & 255u);
          if (cand) wl[nn + __popc(cm & lt_mask)] = key;
          nn += __popc(cm);
        }
        nl = nn;
      }
      __syncthreads();
      // reduce the warp histograms (and clear them for the next pass); every
      // CTA adds its histogram into the bins' owners
      {
        const int b = tid & 255, qq = tid >> 8;
        uint32_t s = 0;
#pragma unroll
        for (int w = 0; w < kWarps / 4; ++w) {
          s += sh.whist[qq * (kWarps / 4) + w][b];
          sh.whist[qq * (kWarps / 4) + w][b] = 0u;
        }
        sh.part[qq][b] = s;
      }
      __syncthreads();
      if (tid < 256) {
        const uint32_t h = sh.part[0][tid] + sh.part[1][tid] + sh.part[2][tid] + sh.part[3][tid];
        if (h) atomicAdd(cl.map_shared_rank(&sh.tot[pass][tid], (tid * C) >> 8), h);
      }
      cl.sync();
      if (tid < 256) sh.totl[tid] = *cl.map_shared_rank(&sh.tot[pass][tid], (tid * C) >> 8);
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
      if (krem == last_count) { whole_bin = true; break; }   // uniform across the cluster
    }
    if (whole_bin) {
      // keep every key >= prefix: key > prefix - 1 with no tie list (prefix 0
      // keeps every candidate; no candidate key is 0)
      thr = prefix ? prefix - 1u : 0u;
      ecut = 0;
    } else {
      thr = prefix;
    }
    // ---- ties: keep the first krem elements with key == thr in (t, g) order
    if (!whole_bin && krem < last_count) {
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
    } else if (!whole_bin) {
      ecut = (uint32_t)nloc;
    }
  }

  const bool thr_mode = a.mode == KVC_SEL_THRESHOLD;
  auto keep = [&](uint32_t key, int j, int hh) -> bool {
    if constexpr (kLens) {
      if (t0 + j >= lenh[hh]) return false;
    }
    return key == 0u || (thr_mode ? key >= thr
                                  : (key > thr || (key == thr && (uint32_t)(j * hps + hh) < ecut)));
  };
  if (a.hand) {
    // ---- hand-off: this range's threshold, tie cut and kept count per head
    // (the placement and the row copies run in emit_compact_kernel)
    const int S = a.hand_sub;
    uint32_t* rec = a.hand + (size_t)rank * (2 + hps * S);
    for (int q = warp; q < hps * S; q += kWarps) {
      const int hh = q / S, sub = q - hh * S;
      const int j1 = min(nt, (sub + 1) * kSubRange);
      uint32_t n = 0;
      for (int j = sub * kSubRange + lane; j < j1; j += 32) n += keep(keys[hh * nt + j], j, hh) ? 1u : 0u;
      n = __reduce_add_sync(0xffffffffu, n);
      if (lane == 0) rec[2 + q] = n;
    }
    if (tid == 0) { rec[0] = thr; rec[1] = ecut; }
    // no CTA may leave while a peer can still read its shared memory
    cl.sync();
    return;
  }

  // ---- phase D: warp w emits the kept tokens of its slice [j_lo, j_hi) of
  // the range, per head, ascending, into its staging segment
  const int per_w = lay.per_w;
  const int j_lo = min(nt, warp * per_w), j_hi = min(nt, j_lo + per_w);
#pragma unroll 2
  for (int hh = 0; hh < hps; ++hh) {
    const uint32_t* __restrict__ kr = keys + hh * nt;                       // keys and staging
    uint32_t* __restrict__ sg = region + (size_t)(hh * kWarps + warp) * per_w;   // never overlap
    uint32_t n = 0;
    for (int j0 = j_lo; j0 < j_hi; j0 += 64) {
      const int ja = j0 + lane, jb = ja + 32;
      const uint32_t ka = ja < j_hi ? kr[ja] : 0u;
      const uint32_t kb = jb < j_hi ? kr[jb] : 0u;
      const bool fa = ja < j_hi && keep(ka, ja, hh);
      const bool fb = jb < j_hi && keep(kb, jb, hh);
      const uint32_t ba = __ballot_sync(0xffffffffu, fa);
      const uint32_t bb = __ballot_sync(0xffffffffu, fb);
      if (fa) sg[n + __popc(ba & lt_mask)] = (uint32_t)(t0 + ja);
      n += __popc(ba);
      if (fb) sg[n + __popc(bb & lt_mask)] = (uint32_t)(t0 + jb);
      n += __popc(bb);
    }
    if (lane == 0) sh.wcnt[hh][warp] = n;
  }
  __syncthreads();
  // per head: exclusive prefix over the warps, CTA total
  if (warp < hps) {
    const uint32_t x = sh.wcnt[warp][lane];
    uint32_t y = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, y, off);
      if (lane >= off) y += n;
    }
    sh.wexcl[warp][lane] = y - x;
    if (lane == 31) sh.xchg_cnt[warp] = y;
  }
  cl.sync();
  if (tid < C * hps) {
    const int r = tid / hps, hh = tid - r * hps;
    sh.xall[r][hh] = cl.map_shared_rank(sh.xchg_cnt, r)[hh];
  }
  __syncthreads();
  // every remote read of this CTA's counts is done once all CTAs pass here
  cluster_arrive_relaxed();
  if (tid < hps) {
    uint32_t base = 0, total = 0;
    for (int r = 0; r < C; ++r) {
      const uint32_t v = sh.xall[r][tid];
      if (r < rank) base += v;
      total += v;
    }
    sh.head_base[tid] = base;
    sh.head_total[tid] = total;
    if (rank == 0) a.counts[head0 + tid] = (int32_t)total;
  }
  __syncthreads();
  // a launch with a single pool writes the offsets itself (no second kernel)
  if (a.offsets && rank == 0 && tid == 0) {
    int64_t o = 0;
    for (int hh = 0; hh < hps; ++hh) { a.offsets[hh] = o; o += sh.head_total[hh]; }
    a.offsets[hps] = o;
  }
  // the staging segments into place (each warp its own, coalesced)
  for (int hh = 0; hh < hps; ++hh) {
    const uint32_t n = sh.wcnt[hh][warp];
    int32_t* dst = a.kept + (int64_t)(head0 + hh) * T + sh.head_base[hh] + sh.wexcl[hh][warp];
    const uint32_t* sg = region + (size_t)(hh * kWarps + warp) * per_w;
    for (uint32_t i = lane; i < n; i += 32) dst[i] = (int32_t)sg[i];
  }
  // no CTA may leave while a peer can still read its shared memory
  cluster_wait_plain();
}

// offsets[i] = sum_{j<i} counts[j], offsets[n] = total (one block).
__global__ void __launch_bounds__(1024)
offsets_kernel(const int32_t* __restrict__ counts, int n, int64_t* __restrict__ offsets) {
  __shared__ int64_t warp_sum[32];
  __shared__ int64_t carry_s;
  pdl_wait();
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

// Second half of kvc_select_compact for a launch with one selection pool:
// CTA (rank * S + sub, hh) takes 512-token sub-range `sub` of the select
// kernel's range `rank` of head hh, decides its tokens again with that
// range's threshold and tie cut, places them after the kept tokens of the
// head's lower ranges and sub-ranges (all counted in the hand-off record),
// writes their indices and copies their K / V rows.  The rule and the
// per-range tie cut are the select kernel's own, so the indices are the ones
// kvc_select writes.
constexpr int kEThreads = 256;
constexpr int kEWarps = kEThreads / 32;
constexpr int kEVec = 8;                 // 16-byte vectors in flight per thread and tensor
static_assert(kSubRange == 2 * kEThreads, "two tokens per thread");
static_assert(kMaxHps <= kEWarps, "a warp per head");

struct EArgs {
  const float* scores;
  int T, hps, C, S, mode, n_sink, n_recent;
  const uint32_t* hand;          // [C][2 + hps * S]
  const uint4* k;
  const uint4* v;
  int vpr_shift, slack;
  uint4* kc;
  uint4* vc;
  int64_t capacity_rows;
  int32_t* kept;
  int32_t* counts;
  int64_t* offsets;
  int64_t* start;
  int32_t* len;
  int* status;
};

__global__ void __launch_bounds__(kEThreads)
emit_compact_kernel(EArgs e) {
  __shared__ uint32_t htot[kMaxHps], base_s, wsum[kEWarps];
  __shared__ int32_t lst_t[kSubRange], lst_p[kSubRange];
  const int T = e.T, hps = e.hps, C = e.C, S = e.S;
  const int rank = blockIdx.x / S, sub = blockIdx.x - rank * S, hh = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = (int)((int64_t)rank * T / C), t1 = (int)((int64_t)(rank + 1) * T / C);
  const int a0 = t0 + sub * kSubRange, a1 = min(t1, a0 + kSubRange);
  const int rs = T - e.n_recent;
  const int stride = 2 + hps * S;
  const float* row = e.scores + (int64_t)hh * T;
  pdl_wait();
  pdl_trigger();
  // two consecutive tokens per thread, in flight while the record is read
  const int tb = a0 + 2 * tid;
  float sv[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) sv[x] = tb + x < a1 ? __ldg(row + tb + x) : 0.0f;
  const uint32_t thr = e.hand[(size_t)rank * stride];
  const uint32_t ecut = e.hand[(size_t)rank * stride + 1];
  if (warp < hps) {
    // warp h: head h's total; for head hh also the part ranked before this
    // CTA (lower ranges, then lower sub-ranges of this range)
    uint32_t tot = 0, below = 0;
    for (int q = lane; q < C * S; q += 32) {
      const int r = q / S, sb = q - r * S;
      const uint32_t x = e.hand[(size_t)r * stride + 2 + warp * S + sb];
      tot += x;
      below += (r < rank || (r == rank && sb < sub)) ? x : 0u;
    }
    tot = __reduce_add_sync(0xffffffffu, tot);
    below = __reduce_add_sync(0xffffffffu, below);
    if (lane == 0) {
      htot[warp] = tot;
      if (warp == hh) base_s = below;
    }
  }
  __syncthreads();
  int64_t off_hh = 0, total = 0;
  for (int h = 0; h < hps; ++h) {
    if (h < hh) off_hh += htot[h];
    total += htot[h];
  }
  if (blockIdx.x == 0 && hh == 0 && tid <= hps) {
    int64_t o = 0;
    for (int h = 0; h < tid; ++h) o += htot[h];
    e.offsets[tid] = o;
    if (tid < hps) {
      e.counts[tid] = (int32_t)htot[tid];
      e.start[tid] = o + (int64_t)tid * e.slack;
      e.len[tid] = (int32_t)htot[tid];
    }
  }
  (void)total;
  const bool thr_mode = e.mode == KVC_SEL_THRESHOLD;
  uint32_t flags = 0u;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const int t = tb + x;
    if (t < a1) {
      const uint32_t key = (t < e.n_sink || t >= rs) ? 0u : score_key(sv[x]);
      const uint32_t jl = (uint32_t)(t - t0);
      const bool kp = key == 0u || (thr_mode ? key >= thr
                                            : (key > thr || (key == thr && jl * hps + hh < ecut)));
      flags |= (kp ? 1u : 0u) << x;
    }
  }
  const uint32_t n = __popc(flags);
  uint32_t incl = n;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  uint32_t before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kEWarps; ++w) {
    const uint32_t v = wsum[w];
    if (w < warp) before += v;
    all += v;
  }
  const uint32_t base = base_s;
  int32_t* out = e.kept + (int64_t)hh * T;
  uint32_t k = before + incl - n;              // this thread's first slot in the list
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    if ((flags >> x) & 1u) {
      const uint32_t pos = base + k;
      lst_t[k] = tb + x;
      lst_p[k] = (int32_t)pos;
      if (pos < (uint32_t)T) out[pos] = tb + x;
      else report(e.status, KVC_ERR_RANGE);
      ++k;
    }
  }
  __syncthreads();
  // the kept rows: K and V, 16-byte vectors, kEVec in flight per tensor
  const int64_t dst0 = off_hh + (int64_t)hh * e.slack;   // head's first compacted row
  const int vpr = 1 << e.vpr_shift;
  const int pairs = (int)all << e.vpr_shift;
  for (int p0 = 0; p0 < pairs; p0 += kEThreads * kEVec) {
    uint4 kv[kEVec], vv[kEVec];
    int64_t dst[kEVec];
#pragma unroll
    for (int x = 0; x < kEVec; ++x) {
      const int p = p0 + x * kEThreads + tid;
      dst[x] = -1;
      if (p < pairs) {
        const int r = p >> e.vpr_shift, vec = p & (vpr - 1);
        const int64_t src = (int64_t)hh * T + lst_t[r];
        const int64_t d = dst0 + lst_p[r];
        if (lst_p[r] < T && d < e.capacity_rows) {
          kv[x] = __ldg(e.k + (src << e.vpr_shift) + vec);
          vv[x] = __ldg(e.v + (src << e.vpr_shift) + vec);
          dst[x] = (d << e.vpr_shift) + vec;
        } else if (vec == 0) {
          report(e.status, KVC_ERR_RANGE);
        }
      }
    }
#pragma unroll
    for (int x = 0; x < kEVec; ++x) {
      if (dst[x] >= 0) {
        e.kc[dst[x]] = kv[x];
        e.vc[dst[x]] = vv[x];
      }
    }
  }
}

size_t shared_bytes(int nt, int hps, int V, bool lens) {
  const Layout lay(nt, hps, V);
  return (lens ? keys_offset<true>() : keys_offset<false>()) +
         (lay.keys_words() + (size_t)lay.region) * 4;
}

}  // namespace

namespace {

// The cluster launch of kvc_select.  With `hand` (one pool only) the kernel
// hands its decision over instead of emitting; *cluster receives the
// cluster size then, or 0 when the pool took the streaming kernel (which
// emits as usual).
int select_launch_ex(const float* scores, int U, int Hkv, int T, int mode, int64_t need_global,
                     float tau, const int32_t* head_budget, int n_sink, int n_recent,
                     int32_t* kept_idx, int32_t* counts, int64_t* offsets, uint32_t* hand,
                     int* cluster, int* sub, const Dev& dev, cudaStream_t s,
                     const int32_t* lens = nullptr) {
  if (cluster) *cluster = 0;
  const int hps = (mode == KVC_SEL_GLOBAL_TOPK) ? Hkv : 1;
  const int nseg = (mode == KVC_SEL_GLOBAL_TOPK) ? U : U * Hkv;
  const int64_t pool = (int64_t)hps * T;
  int nP = 0;
  {
    int rs = T - n_recent;
    nP = n_sink + (T - rs) - (rs < n_sink ? n_sink - rs : 0);
  }
  // pools with more heads than the registers hold, or whose keys and lists
  // do not fit a cluster's shared memory, take the streaming kernel
  // several pools: one more single-block kernel scans the counts into offsets
  auto launch_offsets = [&]() -> int {
    if (nseg == 1) return KVC_OK;
    if (int rc = prefer_max_shared(offsets_kernel, dev.device)) return rc;
    return launch_pdl(offsets_kernel, dim3(1), dim3(1024), 0, s, (const int32_t*)counts,
                      U * Hkv, offsets);
  };
  auto stream = [&]() -> int {
    if (int rc = select_stream_launch(scores, U, Hkv, T, mode, need_global, tau, head_budget,
                                      n_sink, n_recent, nP, kept_idx, counts, offsets,
                                      nseg == 1, dev, s))
      return rc;
    return launch_offsets();
  };
  // per-head lengths need the cluster kernel (the streaming one reads all of T)
  if (lens && (mode != KVC_SEL_GLOBAL_TOPK || n_sink || n_recent || hand)) return KVC_ERR_INVALID;
  if (hps > kMaxHps) return lens ? KVC_ERR_UNSUPPORTED : stream();
  const size_t smem_max = (size_t)dev.max_smem_optin;
  const bool aligned = (reinterpret_cast<uintptr_t>(scores) & 15u) == 0;
  // four keys per thread and step when every CTA's range is a multiple of 4
  auto vec_for = [&](int c) { return (aligned && T % (4 * c) == 0) ? 4 : 1; };
  auto smem_for = [&](int c) {
    return shared_bytes((T + c - 1) / c, hps, vec_for(c), lens != nullptr);
  };
  // the smallest cluster that keeps <= per_cta keys per CTA, else the smallest that fits
  int C = 1;
  // keys per CTA: a threshold pool has no radix passes, so a wider cluster
  // only divides its sweep (four 131 072-key pools in 16-CTA clusters of 8192
  // keys per CTA instead of 8-CTA clusters of 16 K: 14.8 -> 12.7 us); the
  // radix passes of the other modes pay a cluster
  // exchange each, and more, smaller clusters keep more SMs busy (16-CTA
  // clusters for the 32-layer pools: 181 -> 320 us)
  const int64_t per_cta = mode == KVC_SEL_THRESHOLD ? 4096 : 16384;
  while (C < 16 && (pool + C - 1) / C > per_cta) C *= 2;
  while (C < 16 && smem_for(C) > smem_max) C *= 2;
  if (smem_for(C) > smem_max) return lens ? KVC_ERR_UNSUPPORTED : stream();
  Args a;
  a.scores = scores; a.T = T; a.hps = hps; a.mode = mode; a.need_global = need_global;
  a.tau = tau; a.head_budget = head_budget; a.n_sink = n_sink; a.n_recent = n_recent;
  a.nP = nP;
  a.kept = kept_idx; a.counts = counts;
  a.offsets = (nseg == 1) ? offsets : nullptr;
  a.status = dev.status;
  a.hand = (nseg == 1) ? hand : nullptr;
  a.hand_sub = 0;
  a.lens = lens;
  static std::mutex mu;
  static bool attr_done[64];
  static std::map<std::tuple<int, int, size_t>, int> active_memo;
  std::lock_guard<std::mutex> lock(mu);
  if (!attr_done[dev.device & 63]) {
    for (auto fn : {select_kernel<1, false>, select_kernel<4, false>, select_kernel<1, true>,
                    select_kernel<4, true>}) {
      KVC_CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
      KVC_CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        dev.max_smem_optin));
    }
    attr_done[dev.device & 63] = true;
  }
  for (auto fn : {select_kernel<1, false>, select_kernel<4, false>, select_kernel<1, true>,
                  select_kernel<4, true>})
    if (int rc = prefer_max_shared(fn, dev.device)) return rc;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  // a cluster must fit one GPC: shrink it (while the keys still fit) until
  // the occupancy query says at least one cluster can be resident (the
  // answer is remembered per device, cluster size and shared memory)
  for (;;) {
    const size_t smem = smem_for(C);
    cfg.gridDim = dim3((unsigned)C, (unsigned)nseg, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;                 // the occupancy query sees the cluster shape only
    int active = 0;
    const auto key = std::make_tuple(dev.device, C, smem);
    auto it = active_memo.find(key);
    if (it != active_memo.end()) {
      active = it->second;
    } else {
      KVC_CUDA_TRY(cudaOccupancyMaxActiveClusters(&active, select_kernel<1, false>, &cfg));
      active_memo[key] = active;
    }
    if (active > 0) break;
    if (C == 1 || smem_for(C / 2) > smem_max) return lens ? KVC_ERR_UNSUPPORTED : stream();
    C /= 2;
  }
  if (a.hand) {
    // the emission takes 512-token sub-ranges of every CTA's range
    a.hand_sub = (int)(((T + C - 1) / C + kSubRange - 1) / kSubRange);
    if (a.hand_sub > kMaxSub) a.hand = nullptr;
  }
  attr[1] = pdl_attr();
  cfg.numAttrs = 2;
  {
    const bool v4 = vec_for(C) == 4;
    auto kern = lens ? (v4 ? select_kernel<4, true> : select_kernel<1, true>)
                     : (v4 ? select_kernel<4, false> : select_kernel<1, false>);
    KVC_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, a));
  }
  if (a.hand) {
    if (cluster) *cluster = C;
    if (sub) *sub = a.hand_sub;
    return launch_status();
  }
  if (int rc = launch_offsets()) return rc;
  return launch_status();
}

}  // namespace

int select_launch(const float* scores, int U, int Hkv, int T, int mode, int64_t need_global,
                  float tau, const int32_t* head_budget, int n_sink, int n_recent,
                  int32_t* kept_idx, int32_t* counts, int64_t* offsets, const Dev& dev,
                  cudaStream_t s) {
  return select_launch_ex(scores, U, Hkv, T, mode, need_global, tau, head_budget, n_sink,
                          n_recent, kept_idx, counts, offsets, nullptr, nullptr, nullptr, dev,
                          s);
}

int select_lens_launch(const float* keys, int U, int Hkv, int T, const int32_t* lens,
                       int64_t need, int32_t* kept_idx, int32_t* counts, int64_t* offsets,
                       const Dev& dev, cudaStream_t s) {
  return select_launch_ex(keys, U, Hkv, T, KVC_SEL_GLOBAL_TOPK, need, 0.0f, nullptr, 0, 0,
                          kept_idx, counts, offsets, nullptr, nullptr, nullptr, dev, s, lens);
}

size_t select_compact_ws(int U, int Hkv, int T, int mode) {
  const int hps = (mode == KVC_SEL_GLOBAL_TOPK) ? Hkv : 1;
  const int nseg = (mode == KVC_SEL_GLOBAL_TOPK) ? U : U * Hkv;
  if (nseg != 1 || hps > kMaxHps) return 0;
  return (size_t)16 * (2 + hps * kMaxSub) * sizeof(uint32_t);
}

int select_compact_launch(const float* scores, int U, int Hkv, int T, int mode,
                          int64_t need_global, float tau, const int32_t* head_budget, int n_sink,
                          int n_recent, const void* k, const void* v, int row_bytes, int slack,
                          void* kc, void* vc, int64_t capacity_rows, int32_t* kept_idx,
                          int32_t* counts, int64_t* offsets, int64_t* start, int32_t* len,
                          void* ws, size_t ws_bytes, const Dev& dev, cudaStream_t s) {
  const int vpr = row_bytes / 16;
  if (vpr <= 0 || (vpr & (vpr - 1)) || vpr > 32) return KVC_ERR_UNSUPPORTED;
  const size_t need_ws = select_compact_ws(U, Hkv, T, mode);
  uint32_t* hand = (need_ws && ws && ws_bytes >= need_ws) ? static_cast<uint32_t*>(ws) : nullptr;
  int C = 0, S = 0;
  if (int rc = select_launch_ex(scores, U, Hkv, T, mode, need_global, tau, head_budget, n_sink,
                                n_recent, kept_idx, counts, offsets, hand, &C, &S, dev, s))
    return rc;
  if (!hand || C == 0)       // the select emitted: the plain compaction follows
    return compact_launch(k, v, row_bytes, U, Hkv, T, kept_idx, counts, offsets, slack, kc, vc,
                          capacity_rows, start, len, dev, s);
  EArgs e;
  e.scores = scores; e.T = T; e.hps = (mode == KVC_SEL_GLOBAL_TOPK) ? Hkv : 1; e.C = C; e.S = S;
  e.mode = mode; e.n_sink = n_sink; e.n_recent = n_recent; e.hand = hand;
  e.k = static_cast<const uint4*>(k); e.v = static_cast<const uint4*>(v);
  int sh = 0;
  while ((16 << sh) < row_bytes) ++sh;
  e.vpr_shift = sh; e.slack = slack;
  e.kc = static_cast<uint4*>(kc); e.vc = static_cast<uint4*>(vc);
  e.capacity_rows = capacity_rows;
  e.kept = kept_idx; e.counts = counts; e.offsets = offsets; e.start = start; e.len = len;
  e.status = dev.status;
  return launch_pdl(emit_compact_kernel, dim3((unsigned)(C * S), (unsigned)e.hps),
                    dim3(kEThreads), 0, s, e);
}

}  // namespace kvc
