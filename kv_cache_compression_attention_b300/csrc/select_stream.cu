// Budget selection for pools whose keys do not fit one cluster's shared
// memory, or that pool more than 8 heads (for instance every layer and kv
// head of a sequence in one global budget, after KVSculpt §2D's adaptive
// layer-and-head allocation).
//
// Same rules and result as the shared-memory kernel of select.cu (global
// top-k across the pool's heads, per-head top-k or threshold; protected
// sinks and recent window; ties in (token asc, head asc) order), with every
// sweep reading the scores again from global memory (the pool's scores are
// read from L2 after the first sweep) instead of keeping keys and candidate
// lists on chip:
//  * one thread-block cluster of C CTAs per pool, CTA r owning tokens
//    [r*T/C, (r+1)*T/C) of every head of the pool;
//  * radix select, 4 passes of 8-bit digits, each a sweep with warp-private
//    shared-memory histograms, added into the bins' owner CTAs with
//    distributed-shared-memory atomics; early stop when the chosen bin is
//    kept whole;
//  * ties ranked by a cluster prefix of per-CTA tie counts and a block scan
//    over tokens;
//  * emission in two sweeps: per-(head, warp) kept counts, a scan over the
//    warps and a cluster prefix per head, then every warp writes its slice's
//    kept tokens, ascending, straight to their places.
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
constexpr int kMaxHeads = 512;             // heads per pool
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
  int* status;
};

struct Shared {
  uint32_t whist[kWarps][256];        // per-warp histograms of the current pass
  uint32_t part[4][256];
  uint32_t tot[4][256];               // per pass: totals of the bins this CTA owns
  uint32_t totl[256];
  uint32_t warp_tmp[2][kWarps];
  uint32_t warp_tot[2];
  uint32_t xchg_ties;                 // read remotely
  uint32_t sel_bin, sel_above, sel_count, ecut, tie_base;
};

// Per-head arrays after Shared: wcnt[hps][32] (kept per head and warp, then
// its exclusive prefix over the warps), xcnt[hps] (this CTA's count per head,
// read remotely), hbase[hps] (this CTA's first slot per head), htot[hps].
size_t stream_smem_bytes(int hps) {
  return ((sizeof(Shared) + 15) & ~size_t(15)) + (size_t)hps * (kWarps + 3) * 4;
}

__device__ __forceinline__ bool prot(int t, int T, int n_sink, int n_recent) {
  return t < n_sink || t >= T - n_recent;
}

__device__ __forceinline__ uint32_t hist_add(uint32_t* wh, bool cand, uint32_t digit) {
  const uint32_t cm = __ballot_sync(0xffffffffu, cand);
  if (cand) atomicAdd(&wh[digit], 1u);
  return cm;
}

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

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_plain() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
select_stream_kernel(Args a) {
  cg::cluster_group cl = cg::this_cluster();
  const int C = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const int hps = a.hps;
  const int T = a.T;
  const int head0 = blockIdx.y * hps;
  const int t0 = (int)((int64_t)rank * T / C);
  const int t1 = (int)((int64_t)(rank + 1) * T / C);
  const int nt = t1 - t0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  int sbuf = 0;

  extern __shared__ __align__(16) uint8_t smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  uint32_t* wcnt = reinterpret_cast<uint32_t*>(smem_raw + ((sizeof(Shared) + 15) & ~size_t(15)));
  uint32_t* xcnt = wcnt + (size_t)hps * kWarps;
  uint32_t* hbase = xcnt + hps;
  uint32_t* htot = hbase + hps;

  for (int i = tid; i < 4 * 256; i += kThreads) (&sh.tot[0][0])[i] = 0u;
  for (int i = tid; i < kWarps * 256; i += kThreads) (&sh.whist[0][0])[i] = 0u;
  pdl_trigger();
  __syncthreads();
  cl.sync();                            // every CTA's totals are zero before any remote add
  pdl_wait();

  int64_t need = 0;
  if (a.mode == KVC_SEL_GLOBAL_TOPK) {
    need = a.need_global;
  } else if (a.mode == KVC_SEL_PER_HEAD) {
    int64_t b = a.head_budget[head0];
    if (b < a.nP) b = a.nP;
    if (b > T) b = T;
    need = b - a.nP;
  }
  uint32_t* wh = sh.whist[warp];
  const float* base = a.scores + (int64_t)head0 * T + t0;

  // key of (head hh, local token j) from its score: 0 for a protected token
  auto key_of = [&](float x, int j) -> uint32_t {
    return prot(t0 + j, T, a.n_sink, a.n_recent) ? 0u : score_key(x);
  };
  auto key_at = [&](int hh, int j) -> uint32_t {
    return key_of(__ldg(base + (int64_t)hh * T + j), j);
  };
  // sweep over every (head, token) of the range, 32 consecutive tokens of
  // one head per warp group (coalesced), kU groups' loads in flight per
  // lane; f(hh, j, valid, key) is called by every lane of the warp
  auto sweep = [&](auto&& f) {
    constexpr int kU = 8;
    const int per_head = (nt + 31) >> 5;               // 32-token groups per head
    const int groups = per_head * hps;
    for (int q0 = warp; q0 < groups; q0 += kWarps * kU) {
      float x[kU];
      int hv[kU], jv[kU];
      bool ok[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int q = q0 + u * kWarps;
        hv[u] = q / per_head;
        jv[u] = (q - hv[u] * per_head) * 32 + lane;
        ok[u] = q < groups && jv[u] < nt;
        x[u] = ok[u] ? __ldg(base + (int64_t)hv[u] * T + jv[u]) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) f(hv[u], jv[u], ok[u], ok[u] ? key_of(x[u], jv[u]) : 0u);
    }
  };

  // ---- radix select of the need-th largest candidate key
  uint32_t thr = kNoThr;
  uint32_t ecut = 0;
  if (a.mode == KVC_SEL_THRESHOLD) {
    thr = (a.tau != a.tau) ? kNoThr : score_key(a.tau);
  } else if (need > 0) {
    uint32_t prefix = 0, pmask = 0;
    uint32_t krem = (uint32_t)need;
    uint32_t last_count = 0;
    bool whole_bin = false;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      sweep([&](int, int, bool, uint32_t key) {
        const bool cand = key != 0u && (key & pmask) == prefix;
        hist_add(wh, cand, (key >> shift) & 255u);
      });
      __syncthreads();
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
        uint32_t suffix = lsum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          uint32_t n = __shfl_down_sync(0xffffffffu, suffix, off);
          if (lane + off < 32) suffix += n;
        }
        uint32_t above = suffix - lsum;
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
      thr = prefix ? prefix - 1u : 0u;
      ecut = 0;
    } else {
      thr = prefix;
    }
    // ---- ties: keep the first krem elements with key == thr in (t, g) order
    if (!whole_bin && krem < last_count) {
      uint32_t mine = 0;
      sweep([&](int, int, bool ok, uint32_t key) { mine += (ok && key == thr); });
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
      const uint32_t tb = sh.tie_base;
      const uint32_t local_ties = sh.xchg_ties;
      if (tb >= krem) ecut = 0;
      else if (tb + local_ties <= krem) ecut = (uint32_t)nt * hps;
      else {
        const uint32_t want = krem - tb;       // 1 <= want < local_ties
        uint32_t carry = 0;
        for (int j0 = 0; j0 < nt; j0 += kThreads) {
          const int j = j0 + tid;
          uint32_t c = 0;
          if (j < nt)
            for (int hh = 0; hh < hps; ++hh) c += (key_at(hh, j) == thr);
          uint32_t total;
          const uint32_t excl = carry + block_scan(c, sh, sbuf, &total);
          if (c && excl <= want && want < excl + c) {
            uint32_t k = want - excl;
            int hh = 0;
            for (; hh < hps; ++hh)
              if (key_at(hh, j) == thr) { if (k == 0) break; --k; }
            sh.ecut = (uint32_t)(j * hps + hh);
          }
          carry += total;
          if (carry > want) break;             // uniform across the block
        }
        __syncthreads();
        ecut = sh.ecut;
      }
    } else if (!whole_bin) {
      ecut = (uint32_t)nt * hps;
    }
  }

  // ---- emission, sweep 1: kept tokens per (head, warp) of warp slices
  const bool thr_mode = a.mode == KVC_SEL_THRESHOLD;
  auto keep = [&](uint32_t key, int j, int hh) -> bool {
    return key == 0u || (thr_mode ? key >= thr
                                  : (key > thr || (key == thr && (uint32_t)(j * hps + hh) < ecut)));
  };
  const int per_w = (nt + kWarps - 1) / kWarps;
  const int j_lo = min(nt, warp * per_w), j_hi = min(nt, j_lo + per_w);
  // (eight heads per step, so that eight loads per lane are in flight)
  constexpr int kH = 8;
  for (int hh0 = 0; hh0 < hps; hh0 += kH) {
    uint32_t n[kH];
#pragma unroll
    for (int x = 0; x < kH; ++x) n[x] = 0u;
    for (int j0 = j_lo; j0 < j_hi; j0 += 32) {
      const int j = j0 + lane;
      float v[kH];
#pragma unroll
      for (int x = 0; x < kH; ++x)
        v[x] = (hh0 + x < hps && j < j_hi) ? __ldg(base + (int64_t)(hh0 + x) * T + j) : 0.0f;
#pragma unroll
      for (int x = 0; x < kH; ++x) {
        const bool f = hh0 + x < hps && j < j_hi && keep(key_of(v[x], j), j, hh0 + x);
        n[x] += __popc(__ballot_sync(0xffffffffu, f));
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int x = 0; x < kH; ++x)
        if (hh0 + x < hps) wcnt[(hh0 + x) * kWarps + warp] = n[x];
    }
  }
  __syncthreads();
  // per head: exclusive prefix over the warps (in place), CTA total
  for (int hh = warp; hh < hps; hh += kWarps) {
    const uint32_t x = wcnt[hh * kWarps + lane];
    uint32_t y = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, y, off);
      if (lane >= off) y += n;
    }
    wcnt[hh * kWarps + lane] = y - x;
    if (lane == 31) xcnt[hh] = y;
  }
  cl.sync();
  for (int hh = tid; hh < hps; hh += kThreads) {
    uint32_t b = 0, total = 0;
    for (int r = 0; r < C; ++r) {
      const uint32_t v = cl.map_shared_rank(xcnt, r)[hh];
      if (r < rank) b += v;
      total += v;
    }
    hbase[hh] = b;
    htot[hh] = total;
  }
  __syncthreads();
  // every remote read of this CTA's counts is done once all CTAs pass here
  cluster_arrive_relaxed();
  if (rank == 0) {
    for (int hh = tid; hh < hps; hh += kThreads) a.counts[head0 + hh] = (int32_t)htot[hh];
    if (a.offsets && tid == 0) {
      int64_t o = 0;
      for (int hh = 0; hh < hps; ++hh) { a.offsets[hh] = o; o += htot[hh]; }
      a.offsets[hps] = o;
    }
  }
  // ---- emission, sweep 2: every warp writes its slice's kept tokens
  for (int hh0 = 0; hh0 < hps; hh0 += kH) {
    uint32_t n[kH];
#pragma unroll
    for (int x = 0; x < kH; ++x) n[x] = 0u;
    for (int j0 = j_lo; j0 < j_hi; j0 += 32) {
      const int j = j0 + lane;
      float v[kH];
#pragma unroll
      for (int x = 0; x < kH; ++x)
        v[x] = (hh0 + x < hps && j < j_hi) ? __ldg(base + (int64_t)(hh0 + x) * T + j) : 0.0f;
#pragma unroll
      for (int x = 0; x < kH; ++x) {
        const int hh = hh0 + x;
        const bool f = hh < hps && j < j_hi && keep(key_of(v[x], j), j, hh);
        const uint32_t bm = __ballot_sync(0xffffffffu, f);
        if (f)
          a.kept[(int64_t)(head0 + hh) * T + hbase[hh] + wcnt[hh * kWarps + warp] + n[x] +
                 __popc(bm & lt_mask)] = t0 + j;
        n[x] += __popc(bm);
      }
    }
  }
  // no CTA may leave while a peer can still read its shared memory
  cluster_wait_plain();
}

}  // namespace

int select_stream_launch(const float* scores, int U, int Hkv, int T, int mode,
                         int64_t need_global, float tau, const int32_t* head_budget, int n_sink,
                         int n_recent, int nP, int32_t* kept_idx, int32_t* counts,
                         int64_t* offsets, bool offsets_in_kernel, const Dev& dev,
                         cudaStream_t s) {
  const int hps = (mode == KVC_SEL_GLOBAL_TOPK) ? Hkv : 1;
  if (hps > kMaxHeads) return KVC_ERR_UNSUPPORTED;
  const int nseg = (mode == KVC_SEL_GLOBAL_TOPK) ? U : U * Hkv;
  const size_t smem = stream_smem_bytes(hps);
  if (smem > (size_t)dev.max_smem_optin) return KVC_ERR_UNSUPPORTED;
  Args a;
  a.scores = scores; a.T = T; a.hps = hps; a.mode = mode; a.need_global = need_global;
  a.tau = tau; a.head_budget = head_budget; a.n_sink = n_sink; a.n_recent = n_recent;
  a.nP = nP; a.kept = kept_idx; a.counts = counts;
  a.offsets = offsets_in_kernel ? offsets : nullptr;
  a.status = dev.status;
  static std::mutex mu;
  static bool attr_done[64];
  static std::map<std::tuple<int, int, size_t>, int> active_memo;
  std::lock_guard<std::mutex> lock(mu);
  if (!attr_done[dev.device & 63]) {
    KVC_CUDA_TRY(cudaFuncSetAttribute(select_stream_kernel,
                                      cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
    KVC_CUDA_TRY(cudaFuncSetAttribute(select_stream_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      dev.max_smem_optin));
    attr_done[dev.device & 63] = true;
  }
  if (int rc = prefer_max_shared(select_stream_kernel, dev.device)) return rc;
  // the widest cluster (at most 16, at most one CTA per token) that can be resident
  int C = 16;
  while (C > 1 && C > T) C >>= 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  for (;;) {
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
      KVC_CUDA_TRY(cudaOccupancyMaxActiveClusters(&active, select_stream_kernel, &cfg));
      active_memo[key] = active;
    }
    if (active > 0) break;
    if (C == 1) return KVC_ERR_UNSUPPORTED;
    C >>= 1;
  }
  attr[1] = pdl_attr();
  cfg.numAttrs = 2;
  KVC_CUDA_TRY(cudaLaunchKernelEx(&cfg, select_stream_kernel, a));
  return launch_status();
}

}  // namespace kvc
