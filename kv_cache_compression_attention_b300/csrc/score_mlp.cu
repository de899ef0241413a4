// Two-layer surrogate scorer (KVzap: Fast, Adaptive, and Faithful KV Cache
// Pruning, §2.2, the MLP variant: hidden width Dm = Dh / 8 with a GELU):
//   z[r, m]      = b1[m] + hidden[r, :] . W1[:, m]        (r = u * T + t)
//   score[u,g,t] = b2[g] + sum_m GELU(z[r, m]) W2[m, g]
//
// The first layer is a dense GEMM (131072 x 3584 x 448 on the 128k layer,
// 421 GFLOP, 448 FLOP per byte of hidden state: bound by the tensor pipe,
// not by HBM), so it runs on tcgen05 with the accumulator in TMEM, and the
// bias, exact GELU and second layer are its epilogue: the intermediate z
// never leaves the SM.
//
//   prologue  W1 [Dh, Dm] is transposed once per call into the workspace as
//             W1t [Dmp, Dh] (rows m >= Dm zero, Dmp = Dm rounded up to 32),
//             so that both MMA operands are K-major 128-byte-swizzled TMA
//             tiles.
//   main      persistent grid, one CTA per SM, 128-row tiles of hidden
//             states.  Per 64-wide k-block a stage holds the tile's hidden
//             rows (A, 128 x 64) and the W1t slab of the pass (B, Np x 64);
//             one or two MMAs of N = Np or Np / 2 per 16-wide k step
//             accumulate z for all Np columns of the pass in TMEM (448 of the
//             512 columns on the 128k layer).  Dm > 512 runs in two passes of
//             Np = Dmp / 2 columns, each streaming the tile's hidden rows.
//   epilogue  16 warps (warp w reads TMEM lanes 32*(w%4)..+31, w/4 picks a
//             quarter of the pass's columns) drain their accumulator slice
//             into registers as bf16 pairs and free TMEM at once, so the
//             next tile's MMAs overlap the GELU work; each thread then adds
//             b1, applies GELU(z) = z (1 + erf(z / sqrt 2)) / 2 (erf by
//             Abramowitz & Stegun 7.1.26, absolute error <= 1.5e-7) and
//             accumulates the Hkv dot products with W2 (read through L1);
//             the four quarters of a row are added in a fixed order through
//             shared memory, b2 is added, and the row's Hkv scores stored.
//
// Warp roles (576 threads): warps 0-15 epilogue, warp 16 TMA producer,
// warp 17 MMA issuer and TMEM owner.  Every wait is bounded (2 s): on expiry
// the status word records KVC_ERR_TIMEOUT and the kernel runs to its end.
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_ptx.cuh"

namespace kvc {
namespace {

constexpr int kTileRows = 128;
constexpr int kKBlock = 64;                 // k elements per stage (128-byte rows)
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = kEpiThreads + 64;
constexpr int kProducerWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxPassCols = 512;
constexpr int kMaxDm = 1024;
constexpr int kMaxGroups = 8;               // 16-column groups per epilogue thread and pass
constexpr uint32_t kABytes = kTileRows * kKBlock * 2;   // 16 KiB
constexpr int kMaxSmem = 232448;            // opt-in shared memory per block on sm_100

struct Params {
  int64_t rows;      // U * T
  int T, Dh, Dm, Hkv;
  int n_kb;          // k-blocks of 64
  int n_tiles;       // 128-row tiles
  int n_pass;        // 1 or 2
  int np;            // columns per pass (multiple of 32, <= 512)
  int bn;            // columns per MMA (np or np / 2, <= 256)
  int bw;            // rows per W1t box (a CTA's share of the slab, <= 256)
  int stages;
  const float* b1;
  const uint16_t* w2;   // bf16 [Dm, Hkv]
  const float* b2;
  float* scores;
  int* status;
};

struct SmemHead {
  uint64_t full[8], empty[8];
  uint64_t tmem_full, tmem_empty;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ uint32_t align1024(uint32_t a) { return (a + 1023u) & ~1023u; }

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2-D TMA tile load with an L2 cache-eviction hint.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int x,
                                                 int y, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// The same load delivered to every CTA of the cluster in `mask` (same
// shared-memory offset and mbarrier offset in each).
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* map, int x, int y,
                                               uint64_t* bar, uint16_t mask, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".multicast::cluster.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5, %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "h"(mask),
      "l"(policy)
      : "memory");
}

// Arrive on the mbarrier at the same offset in every CTA of `mask` once the
// tcgen05 operations issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)), "h"(mask)
      : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (warp-collective,
// completed by the caller's tcgen05.wait::ld).
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait16(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// Two fp32 -> one word of two bf16 (round to nearest even), low half first.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// erf by Abramowitz & Stegun, Handbook of Mathematical Functions, formula
// 7.1.26: erf(x) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-x^2),
// t = 1 / (1 + p x) for x >= 0, odd in x; absolute error at most 1.5e-7.
__device__ __forceinline__ float erf_as(float x) {
  const float ax = fabsf(x);
  float t;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(fmaf(0.3275911f, ax, 1.0f)));
  float q = fmaf(t, 1.061405429f, -1.453152027f);
  q = fmaf(t, q, 1.421413741f);
  q = fmaf(t, q, -0.284496736f);
  q = fmaf(t, q, 0.254829592f);
  const float e = tc::ex2(-ax * ax * 1.4426950408889634f);   // exp(-x^2)
  return copysignf(fmaf(-t * q, e, 1.0f), x);
}

// GELU(z) = z Phi(z) = z (1 + erf(z / sqrt 2)) / 2
__device__ __forceinline__ float gelu_exact(float z) {
  return 0.5f * z * (1.0f + erf_as(z * 0.70710678118654752f));
}

// W1 [Dh, Dm] -> W1t [Dmp, Dh] (rows m >= Dm are zero): 32 x 32 tiles
// through shared memory, so both the read and the write are coalesced.
__global__ void __launch_bounds__(256)
w1_transpose_kernel(const uint16_t* __restrict__ w1, int Dh, int Dm, int Dmp,
                    uint16_t* __restrict__ w1t) {
  __shared__ uint16_t tile[32][33];
  const int j0 = blockIdx.x * 32, m0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
  pdl_wait();
  for (int y = ty; y < 32; y += 8) {
    const int j = j0 + y, m = m0 + tx;
    tile[y][tx] = (j < Dh && m < Dm) ? w1[(int64_t)j * Dm + m] : (uint16_t)0;
  }
  __syncthreads();
  pdl_trigger();
  for (int y = ty; y < 32; y += 8) {
    const int m = m0 + y, j = j0 + tx;
    if (m < Dmp && j < Dh) w1t[(int64_t)m * Dh + j] = tile[tx][y];
  }
}

template <int HK>
__global__ void __launch_bounds__(kThreads, 1)
mlp_tc_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
              Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  SmemHead& sm = *reinterpret_cast<SmemHead*>(smem_raw);
  // quarter sums of the rows of quarters 1-3, [3][128][HK]
  float* red = reinterpret_cast<float*>(smem_raw + sizeof(SmemHead));
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t st0 = align1024(raw + (uint32_t)(sizeof(SmemHead) + 3 * 128 * HK * 4));
  const uint32_t b_bytes = (uint32_t)p.np * kKBlock * 2;
  const uint32_t stage_bytes = kABytes + b_bytes;
  const int S = p.stages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // cluster of cl CTAs (1 or 2): each CTA streams its own hidden rows and 1/cl
  // of every W1t slab, delivered to all of them; a slab is refilled only when
  // every CTA of the cluster has finished with it
  const int cl = (int)tc::cluster_nctarank();
  const int rank = (int)tc::cluster_ctarank();
  const uint16_t cmask = (uint16_t)((1u << cl) - 1u);
  const int n_groups = (p.n_tiles + cl - 1) / cl;
  const int group0 = blockIdx.x / cl, group_step = gridDim.x / cl;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) { mbar_init(&sm.full[s], 1); mbar_init(&sm.empty[s], cl); }
    mbar_init(&sm.tmem_full, 1);
    mbar_init(&sm.tmem_empty, kEpiWarps);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tc::tmem_alloc(&sm.tmem_base, kTmemCols);
  __syncthreads();
  // the peers' barriers are initialised before any multicast reaches them
  tc::cluster_arrive();
  tc::cluster_wait();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;
  // W1t is written by the transpose kernel just before this one
  pdl_wait();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_h);
      tc::prefetch_tmap(&tm_w);
      const uint64_t pol_h = policy_evict_first(), pol_w = policy_evict_last();
      // this CTA's share of a slab: rows [rank * rpc, (rank + 1) * rpc) in boxes of bw
      const int rpc = p.np / cl, bw = p.bw;
      int J = 0;
      for (int grp = group0; grp < n_groups; grp += group_step) {
        const int tile = grp * cl + rank;      // past the last tile: zero rows, not stored
        for (int ps = 0; ps < p.n_pass; ++ps)
          for (int kb = 0; kb < p.n_kb; ++kb, ++J) {
            const int s = J % S;
            if (J >= S) mbar_wait(&sm.empty[s], ((J / S) - 1) & 1, p.status, abort_flag);
            const uint32_t dst = st0 + (uint32_t)s * stage_bytes;
            mbar_arrive_expect_tx(&sm.full[s], stage_bytes);
            tma_load_2d_hint(dst, &tm_h, kb * kKBlock, tile * kTileRows, &sm.full[s], pol_h);
            for (int r0 = rank * rpc; r0 < (rank + 1) * rpc; r0 += bw) {
              const uint32_t bdst = dst + kABytes + (uint32_t)r0 * 128u;
              if (cl > 1)
                tma_load_2d_mc(bdst, &tm_w, kb * kKBlock, ps * p.np + r0, &sm.full[s], cmask,
                               pol_w);
              else
                tma_load_2d_hint(bdst, &tm_w, kb * kKBlock, ps * p.np + r0, &sm.full[s], pol_w);
            }
          }
      }
      // every load into this CTA has landed and every CTA of the cluster has
      // released the last use of every stage before the CTA can exit
      // (normally all of this is long done; after a timeout it may not be)
      for (int j = (J > S ? J - S : 0); j < J; ++j) {
        mbar_wait(&sm.full[j % S], (j / S) & 1, p.status, nullptr);
        mbar_wait(&sm.empty[j % S], (j / S) & 1, p.status, nullptr);
      }
    }
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(kTileRows, p.bn);
      const int nb = p.np / p.bn;
      // the second MMA's B rows start bn rows after the first's
      const uint64_t bstep = (uint64_t)((uint32_t)p.bn * 128u >> 4);
      int J = 0, item = 0;
      for (int grp = group0; grp < n_groups; grp += group_step)
        for (int ps = 0; ps < p.n_pass; ++ps, ++item) {
          // the epilogue has drained the previous item's accumulator
          if (item > 0) mbar_wait(&sm.tmem_empty, (item - 1) & 1, p.status, abort_flag);
          tc::fence_after_sync();
          for (int kb = 0; kb < p.n_kb; ++kb, ++J) {
            const int s = J % S;
            mbar_wait(&sm.full[s], (J / S) & 1, p.status, abort_flag);
            tc::fence_after_sync();
            // descriptors of the stage's operands; a k step moves both by 32
            // bytes (2 in the descriptor's address field, which cannot carry:
            // shared memory ends below 256 KiB)
            const uint32_t a0 = st0 + (uint32_t)s * stage_bytes;
            const uint64_t ad0 = tc::smem_desc_sw128(a0);
            const uint64_t bd0 = tc::smem_desc_sw128(a0 + kABytes);
            const uint64_t bd1 = bd0 + bstep;
            const uint32_t acc0 = kb != 0;
#pragma unroll
            for (int kk = 0; kk < kKBlock / 16; ++kk) {
              const uint32_t acc = kk != 0 ? 1u : acc0;
              tc::mma_bf16(tmem, ad0 + 2u * kk, bd0 + 2u * kk, idesc, acc);
              if (nb == 2)
                tc::mma_bf16(tmem + (uint32_t)p.bn, ad0 + 2u * kk, bd1 + 2u * kk, idesc, acc);
            }
            if (cl > 1) mma_commit_mc(&sm.empty[s], cmask);
            else tc::mma_commit(&sm.empty[s]);
          }
          tc::mma_commit(&sm.tmem_full);
        }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q4 = warp & 3, wq = warp >> 2;            // lane quadrant, column quarter
    const int r_in = 32 * q4 + lane;                    // row of the tile
    const uint32_t lane_addr = (uint32_t)(32 * q4) << 16;
    const int cs = ((p.np + 63) / 64) * 16;             // columns per quarter (<= 128)
    const int c_lo = wq * cs, c_hi = min(p.np, c_lo + cs);
    const int ng = c_hi > c_lo ? (c_hi - c_lo) / 16 : 0;
    int item = 0;
    for (int grp = group0; grp < n_groups; grp += group_step) {
      const int tile = grp * cl + rank;
      float acc[HK];
#pragma unroll
      for (int g = 0; g < HK; ++g) acc[g] = 0.0f;
      for (int ps = 0; ps < p.n_pass; ++ps, ++item) {
        mbar_wait(&sm.tmem_full, item & 1, p.status, abort_flag);
        tc::fence_after_sync();
        // drain this thread's slice of z into registers (bf16 pairs)
        uint32_t zp[kMaxGroups * 8];
#pragma unroll
        for (int gi = 0; gi < kMaxGroups; ++gi) {
          if (gi < ng) {
            uint32_t r[16];
            tmem_ld16_async(tmem + lane_addr + (uint32_t)(c_lo + 16 * gi), r);
            tmem_wait16(r);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              zp[gi * 8 + e] = pack_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.tmem_empty);
        // bias, GELU and the second layer on this thread's columns
        const int m0 = ps * p.np + c_lo;
#pragma unroll
        for (int gi = 0; gi < kMaxGroups; ++gi) {
          if (gi < ng) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int m = m0 + 16 * gi + e;
              if (m < p.Dm) {
                const uint32_t w = zp[gi * 8 + (e >> 1)];
                float z = (e & 1) ? bf16hi(w) : bf16lo(w);
                if (p.b1) z += __ldg(p.b1 + m);
                const float a = gelu_exact(z);
                const uint16_t* w2r = p.w2 + (int64_t)m * HK;
#pragma unroll
                for (int g = 0; g < HK; ++g) acc[g] = fmaf(a, bf16lo(__ldg(w2r + g)), acc[g]);
              }
            }
          }
        }
      }
      // the four quarters of each row, added in a fixed order
      if (wq > 0) {
#pragma unroll
        for (int g = 0; g < HK; ++g) red[((wq - 1) * 128 + r_in) * HK + g] = acc[g];
      }
      tc::named_sync(1, kEpiThreads);
      if (wq == 0) {
        const int64_t row = (int64_t)tile * kTileRows + r_in;
        if (row < p.rows) {
          const int64_t u = row / p.T, t = row - u * p.T;
#pragma unroll
          for (int g = 0; g < HK; ++g) {
            float v = acc[g];
            for (int x = 0; x < 3; ++x) v += red[(x * 128 + r_in) * HK + g];
            if (p.b2) v += __ldg(p.b2 + g);
            p.scores[(u * HK + g) * (int64_t)p.T + t] = v;
          }
        }
      }
      tc::named_sync(1, kEpiThreads);
    }
  }
  __syncthreads();
  // no CTA leaves while a peer may still deliver into its shared memory
  tc::cluster_arrive();
  tc::cluster_wait();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? KVC_OK : KVC_ERR_CUDA;
}

int padded_dm(int Dm) { return (Dm + 31) / 32 * 32; }

// Passes over the hidden states and W1t columns per pass for a given Dm.
void pass_split(int Dm, int* n_pass, int* np) {
  const int Dmp = padded_dm(Dm);
  *n_pass = Dmp <= kMaxPassCols ? 1 : 2;
  *np = *n_pass == 1 ? Dmp : (Dmp / 2 + 31) / 32 * 32;
}

size_t head_bytes(int Hkv) { return sizeof(SmemHead) + 3 * 128 * (size_t)Hkv * 4 + 1024; }

// CTAs per cluster.  The kernel can run as pairs that share every W1t slab
// (each CTA loads half of it and multicasts it to both), which halves the L2
// reads of the first-layer weight; on the 128k layer that measured 406 us
// against 392 us for single CTAs (ncu: L2 29 %, DRAM 32 %, tensor pipe 48 %),
// so single CTAs are launched.  Neither L2 bandwidth nor the DRAM latency of
// the hidden rows holds the kernel: fetching each stage's hidden rows into L2
// eight k-blocks ahead of their load made it slower (324 against 314 us).
int cluster_size(int n_tiles, int sms) {
  (void)n_tiles;
  (void)sms;
  return 1;
}

template <int HK>
int launch_tc(const CUtensorMap& tm_h, const CUtensorMap& tm_w, const Params& p, size_t smem,
              const Dev& dev, cudaStream_t s) {
  static std::mutex mu;
  static bool attr_done[64] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_done[dev.device & 63]) {
      KVC_CUDA_TRY(cudaFuncSetAttribute(mlp_tc_kernel<HK>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem));
      attr_done[dev.device & 63] = true;
    }
  }
  if (int rc = prefer_max_shared(mlp_tc_kernel<HK>, dev.device)) return rc;
  const int cl = cluster_size(p.n_tiles, dev.sms);
  const int groups = (p.n_tiles + cl - 1) / cl;
  const int grid = cl * (groups < dev.sms / cl ? groups : dev.sms / cl);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0] = pdl_attr();
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cl;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  KVC_CUDA_TRY(cudaLaunchKernelEx(&cfg, mlp_tc_kernel<HK>, tm_h, tm_w, p));
  return KVC_OK;
}

}  // namespace

size_t score_mlp_ws_bytes(int Dh, int Dm) {
  int n_pass, np;
  pass_split(Dm, &n_pass, &np);
  return (((size_t)n_pass * np * Dh * 2) + 255) & ~(size_t)255;
}

int score_mlp_launch(const void* hidden, const void* w1, const float* b1, const void* w2,
                     const float* b2, int U, int T, int Dh, int Dm, int Hkv, float* scores,
                     void* workspace, const Dev& dev, cudaStream_t s) {
  const int64_t rows = (int64_t)U * T;
  if (rows == 0) return KVC_OK;
  if (Dm > kMaxDm || Hkv < 1 || Hkv > 8) return KVC_ERR_UNSUPPORTED;
  if (rows > 0x7fffffffLL) return KVC_ERR_UNSUPPORTED;
  if (int rc = get_encoder()) return rc;
  Params p;
  p.rows = rows; p.T = T; p.Dh = Dh; p.Dm = Dm; p.Hkv = Hkv;
  p.n_kb = (Dh + kKBlock - 1) / kKBlock;
  p.n_tiles = (int)((rows + kTileRows - 1) / kTileRows);
  pass_split(Dm, &p.n_pass, &p.np);
  p.bn = p.np <= 256 ? p.np : p.np / 2;
  {
    const int rpc = p.np / cluster_size(p.n_tiles, dev.sms);   // a CTA's rows of a slab
    p.bw = rpc <= 256 ? rpc : rpc / 2;
  }
  p.b1 = b1;
  p.w2 = static_cast<const uint16_t*>(w2);
  p.b2 = b2;
  p.scores = scores;
  p.status = dev.status;
  // as many stages as shared memory holds (at least 2, at most 8)
  const size_t stage = (size_t)kABytes + (size_t)p.np * kKBlock * 2;
  const size_t head = head_bytes(Hkv);
  int stages = (int)((kMaxSmem - head) / stage);
  if (stages > 8) stages = 8;
  if (stages < 2 || kMaxSmem > dev.max_smem_optin) return KVC_ERR_UNSUPPORTED;
  p.stages = stages;
  const size_t smem = head + (size_t)stages * stage;

  uint16_t* w1t = static_cast<uint16_t*>(workspace);
  CUtensorMap tm_h, tm_w;
  {
    cuuint64_t dims[2] = {(cuuint64_t)Dh, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)Dh * 2};
    cuuint32_t box[2] = {(cuuint32_t)kKBlock, (cuuint32_t)kTileRows};
    cuuint32_t es[2] = {1, 1};
    if (g_encode(&tm_h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(hidden), dims,
                 strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return KVC_ERR_CUDA;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)Dh, (cuuint64_t)(p.n_pass * p.np)};
    cuuint64_t strides[1] = {(cuuint64_t)Dh * 2};
    cuuint32_t box[2] = {(cuuint32_t)kKBlock, (cuuint32_t)p.bw};
    cuuint32_t es[2] = {1, 1};
    if (g_encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w1t, dims, strides, box, es,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return KVC_ERR_CUDA;
  }
  // W1t rows up to n_pass * np (>= Dmp) are written, the padding with zeros
  const int rows_t = p.n_pass * p.np;
  if (int rc = launch_pdl(w1_transpose_kernel, dim3((unsigned)((Dh + 31) / 32), (unsigned)((rows_t + 31) / 32)),
                          dim3(256), 0, s, static_cast<const uint16_t*>(w1), Dh, Dm, rows_t, w1t))
    return rc;
  switch (Hkv) {
    case 1: return launch_tc<1>(tm_h, tm_w, p, smem, dev, s);
    case 2: return launch_tc<2>(tm_h, tm_w, p, smem, dev, s);
    case 3: return launch_tc<3>(tm_h, tm_w, p, smem, dev, s);
    case 4: return launch_tc<4>(tm_h, tm_w, p, smem, dev, s);
    case 5: return launch_tc<5>(tm_h, tm_w, p, smem, dev, s);
    case 6: return launch_tc<6>(tm_h, tm_w, p, smem, dev, s);
    case 7: return launch_tc<7>(tm_h, tm_w, p, smem, dev, s);
    case 8: return launch_tc<8>(tm_h, tm_w, p, smem, dev, s);
  }
  return KVC_ERR_UNSUPPORTED;
}

}  // namespace kvc
