// Attention-mass scoring on the 5th-generation tensor cores (bf16, d = 128).
//
// Definition (KVSculpt §1 / §2B, KVzap §2.1): for unit u, kv head g, the
// R = G*W window rows r = (h, w) of its query heads and every cached token t,
//   s[r,t] = scale * f[u,h] * <q[u,h,w], k[u,g,t]>   (t <= T-W+w if causal)
//   score[u,g,t] = sum_r exp(s[r,t] - lse_r),  lse_r = log sum_t exp(s[r,t]).
//
// The contraction Q_g (R x 128) . K_g^T (128 x T) is a real dense GEMM, so it
// runs on tcgen05 with fp32 accumulators in TMEM.  The column mass needs
// every row's normaliser first, so the kernel makes two passes over the
// CTA's K tiles (the second pass finds them in L2):
//
//   pass 1  S = Q . K_tile^T  (rows on TMEM lanes, M = 128 per m-tile,
//           N = 128 tokens): each epilogue thread owns one window row and
//           keeps an online (max, sum) in base 2;
//   merge   the cluster's CTAs (one cluster per (u, g), each CTA a token
//           range) exchange their per-row partial (max, sum) through
//           distributed shared memory -> lse_r for all R rows;
//   pass 2  S^T = K_tile . Q^T (tokens on TMEM lanes, M = 128, N = R): each
//           epilogue thread owns one token and sums exp2(s*c_r - lse2_r)
//           over its half of the R columns; the two halves add in shared
//           memory and the token's score is stored (coalesced).
//
// Warp roles (320 threads): warps 0-7 epilogue (warp w reads TMEM lanes
// 32*(w%4)..+31, half w/4 of the columns), warp 8 TMA producer, warp 9 MMA
// issuer and TMEM owner.  K tiles stream through a 4-stage TMA ring
// (128 tokens x 128 dims, two 128-byte-swizzled boxes per stage); the
// accumulator is double-buffered in TMEM (2 x 256 of the 512 columns), so
// the MMA of tile j+1 overlaps the epilogue of tile j.  Every mbarrier wait
// is bounded (2 s); on expiry the status word records KVC_ERR_TIMEOUT and
// the kernel runs to completion without hanging.
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_ptx.cuh"

namespace kvc {
namespace {

constexpr int kD = 128;              // head dim handled here
constexpr int kTile = 128;           // tokens per K tile
constexpr int kStages = 4;
constexpr int kEpiWarps = 8;
constexpr int kThreads = (kEpiWarps + 2) * 32;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kStageBytes = kTile * kD * 2;          // 32 KiB
constexpr uint32_t kHalfBytes = kTile * 64 * 2;           // one 64-dim box: 16 KiB
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
  int T, W, R, Hq, Hkv, G;
  float scale;
  const float* head_scale;
  int causal;
  float* scores;
  int n_tiles;       // tiles of T
  int* status;
};

struct SmemSmall {
  uint64_t full[kStages], empty[kStages];
  uint64_t tmem_full[2], tmem_empty[2];
  uint64_t q_full;
  uint32_t tmem_base;
  int abort_flag;
  float m_part[256], l_part[256];      // read by the other CTAs of the cluster
  float2 cl[256];                      // (c_r, lse2_r) for pass 2
  float coef[256];
  float psum[2][kTile];                // pass-2 half sums
  float mh[2][128], lh[2][128];        // R = 128: the two column halves' stats
};

__device__ __forceinline__ uint32_t align1024(uint32_t a) { return (a + 1023u) & ~1023u; }

__global__ void __launch_bounds__(kThreads, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  SmemSmall& sm = *reinterpret_cast<SmemSmall*>(smem_raw);
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t q_smem = align1024(raw + (uint32_t)sizeof(SmemSmall));
  const uint32_t q_half_bytes = (uint32_t)p.R * 128u;        // R rows x 64 dims x 2 B
  const uint32_t k_smem = q_smem + 2u * q_half_bytes;        // 1024-aligned (R % 8 == 0)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = tc::cluster_ctarank();
  const uint32_t csize = tc::cluster_nctarank();
  const int ug = blockIdx.y;                                  // u * Hkv + g
  const int u = ug / p.Hkv, g = ug - u * p.Hkv;
  const int tile_lo = (int)((int64_t)crank * p.n_tiles / csize);
  const int tile_hi = (int)((int64_t)(crank + 1) * p.n_tiles / csize);
  const int nt = tile_hi - tile_lo;
  const int R = p.R, W = p.W, T = p.T;
  const int n_mt = R / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(&sm.full[s], 1); mbar_init(&sm.empty[s], 1); }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.tmem_full[b], 1);
      mbar_init(&sm.tmem_empty[b], kEpiWarps * 32);
    }
    mbar_init(&sm.q_full, 1);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tc::tmem_alloc(&sm.tmem_base, kTmemCols);
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------ TMA producer
    tc::cluster_arrive();                       // phase 0 needs no producer work
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_k);
      const int qrow = (u * p.Hq + g * p.G) * W;
      mbar_arrive_expect_tx(&sm.q_full, 2u * q_half_bytes);
      tc::tma_load_2d(q_smem, &tm_q, 0, qrow, &sm.q_full);
      tc::tma_load_2d(q_smem + q_half_bytes, &tm_q, 64, qrow, &sm.q_full);
      for (int J = 0; J < 2 * nt; ++J) {
        const int s = J % kStages;
        if (J >= kStages) mbar_wait(&sm.empty[s], ((J / kStages) - 1) & 1, p.status, abort_flag);
        const int t0 = (tile_lo + J % nt) * kTile;
        const uint32_t dst = k_smem + (uint32_t)s * kStageBytes;
        mbar_arrive_expect_tx(&sm.full[s], kStageBytes);
        tc::tma_load_3d(dst, &tm_k, 0, t0, ug, &sm.full[s]);
        tc::tma_load_3d(dst + kHalfBytes, &tm_k, 64, t0, ug, &sm.full[s]);
      }
    }
    __syncwarp();
    tc::cluster_wait();
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------- MMA issuer
    tc::cluster_arrive();
    if (lane == 0) {
      mbar_wait(&sm.q_full, 0, p.status, abort_flag);
      tc::fence_after_sync();
      const uint32_t idesc1 = tc::idesc_bf16_f32(128, kTile);   // pass 1: N = tokens
      const uint32_t idesc2 = tc::idesc_bf16_f32(128, R);       // pass 2: N = rows
      for (int J = 0; J < 2 * nt; ++J) {
        const int s = J % kStages, b = J & 1;
        mbar_wait(&sm.full[s], (J / kStages) & 1, p.status, abort_flag);
        if (J >= 2) mbar_wait(&sm.tmem_empty[b], ((J >> 1) - 1) & 1, p.status, abort_flag);
        tc::fence_after_sync();
        const uint32_t kst = k_smem + (uint32_t)s * kStageBytes;
        const uint32_t dcol = tmem + (uint32_t)b * 256u;
        if (J < nt) {
          for (int mt = 0; mt < n_mt; ++mt) {
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t kh = kk >> 2, ko = (kk & 3) * 32u;
              const uint64_t a = tc::smem_desc_sw128(q_smem + kh * q_half_bytes + mt * 128u * 128u + ko);
              const uint64_t bd = tc::smem_desc_sw128(kst + kh * kHalfBytes + ko);
              tc::mma_bf16(dcol + (uint32_t)mt * 128u, a, bd, idesc1, kk > 0);
            }
          }
        } else {
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t kh = kk >> 2, ko = (kk & 3) * 32u;
            const uint64_t a = tc::smem_desc_sw128(kst + kh * kHalfBytes + ko);
            const uint64_t bd = tc::smem_desc_sw128(q_smem + kh * q_half_bytes + ko);
            tc::mma_bf16(dcol, a, bd, idesc2, kk > 0);
          }
        }
        tc::mma_commit(&sm.empty[s]);
        tc::mma_commit(&sm.tmem_full[b]);
      }
    }
    __syncwarp();
    tc::cluster_wait();
  } else {
    // ---------------------------------------------------------- epilogue
    const int q4 = warp & 3, hf = warp >> 2;
    const int et = threadIdx.x;                 // 0..255
    for (int r = et; r < R; r += kEpiWarps * 32) {
      const int h = g * p.G + r / W;
      const float f = p.head_scale ? p.head_scale[(int64_t)u * p.Hq + h] : 1.0f;
      sm.coef[r] = p.scale * f * kLog2e;
    }
    tc::named_sync(1, kEpiWarps * 32);
    const uint32_t lane_addr = (uint32_t)(32 * q4) << 16;
    // pass 1: this thread's window row and column range
    const int row = (R == 256) ? hf * 128 + 32 * q4 + lane : 32 * q4 + lane;
    const int col0 = (R == 256) ? 0 : hf * 64;
    const int ncol = (R == 256) ? 128 : 64;
    const uint32_t mcol = (R == 256) ? (uint32_t)hf * 128u : 0u;
    const float c_r = sm.coef[row];
    const int tlim = p.causal ? (T - W + row % W) : (T - 1);   // last visible token
    float m = -INFINITY, l = 0.0f;
    for (int J = 0; J < nt; ++J) {
      const int b = J & 1;
      mbar_wait(&sm.tmem_full[b], (J >> 1) & 1, p.status, abort_flag);
      tc::fence_after_sync();
      const int t0 = (tile_lo + J) * kTile + col0;
      for (int c = 0; c < ncol; c += 32) {
        float v[32];
        tc::tmem_ld32(tmem + lane_addr + (uint32_t)b * 256u + mcol + (uint32_t)(col0 + c), v);
        const int tc0 = t0 + c;
        float cmax = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          v[j] = (tc0 + j <= tlim) ? v[j] * c_r : -INFINITY;
          cmax = fmaxf(cmax, v[j]);
        }
        const float mn = fmaxf(m, cmax);
        if (mn != -INFINITY) {
          float sum = 0.0f;
#pragma unroll
          for (int j = 0; j < 32; ++j) sum += tc::ex2(v[j] - mn);
          l = l * tc::ex2(m - mn) + sum;
          m = mn;
        }
      }
      tc::fence_before_sync();
      mbar_arrive(&sm.tmem_empty[b]);
    }
    if (R == 256) {
      sm.m_part[row] = m;
      sm.l_part[row] = l;
    } else {
      sm.mh[hf][row] = m;
      sm.lh[hf][row] = l;
      tc::named_sync(1, kEpiWarps * 32);
      if (hf == 0) {
        const float m2 = sm.mh[1][row], l2 = sm.lh[1][row];
        const float mn = fmaxf(m, m2);
        float ls = 0.0f;
        if (mn != -INFINITY) ls = l * tc::ex2(m - mn) + l2 * tc::ex2(m2 - mn);
        sm.m_part[row] = mn;
        sm.l_part[row] = ls;
      }
    }
    // cluster-wide merge of the per-row partials -> lse2 per row
    tc::cluster_arrive();
    tc::cluster_wait();
    for (int r = et; r < R; r += kEpiWarps * 32) {
      float M = -INFINITY;
      const uint32_t ma = smem_u32(&sm.m_part[r]), la = smem_u32(&sm.l_part[r]);
      for (uint32_t c = 0; c < csize; ++c) M = fmaxf(M, tc::ld_cluster_f32(tc::map_rank(ma, c)));
      float L = 0.0f;
      for (uint32_t c = 0; c < csize; ++c) {
        const float mc = tc::ld_cluster_f32(tc::map_rank(ma, c));
        if (mc != -INFINITY) L += tc::ld_cluster_f32(tc::map_rank(la, c)) * tc::ex2(mc - M);
      }
      sm.cl[r] = make_float2(sm.coef[r], M + __log2f(L));
    }
    tc::named_sync(1, kEpiWarps * 32);
    // pass 2: this thread's token and half of the R columns
    const int half_cols = R / 2;
    const int rc0 = hf * half_cols;
    for (int J = nt; J < 2 * nt; ++J) {
      const int b = J & 1;
      mbar_wait(&sm.tmem_full[b], (J >> 1) & 1, p.status, abort_flag);
      tc::fence_after_sync();
      const int tok = (tile_lo + J - nt) * kTile + 32 * q4 + lane;
      // causal: window row w sees token tok iff w >= tok - (T - W)
      const int wmin = p.causal ? tok - (T - W) : 0;
      float sum = 0.0f;
      for (int c = 0; c < half_cols; c += 32) {
        float v[32];
        tc::tmem_ld32(tmem + lane_addr + (uint32_t)b * 256u + (uint32_t)(rc0 + c), v);
        if (wmin <= 0) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float2 cl = sm.cl[rc0 + c + j];
            sum += tc::ex2(fmaf(v[j], cl.x, -cl.y));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int r = rc0 + c + j;
            const float2 cl = sm.cl[r];
            if (r % W >= wmin) sum += tc::ex2(fmaf(v[j], cl.x, -cl.y));
          }
        }
      }
      tc::fence_before_sync();
      mbar_arrive(&sm.tmem_empty[b]);
      if (hf == 1) sm.psum[J & 1][32 * q4 + lane] = sum;
      tc::named_sync(2, kEpiWarps * 32);
      if (hf == 0 && tok < T)
        p.scores[(int64_t)ug * T + tok] = sum + sm.psum[J & 1][32 * q4 + lane];
    }
  }
  // no CTA may leave while a peer still reads its shared memory
  __syncwarp();
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

size_t smem_bytes(int R) {
  return sizeof(SmemSmall) + 1024 /*alignment slack*/ + 2ull * R * 128 + (size_t)kStages * kStageBytes;
}

}  // namespace

bool score_attn_tc_supported(int dtype, int Hq, int Hkv, int W, int d) {
  if (dtype != KVC_BF16 || d != kD || Hkv <= 0 || Hq % Hkv) return false;
  const int R = (Hq / Hkv) * W;
  return R == 128 || R == 256;
}

int score_attn_tc(const void* q, const void* k, int U, int Hq, int Hkv, int T, int W,
                  float scale, const float* head_scale, int causal, float* scores,
                  const Dev& dev, cudaStream_t s) {
  int rc = get_encoder();
  if (rc) return rc;
  const int G = Hq / Hkv, R = G * W;
  CUtensorMap tm_q, tm_k;
  {
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)U * Hq * W};
    cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)R};
    cuuint32_t es[2] = {1, 1};
    if (g_encode(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides,
                 box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return KVC_ERR_CUDA;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)T, (cuuint64_t)U * Hkv};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)T * kD * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (g_encode(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k), dims, strides,
                 box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return KVC_ERR_CUDA;
  }
  Params p;
  p.T = T; p.W = W; p.R = R; p.Hq = Hq; p.Hkv = Hkv; p.G = G; p.scale = scale;
  p.head_scale = head_scale; p.causal = causal; p.scores = scores;
  p.n_tiles = (T + kTile - 1) / kTile; p.status = dev.status;
  const size_t smem = smem_bytes(R);
  if ((int)smem > dev.max_smem_optin) return KVC_ERR_UNSUPPORTED;
  KVC_CUDA_TRY(cudaFuncSetAttribute(score_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem));
  KVC_CUDA_TRY(cudaFuncSetAttribute(score_tc_kernel,
                                    cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
  // cluster size: about 16 tiles (512 KiB of K) per CTA, so that the second
  // pass re-reads K from L2; at most 16; shrink until a cluster fits a GPC
  int C = 1;
  while (C < 16 && (p.n_tiles + C - 1) / C > 16) C *= 2;
  while (C > 1 && (int64_t)U * Hkv * C > 4ll * dev.sms && (p.n_tiles + C / 2 - 1) / (C / 2) <= 32) C /= 2;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  for (;;) {
    cfg.gridDim = dim3((unsigned)C, (unsigned)(U * Hkv), 1);
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
    KVC_CUDA_TRY(cudaOccupancyMaxActiveClusters(&active, score_tc_kernel, &cfg));
    if (active > 0) break;
    if (C == 1) return KVC_ERR_UNSUPPORTED;
    C /= 2;
  }
  KVC_CUDA_TRY(cudaLaunchKernelEx(&cfg, score_tc_kernel, tm_q, tm_k, p));
  return launch_status();
}

}  // namespace kvc
