// Attention-mass scoring on the 5th-generation tensor cores (bf16, d = 128).
//
// Definition (KVSculpt §1 / §2B, KVzap §2.1): for unit u, kv head g, the
// R = G*W window rows r = (h, w) of its query heads and every cached token t,
//   s[r,t] = scale * f[u,h] * <q[u,h,w], k[u,g,t]>   (t <= T-W+w if causal)
//   score[u,g,t] = sum_r exp(s[r,t] - lse_r),  lse_r = log sum_t exp(s[r,t]).
//
// The contraction Q_g (R x 128) . K_g^T (128 x T) is a real dense GEMM, so it
// runs on tcgen05 with fp32 accumulators in TMEM.  The column mass needs
// every row's normaliser first, so each CTA makes two passes over its K
// (the second pass finds it in L2).  K streams in stages of two 128-token
// tiles (a range's last stage holds one when its tile count is odd); every
// MMA item is 8 MMAs (K = 16 each) into one 256-column TMEM buffer:
//
//   pass 1  S = Q_m . K_stage^T, one item per 128-row m-tile (rows on TMEM
//           lanes, the stage's tokens on columns, N = 256 or 128): each
//           epilogue thread owns one window row and 64 of the columns and
//           keeps a running (max, sum) in base 2;
//   merge   the CTAs that share a (u, g) publish their per-row partial
//           (max, sum) in global memory, each 32-bit value paired with a
//           per-launch tag in one 64-bit word, and poll (bounded) the
//           others' partials until the tags match -> lse_r of every row;
//   pass 2  S^T = K_tile . Q^T, one item per 128-token tile (tokens on TMEM
//           lanes, N = R): each epilogue thread owns one token and a quarter
//           of the R columns and sums exp2(c_r * s - lse2_r); quarters 1-3
//           hand their sums to quarter 0 through double-buffered shared slots
//           guarded by mbarriers, and quarter 0 stores the token's score.
//
// Work split: one persistent CTA per SM (cooperative launch, so every CTA
// of a group is resident while its peers wait for it).  The (u, g) pairs
// are processed in rounds; in a round, group i of gs CTAs owns one (u, g)
// and CTA j of the group a contiguous range of 128-token tiles (about 16,
// 512 KiB of K; ranges differ by at most one tile), so that the second pass
// re-reads K from L2 while every SM is busy.
//
// Warp roles (576 threads): warps 0-15 epilogue (warp w reads TMEM lanes
// 32*(w%4)..+31; w/4 picks its column slice), warp 16 TMA producer, warp 17
// MMA issuer and TMEM owner.  Stages stream through a 2-stage TMA ring
// (256 tokens x 128 dims, four 128-byte-swizzled boxes per stage); the
// accumulator is double-buffered in TMEM (2 x 256 of the 512 columns), so
// the MMA of item j+1 overlaps the epilogue of item j.  The window queries
// of the round's (u, g) sit in shared memory for both passes.  Every wait
// is bounded (2 s): on expiry the status word records KVC_ERR_TIMEOUT and
// the kernel runs to completion without hanging.
#include <cudaTypedefs.h>

#include <atomic>
#include <chrono>
#include <mutex>

#include "tc_ptx.cuh"

namespace kvc {
namespace {

constexpr int kD = 128;              // head dim handled here
constexpr int kTile = 128;           // tokens per K tile
constexpr int kStages = 2;         // super-stages of 256 tokens
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = kEpiThreads + 64;
constexpr int kProducerWarp = kEpiWarps;
constexpr int kMmaWarp = kEpiWarps + 1;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBoxBytes = kTile * 64 * 2;            // one 128 x 64 box: 16 KiB
constexpr uint32_t kHalfBytes = 2 * kBoxBytes;            // 256 tokens x 64 dims: 32 KiB
constexpr uint32_t kStageBytes = 2 * kHalfBytes;          // 256 tokens x 128 dims: 64 KiB
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxGroup = 32;        // CTAs sharing one (u, g)
constexpr int kMaxCtas = 1024;       // grid bound (workspace sizing)
constexpr int kSupersPerCta = 8;     // target super-tiles (256 tokens) per CTA and round

struct Params {
  int T, W, R, Hq, Hkv, G;
  float scale;
  const float* head_scale;
  int causal;
  float* scores;
  int n_tiles;       // 128-token tiles of T
  int heads;         // U * Hkv
  int gs;            // CTAs per (u, g)
  int hpr;           // (u, g) pairs per round
  int rounds;
  ulonglong2* parts; // [2][grid][R] per-CTA row partials: (max2 | tag, sum | tag)
  uint64_t tag0;     // this launch's tag base (unique per launch)
  int* status;
  const float* hnorm;  // KVzip+ only: hidden-state norm per (unit, window row)
  const float* vnorm;  // KVzip+ only: ||W_O^h v_t|| per (unit, query head, token)
};

struct SmemSmall {
  uint64_t full[kStages], empty[kStages];
  uint64_t tmem_full[2], tmem_empty[2];
  uint64_t q_full, q_empty;
  uint64_t psum_full[2], psum_empty[2];  // pass-2 quarter sums: written / consumed
  uint32_t tmem_base;
  int abort_flag;
  float4 cl4[128];                     // column pairs (c, c', -lse2, -lse2') for pass 2
  float4 nl4[64];                      // -lse2 of four consecutive columns (uniform c)
  float coef[256];                     // c_r = scale * f * log2(e) per window row
  float nlse[256];                     // -lse2 per window row
  float mpart[4][256], lpart[4][256];  // per column slice (max2, sum) of each row
  float psum[2][4][kTile];             // pass-2 quarter sums per token
};

__device__ __forceinline__ uint32_t align1024(uint32_t a) { return (a + 1023u) & ~1023u; }

// A row partial travels as two 64-bit words, each a 32-bit value and the
// round's 32-bit tag; a 64-bit access is single-copy atomic, so a reader
// that sees the tag in both words has the value too (no fence, no flag).
__device__ __forceinline__ ulonglong2 ld_relaxed_v2(const ulonglong2* p) {
  ulonglong2 v;
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];"
               : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_v2(ulonglong2* p, uint64_t a, uint64_t b) {
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b)
               : "memory");
}

// Merge of two base-2 (max, sum) pairs.
__device__ __forceinline__ void merge_ms(float& M, float& L, float m, float l) {
  if (m == -INFINITY) return;
  if (m > M) { L = L * tc::ex2(M - m) + l; M = m; }
  else       { L += l * tc::ex2(m - M); }
}

// Pass-2 accumulation of the window rows' weights of a token: their sum (the
// attention mass) or, with kMax, their maximum.  Two lanes per 64-bit word.
template <bool kMax>
__device__ __forceinline__ uint64_t acc2(uint64_t s, float e0, float e1) {
  if constexpr (kMax) {
    const float2 a = tc::upk2(s);
    return tc::pk2(fmaxf(a.x, e0), fmaxf(a.y, e1));
  } else {
    return tc::fadd2(s, tc::pk2(e0, e1));
  }
}
template <bool kMax>
__device__ __forceinline__ uint64_t comb2(uint64_t a, uint64_t b) {
  const float2 y = tc::upk2(b);
  return acc2<kMax>(a, y.x, y.y);
}
template <bool kMax>
__device__ __forceinline__ float comb(float a, float b) {
  return kMax ? fmaxf(a, b) : a + b;
}

// kPlus (with kMax): the KVzip+ score -- each row's weights divided by the
// row's hidden-state norm (folded into its normaliser), each quarter's
// maximum (one query head's rows) times the token's value norm for that head
template <bool kMax, bool kPlus = false>
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
  const int cta = blockIdx.x;
  const int grp = cta / p.gs, slot = cta - grp * p.gs;
  const bool in_group = grp < p.hpr;
  // this CTA's 128-token K tiles [tl_lo, tl_hi) of its (u, g), streamed as
  // ns stages of two tiles (the last stage holds one when ntl is odd)
  const int tl_lo = (int)((int64_t)slot * p.n_tiles / p.gs);
  const int tl_hi = (int)((int64_t)(slot + 1) * p.n_tiles / p.gs);
  const int ntl = tl_hi - tl_lo;
  const int ns = (ntl + 1) >> 1;
  const int R = p.R, W = p.W, T = p.T;
  const int n_mt = R / 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(&sm.full[s], 1); mbar_init(&sm.empty[s], 1); }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.tmem_full[b], 1);
      mbar_init(&sm.tmem_empty[b], kEpiThreads);
    }
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.psum_full[b], 12);    // the 12 warps of quarters 1-3
      mbar_init(&sm.psum_empty[b], 4);    // the 4 warps of quarter 0
    }
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
    // Stage layout (64 KiB): [dims 0-63 of tokens 0-255 | dims 64-127 of
    // tokens 0-255], so each 64-dim half of a super-tile is one contiguous
    // 256-row swizzled operand.
    if (lane == 0 && in_group && ns > 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_k);
      int J = 0, qk = 0;
      for (int k = 0; k < p.rounds; ++k) {
        const int head = k * p.hpr + grp;
        if (head >= p.heads) break;
        const int u = head / p.Hkv, g = head - u * p.Hkv;
        if (qk > 0) mbar_wait(&sm.q_empty, (qk - 1) & 1, p.status, abort_flag);
        const int qrow = (u * p.Hq + g * p.G) * W;
        mbar_arrive_expect_tx(&sm.q_full, 2u * q_half_bytes);
        tc::tma_load_2d(q_smem, &tm_q, 0, qrow, &sm.q_full);
        tc::tma_load_2d(q_smem + q_half_bytes, &tm_q, 64, qrow, &sm.q_full);
        for (int i = 0; i < 2 * ns; ++i, ++J) {
          const int s = J % kStages;
          if (J >= kStages) mbar_wait(&sm.empty[s], ((J / kStages) - 1) & 1, p.status, abort_flag);
          const int si = i % ns, nti = min(2, ntl - 2 * si);   // tiles in this stage
          const int t0 = (tl_lo + 2 * si) * kTile;
          const uint32_t dst = k_smem + (uint32_t)s * kStageBytes;
          mbar_arrive_expect_tx(&sm.full[s], (uint32_t)nti * 2u * kBoxBytes);
#pragma unroll
          for (int h = 0; h < 2; ++h)
            for (int tt = 0; tt < nti; ++tt)
              tc::tma_load_3d(dst + h * kHalfBytes + tt * kBoxBytes, &tm_k, 64 * h,
                              t0 + tt * kTile, head, &sm.full[s]);
        }
        ++qk;
      }
    }
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------- MMA issuer
    // pass 1 items: (stage, m-tile), D = Q_mtile . K_stage^T, N = 128 x tiles
    // pass 2 items: (stage, tile),   D = K_tile . Q^T,         N = R
    // every item is 8 MMAs (K = 16 each) into one 256-column TMEM buffer
    if (lane == 0 && in_group && ns > 0) {
      const uint32_t idesc1 = tc::idesc_bf16_f32(128, 2 * kTile);
      const uint32_t idesc1h = tc::idesc_bf16_f32(128, kTile);    // a one-tile stage
      const uint32_t idesc2 = tc::idesc_bf16_f32(128, R);
      int J = 0, item = 0, qk = 0;
      for (int k = 0; k < p.rounds; ++k) {
        const int head = k * p.hpr + grp;
        if (head >= p.heads) break;
        mbar_wait(&sm.q_full, qk & 1, p.status, abort_flag);
        tc::fence_after_sync();
        for (int i = 0; i < 2 * ns; ++i, ++J) {
          const int s = J % kStages;
          mbar_wait(&sm.full[s], (J / kStages) & 1, p.status, abort_flag);
          tc::fence_after_sync();
          const uint32_t kst = k_smem + (uint32_t)s * kStageBytes;
          const int nti = min(2, ntl - 2 * (i < ns ? i : i - ns));
          const int n_items = (i < ns) ? n_mt : nti;
          for (int x = 0; x < n_items; ++x, ++item) {
            const int b = item & 1;
            if (item >= 2) mbar_wait(&sm.tmem_empty[b], ((item >> 1) - 1) & 1, p.status, abort_flag);
            tc::fence_after_sync();
            const uint32_t dcol = tmem + (uint32_t)b * 256u;
            // operand descriptors of the item's first k step, for each 64-dim
            // half; a 16-wide k step adds 32 bytes (2 in the descriptor's
            // address field, which cannot carry below 256 KiB)
            uint32_t a_lo, b_lo, id;
            if (i < ns) {
              a_lo = q_smem + x * 128u * 128u;
              b_lo = kst;
              id = nti == 2 ? idesc1 : idesc1h;
            } else {
              a_lo = kst + x * kBoxBytes;
              b_lo = q_smem;
              id = idesc2;
            }
            const uint32_t a_hstep = i < ns ? q_half_bytes : kHalfBytes;
            const uint32_t b_hstep = i < ns ? kHalfBytes : q_half_bytes;
            const uint64_t ad0 = tc::smem_desc_sw128(a_lo), bd0 = tc::smem_desc_sw128(b_lo);
            const uint64_t ad1 = tc::smem_desc_sw128(a_lo + a_hstep);
            const uint64_t bd1 = tc::smem_desc_sw128(b_lo + b_hstep);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) tc::mma_bf16(dcol, ad0 + 2u * kk, bd0 + 2u * kk, id, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) tc::mma_bf16(dcol, ad1 + 2u * kk, bd1 + 2u * kk, id, 1u);
            tc::mma_commit(&sm.tmem_full[b]);
          }
          tc::mma_commit(&sm.empty[s]);
        }
        tc::mma_commit(&sm.q_empty);       // the queries are free once these MMAs finish
        ++qk;
      }
    }
  } else if (in_group && ns > 0) {
    // ---------------------------------------------------------- epilogue
    // Per element the inner loops issue one ex2 plus about one and a half
    // other instructions (packed f32x2 FMA / add, three-input max trees,
    // several independent accumulators); four epilogue warps per SM
    // sub-partition keep the exponential unit busy across TMEM-load waits.
    const int q4 = warp & 3, wq = warp >> 2;     // lane quadrant, column slice
    const int et = threadIdx.x;                  // 0..511
    const uint32_t lane_addr = (uint32_t)(32 * q4) << 16;
    // pass 1: rows on lanes; this thread owns row mt*128 + 32*q4 + lane of
    // each m-tile and tokens [64*wq, 64*wq + 64) of every super-tile
    const int lrow = 32 * q4 + lane;
    // pass 2: tokens on lanes; this thread owns a quarter of the R columns
    const int qcols = R / 4;
    const int rc0 = wq * qcols;
    int item = 0, kr = 0, p2 = 0;
    for (int k = 0; k < p.rounds; ++k, ++kr) {
      const int head = k * p.hpr + grp;
      if (head >= p.heads) break;
      const int u = head / p.Hkv, g = head - u * p.Hkv;
      for (int r = et; r < R; r += kEpiThreads) {
        const int h = g * p.G + r / W;
        const float f = p.head_scale ? p.head_scale[(int64_t)u * p.Hq + h] : 1.0f;
        if (!(f > 0.0f && f < INFINITY)) report(p.status, KVC_ERR_INVALID);
        sm.coef[r] = p.scale * f * kLog2e;
      }
      tc::named_sync(1, kEpiThreads);
      // ---- pass 1: running (max, sum) of this thread's row slices
      float c_r[2], m[2];
      uint64_t acc[2][4];
      int tlim[2];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int row = mt * 128 + lrow;
        c_r[mt] = (mt < n_mt) ? sm.coef[row] : 0.0f;
        m[mt] = -INFINITY;
        tlim[mt] = p.causal ? (T - W + row % W) : (T - 1);   // last visible token
#pragma unroll
        for (int x = 0; x < 4; ++x) acc[mt][x] = 0ull;
      }
      for (int i = 0; i < ns; ++i) {
        // a one-tile stage fills columns 0-127 only: slices 2 and 3 idle
        const bool cols = 64 * wq < min(2, ntl - 2 * i) * kTile;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          if (mt >= n_mt) break;
          const int b = item & 1;
          mbar_wait(&sm.tmem_full[b], (item >> 1) & 1, p.status, abort_flag);
          tc::fence_after_sync();
          const uint64_t c2 = tc::pk2(c_r[mt], c_r[mt]);
          const int t0 = (tl_lo + 2 * i) * kTile + 64 * wq;
#pragma unroll 1
          for (int c = 0; c < (cols ? 64 : 0); c += 32) {
            float v[32];
            tc::tmem_ld32(tmem + lane_addr + (uint32_t)b * 256u + (uint32_t)(64 * wq + c), v);
            const int tc0 = t0 + c;
            if (tc0 + 31 > tlim[mt]) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = (tc0 + j <= tlim[mt]) ? v[j] : -INFINITY;
            }
            // The row's reference m only moves when a chunk's terms relative
            // to it would reach 2^64: the chunk is summed against the current
            // m, and only a first chunk, a chunk that large (or one holding
            // inf / NaN) takes the maximum and rescales.  The running sum
            // stays below 2^80, far from fp32's range.
            uint64_t cs[4] = {0ull, 0ull, 0ull, 0ull};
            bool redo = m[mt] == -INFINITY;
            if (!redo) {
              const float nm = -c_r[mt] * m[mt];
              const uint64_t nm2 = tc::pk2(nm, nm);
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float2 x = tc::upk2(tc::ffma2(tc::pk2(v[2 * j], v[2 * j + 1]), c2, nm2));
                cs[j & 3] = tc::fadd2(cs[j & 3], tc::pk2(tc::ex2(x.x), tc::ex2(x.y)));
              }
              const float2 t = tc::upk2(tc::fadd2(tc::fadd2(cs[0], cs[1]), tc::fadd2(cs[2], cs[3])));
              redo = !(t.x + t.y < 1.8e19f);
            }
            if (redo) {
              const float cm = tc::max32(v);
              if (cm > m[mt]) {
                const float sc = (m[mt] == -INFINITY) ? 0.0f : tc::ex2(c_r[mt] * (m[mt] - cm));
                const uint64_t sc2 = tc::pk2(sc, sc);
#pragma unroll
                for (int x = 0; x < 4; ++x) acc[mt][x] = tc::ffma2(acc[mt][x], sc2, 0ull);
                m[mt] = cm;
              }
#pragma unroll
              for (int x = 0; x < 4; ++x) cs[x] = 0ull;
              if (m[mt] != -INFINITY) {
                const float nm = -c_r[mt] * m[mt];
                const uint64_t nm2 = tc::pk2(nm, nm);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  const float2 x = tc::upk2(tc::ffma2(tc::pk2(v[2 * j], v[2 * j + 1]), c2, nm2));
                  cs[j & 3] = tc::fadd2(cs[j & 3], tc::pk2(tc::ex2(x.x), tc::ex2(x.y)));
                }
              }
            }
#pragma unroll
            for (int x = 0; x < 4; ++x) acc[mt][x] = tc::fadd2(acc[mt][x], cs[x]);
          }
          tc::fence_before_sync();
          mbar_arrive(&sm.tmem_empty[b]);
          ++item;
        }
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        if (mt >= n_mt) break;
        const float2 a = tc::upk2(tc::fadd2(tc::fadd2(acc[mt][0], acc[mt][1]),
                                            tc::fadd2(acc[mt][2], acc[mt][3])));
        sm.mpart[wq][mt * 128 + lrow] = (m[mt] == -INFINITY) ? -INFINITY : c_r[mt] * m[mt];
        sm.lpart[wq][mt * 128 + lrow] = a.x + a.y;
      }
      tc::named_sync(1, kEpiThreads);
      // ---- publish this CTA's row partials, then gather the group's: every
      // partial carries the round's tag, so readers poll the data itself
      const uint64_t tg = (uint64_t)(uint32_t)((p.tag0 + (uint64_t)kr) ^ ((p.tag0 + (uint64_t)kr) >> 32)) << 32;
      ulonglong2* parts = p.parts + (size_t)(kr & 1) * gridDim.x * R;
      if (et < R) {
        float M = -INFINITY, L = 0.0f;
#pragma unroll
        for (int x = 0; x < 4; ++x) merge_ms(M, L, sm.mpart[x][et], sm.lpart[x][et]);
        st_relaxed_v2(parts + (size_t)cta * R + et, tg | __float_as_uint(M), tg | __float_as_uint(L));
      }
      tc::named_sync(1, kEpiThreads);
      // gather: thread (row, half) polls its half of the group's partials
      // (bounded), eight members at a time with all loads in flight, and
      // merges them in member order
      {
        const int gr = et & 255, gq = et >> 8;       // row, half of the group
        float M = -INFINITY, L = 0.0f;
        if (gr < R) {
          const ulonglong2* gp = parts + (size_t)grp * p.gs * R + gr;
          const int x0 = gq * ((p.gs + 1) >> 1), x1 = min(p.gs, x0 + ((p.gs + 1) >> 1));
          uint64_t t_start = 0;
#pragma unroll 1
          for (int xb = x0; xb < x1; xb += 8) {
            const int nx = min(8, x1 - xb);
            float mv[8], lv[8];
            uint32_t pending = 0xffu >> (8 - nx);
            for (uint32_t it = 0; pending; ++it) {
#pragma unroll
              for (int y = 0; y < 8; ++y) {
                if ((pending >> y) & 1u) {
                  const ulonglong2 w = ld_relaxed_v2(gp + (size_t)(xb + y) * R);
                  if ((w.x & 0xffffffff00000000ull) == tg && (w.y & 0xffffffff00000000ull) == tg) {
                    mv[y] = __uint_as_float((uint32_t)w.x);
                    lv[y] = __uint_as_float((uint32_t)w.y);
                    pending &= ~(1u << y);
                  }
                }
              }
              if (pending && (it & 7u) == 7u) {
                if (*abort_flag) break;
                const uint64_t now = globaltimer_ns();
                if (t_start == 0) t_start = now;
                else if (now - t_start > kWaitTimeoutNs) {
                  report(p.status, KVC_ERR_TIMEOUT);
                  *abort_flag = 1;
                  break;
                }
              }
            }
#pragma unroll
            for (int y = 0; y < 8; ++y)
              if (y < nx && !((pending >> y) & 1u)) merge_ms(M, L, mv[y], lv[y]);
          }
          sm.mpart[gq][gr] = M;
          sm.lpart[gq][gr] = L;
        }
      }
      tc::named_sync(1, kEpiThreads);
      if (et < R) {
        float M = sm.mpart[0][et], L = sm.lpart[0][et];
        merge_ms(M, L, sm.mpart[1][et], sm.lpart[1][et]);
        float nl = -(M + __log2f(L));      // -lse2 of row et
        if constexpr (kPlus) nl -= __log2f(p.hnorm[(int64_t)u * W + et % W]);
        sm.nlse[et] = nl;
      }
      tc::named_sync(1, kEpiThreads);
      if (et < R / 2)
        sm.cl4[et] = make_float4(sm.coef[2 * et], sm.coef[2 * et + 1], sm.nlse[2 * et],
                                 sm.nlse[2 * et + 1]);
      if (et < R / 4)
        sm.nl4[et] = make_float4(sm.nlse[4 * et], sm.nlse[4 * et + 1], sm.nlse[4 * et + 2],
                                 sm.nlse[4 * et + 3]);
      tc::named_sync(1, kEpiThreads);
      // one softmax scale for this thread's quarter of the columns: no
      // per-row temperature, or a quarter inside one query head's rows
      const bool cuni = !p.head_scale || (rc0 / W == (rc0 + qcols - 1) / W);
      const float cq = sm.cl4[rc0 >> 1].x;   // (sm.coef belongs to the next round once
                                             // a warp finishes this one)
      const uint64_t cq2 = tc::pk2(cq, cq);
      // the next kernel of the stream may be scheduled once every CTA is here
      if (et == 0 && kr == 0) pdl_trigger();
      // ---- pass 2: this thread's token and quarter of the R columns
      for (int i = 0; i < ntl; ++i, ++item) {
        const int b = item & 1;
        mbar_wait(&sm.tmem_full[b], (item >> 1) & 1, p.status, abort_flag);
        tc::fence_after_sync();
        const int tl = 32 * q4 + lane;
        const int tok = (tl_lo + i) * kTile + tl;
        // causal: window row w sees token tok iff w >= tok - (T - W)
        const int wmin = p.causal ? tok - (T - W) : 0;
        uint64_t s2[4] = {0ull, 0ull, 0ull, 0ull};
        for (int c = 0; c < qcols; c += 32) {
          float v[32];
          tc::tmem_ld32(tmem + lane_addr + (uint32_t)b * 256u + (uint32_t)(rc0 + c), v);
          const float4* cp = &sm.cl4[(rc0 + c) >> 1];
          if (wmin <= 0 && cuni) {
            const float4* np4 = &sm.nl4[(rc0 + c) >> 2];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 q = np4[j];
              const float2 x0 = tc::upk2(tc::ffma2(tc::pk2(v[4 * j], v[4 * j + 1]), cq2,
                                                   tc::pk2(q.x, q.y)));
              const float2 x1 = tc::upk2(tc::ffma2(tc::pk2(v[4 * j + 2], v[4 * j + 3]), cq2,
                                                   tc::pk2(q.z, q.w)));
              s2[(2 * j) & 3] = acc2<kMax>(s2[(2 * j) & 3], tc::ex2(x0.x), tc::ex2(x0.y));
              s2[(2 * j + 1) & 3] = acc2<kMax>(s2[(2 * j + 1) & 3], tc::ex2(x1.x), tc::ex2(x1.y));
            }
          } else if (wmin <= 0) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float4 q = cp[j];
              const float2 x = tc::upk2(tc::ffma2(tc::pk2(v[2 * j], v[2 * j + 1]),
                                                  tc::pk2(q.x, q.y), tc::pk2(q.z, q.w)));
              s2[j & 3] = acc2<kMax>(s2[j & 3], tc::ex2(x.x), tc::ex2(x.y));
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int r = rc0 + c + 2 * j;
              const float4 q = cp[j];
              const float e0 = (r % W >= wmin) ? tc::ex2(fmaf(v[2 * j], q.x, q.z)) : 0.0f;
              const float e1 = ((r + 1) % W >= wmin) ? tc::ex2(fmaf(v[2 * j + 1], q.y, q.w)) : 0.0f;
              s2[j & 3] = acc2<kMax>(s2[j & 3], e0, e1);
            }
          }
        }
        tc::fence_before_sync();
        mbar_arrive(&sm.tmem_empty[b]);
        const float2 a = tc::upk2(comb2<kMax>(comb2<kMax>(s2[0], s2[1]), comb2<kMax>(s2[2], s2[3])));
        float part = comb<kMax>(a.x, a.y);
        if constexpr (kPlus)
          part *= (tok < T) ? p.vnorm[((int64_t)u * p.Hq + g * p.G + rc0 / W) * T + tok] : 0.0f;
        // quarters 1-3 hand their sums to quarter 0 through a double-buffered
        // slot; only the two quarters involved wait, never the whole epilogue
        const int pb = p2 & 1, use = p2 >> 1;
        if (wq != 0) {
          if (use > 0) mbar_wait(&sm.psum_empty[pb], (use - 1) & 1, p.status, abort_flag);
          sm.psum[pb][wq][tl] = part;
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.psum_full[pb]);
        } else {
          mbar_wait(&sm.psum_full[pb], use & 1, p.status, abort_flag);
          const float* ps = &sm.psum[pb][0][tl];
          if (tok < T)
            p.scores[(int64_t)head * T + tok] =
                comb<kMax>(comb<kMax>(part, ps[kTile]), comb<kMax>(ps[2 * kTile], ps[3 * kTile]));
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.psum_empty[pb]);
        }
        ++p2;
      }
    }
  }
  __syncthreads();
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

size_t parts_bytes(int R) { return 2ull * kMaxCtas * R * sizeof(ulonglong2); }

// Launch tags: a process-wide counter seeded from the clock, in steps of
// 2^16 (a launch uses tag_base + round, rounds < 2^16).
uint64_t next_tag_base() {
  static std::atomic<uint64_t> counter{
      (uint64_t)std::chrono::steady_clock::now().time_since_epoch().count() << 20};
  return counter.fetch_add(1ull << 16) + (1ull << 16);
}

}  // namespace

bool score_attn_tc_supported(int dtype, int Hq, int Hkv, int W, int d) {
  if (dtype != KVC_BF16 || d != kD || Hkv <= 0 || Hq % Hkv) return false;
  const int R = (Hq / Hkv) * W;
  return R == 128 || R == 256;
}

size_t score_attn_tc_ws(int Hq, int Hkv, int W) {
  const int R = (Hq / Hkv) * W;
  return parts_bytes(R);
}

int score_attn_tc(const void* q, const void* k, int U, int Hq, int Hkv, int T, int W,
                  float scale, const float* head_scale, int causal, int agg, float* scores,
                  void* ws, const Dev& dev, cudaStream_t s, const float* hnorm,
                  const float* vnorm) {
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
  p.hnorm = hnorm; p.vnorm = vnorm;
  p.n_tiles = (T + kTile - 1) / kTile; p.status = dev.status;
  p.heads = U * Hkv;
  const size_t smem = smem_bytes(R);
  if ((int)smem > dev.max_smem_optin) return KVC_ERR_UNSUPPORTED;
  // attribute set-up and occupancy check, once per device and row count
  {
    static std::mutex mu;
    static int per_sm_memo[64][2];
    std::lock_guard<std::mutex> lock(mu);
    int& per_sm = per_sm_memo[dev.device & 63][R == 256];
    if (per_sm == 0) {
      // the attribute is the kernel's, shared by both row counts: the larger
      const size_t smax = smem_bytes(256);
      if ((int)smax > dev.max_smem_optin) return KVC_ERR_UNSUPPORTED;
      for (auto fn : {score_tc_kernel<false>, score_tc_kernel<true>, score_tc_kernel<true, true>})
        KVC_CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)smax));
      KVC_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, score_tc_kernel<false>,
                                                                 kThreads, smem));
      if (per_sm < 1) per_sm = -1;
    }
    if (per_sm < 1) return KVC_ERR_UNSUPPORTED;
  }
  // work split: P resident CTAs; gs CTAs per (u, g), hpr pairs per round
  const int P = dev.sms < kMaxCtas ? dev.sms : kMaxCtas;
  int gs;
  if (p.heads <= P) {
    gs = P / p.heads;
  } else {
    gs = (p.n_tiles + 2 * kSupersPerCta - 1) / (2 * kSupersPerCta);
    if (gs > P) gs = P;
  }
  if (gs > p.n_tiles) gs = p.n_tiles;
  if (gs > kMaxGroup) gs = kMaxGroup;
  if (gs < 1) gs = 1;
  p.gs = gs;
  p.hpr = P / gs;
  if (p.hpr > p.heads) p.hpr = p.heads;
  p.rounds = (p.heads + p.hpr - 1) / p.hpr;
  p.parts = static_cast<ulonglong2*>(ws);
  // tags are unique per launch (and per round inside it), so the workspace
  // needs no clearing: stale partials of earlier launches never match
  p.tag0 = next_tag_base();
  const int grid = p.hpr * gs;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: peers wait on each other
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto kern = agg == kAggKvzipPlus ? score_tc_kernel<true, true>
              : agg == KVC_AGG_MAX  ? score_tc_kernel<true>
                                    : score_tc_kernel<false>;
  if (int rc2 = prefer_max_shared(kern, dev.device)) return rc2;
  KVC_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, tm_q, tm_k, p));
  return launch_status();
}

}  // namespace kvc
