// VECTOR three-way routing of a selected pool ("A Simple Plug-in for
// Improving Eviction-Based KV Cache Compression", Méthodologie : VECTOR):
// keys stay exact for every pool token, values are kept, or dropped and
// rebuilt from the key by an offline OLS predictor W (v ~ W k), or evicted.
//
//   vector_residual_kernel  step 2: eps = ||v - W k||^2 of every pool token,
//                           written as a selection key -eps per pool position
//                           (NaN for protected tokens and empty positions), so
//                           that the global top-k picks the lowest errors;
//   vector_compact_kernel   step 3: K rows of all pool tokens (approximated
//                           first), V rows of the exact ones only.
//
// The residual is a small dense contraction per token (d x d multiply-adds for
// 2 d bf16 loads): it runs on warp-level bf16 MMAs, W staged once per CTA in
// shared memory and reused for every 16-token tile the CTA's warps gather.
#include <atomic>

#include "kvc_internal.cuh"
#include "mma_sync.cuh"

namespace kvc {
namespace {

using namespace ::kvc::mmasync;

constexpr int D = 128;              // head dimension of the VECTOR path
constexpr int RS = D + 8;           // padded smem row (bf16 elements): conflict-free ldmatrix
constexpr int kResWarps = 8;        // 16 pool positions per warp and tile
constexpr int kTile = kResWarps * 16;

struct ResidualSmem {
  uint16_t w[D * RS];                       // W_g, row = output dimension
  uint16_t kt[kResWarps][16 * RS];          // gathered K rows of each warp's tile
  uint16_t vt[kResWarps][16 * RS];          // and their V rows
};

__global__ void __launch_bounds__(kResWarps * 32)
vector_residual_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                       const uint16_t* __restrict__ W, int Hkv, int T,
                       const int32_t* __restrict__ kept_idx, const int32_t* __restrict__ counts,
                       int n_sink, int n_recent, float* __restrict__ key, int* status) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  ResidualSmem& sm = *reinterpret_cast<ResidualSmem*>(smem_raw);
  const int i = blockIdx.y;
  const int g = i % Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // stage W_g once (16-byte chunks, row-padded); W does not depend on the
  // previous kernel, so the copy overlaps its tail
  {
    const uint16_t* wg = W + (int64_t)g * D * D;
    const uint32_t wb = smem_u32(sm.w);
    for (int x = threadIdx.x; x < D * (D / 8); x += kResWarps * 32) {
      const int r = x / (D / 8), ch = x - r * (D / 8);
      cp_async16(wb + (uint32_t)(r * RS + ch * 8) * 2u, wg + r * D + ch * 8, 16u);
    }
    cp_commit();
  }
  pdl_wait();
  pdl_trigger();
  const int cnt = counts[i];
  const int ntiles = (T + kTile - 1) / kTile;
  const int64_t head_row0 = (int64_t)i * T;     // row of token 0 of head i in k / v
  cp_wait<0>();
  __syncthreads();
  const uint32_t kb = smem_u32(sm.kt[warp]), vb = smem_u32(sm.vt[warp]);
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int j0 = tile * kTile + warp * 16;           // this warp's first pool position
    // lanes 0..15 resolve position j0 + lane -> token (or -1: not eligible)
    int tok = -1;
    if (lane < 16) {
      const int j = j0 + lane;
      if (j < T && j < cnt) {
        const int t = kept_idx[(int64_t)i * T + j];
        if (t < 0 || t >= T) {
          report(status, KVC_ERR_RANGE);
        } else if (t >= n_sink && t < T - n_recent) {
          tok = t;
        }
      }
    }
    const unsigned any = __ballot_sync(0xffffffffu, tok >= 0);
    if (!any) {
      if (lane < 16 && j0 + lane < T) key[(int64_t)i * T + j0 + lane] = __int_as_float(0x7fc00000);
      continue;
    }
    // gather the 16 K and V rows (zero rows for ineligible positions)
    for (int x = lane; x < 16 * (D / 8); x += 32) {
      const int r = x / (D / 8), ch = x - r * (D / 8);
      const int t = __shfl_sync(0xffffffffu, tok, r);   // every lane takes part
      const bool ok = t >= 0;
      const int64_t off = (head_row0 + (ok ? t : 0)) * D + ch * 8;
      const uint32_t so = (uint32_t)(r * RS + ch * 8) * 2u;
      cp_async16(kb + so, k + off, ok ? 16u : 0u);
      cp_async16(vb + so, v + off, ok ? 16u : 0u);
    }
    cp_commit();
    cp_wait<0>();
    __syncwarp();
    // R = K W^T: A = K tile (16 x D), B = W rows (output dims as N)
    float acc[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const int j8 = lane >> 3, r8 = lane & 7;
    const uint32_t a_addr = kb + (uint32_t)(((j8 & 1) * 8 + r8) * RS + (j8 >> 1) * 8) * 2u;
    const uint32_t w_addr = smem_u32(sm.w) + (uint32_t)(((j8 >> 1) * 8 + r8) * RS + (j8 & 1) * 8) * 2u;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a[4];
      ldsm_x4(a_addr + kk * 32u, a);
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        uint32_t b[4];
        ldsm_x4(w_addr + (uint32_t)(np * 16 * RS) * 2u + kk * 32u, b);
        mma_bf16(acc[2 * np], a[0], a[1], a[2], a[3], b[0], b[1]);
        mma_bf16(acc[2 * np + 1], a[0], a[1], a[2], a[3], b[2], b[3]);
      }
    }
    // eps per row: rows lane/4 (c0, c1) and lane/4 + 8 (c2, c3)
    const int gr = lane >> 2, tc = (lane & 3) * 2;
    const uint16_t* vrow0 = sm.vt[warp] + gr * RS;
    const uint16_t* vrow1 = sm.vt[warp] + (gr + 8) * RS;
    float e0 = 0.f, e1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const uint32_t v0 = *reinterpret_cast<const uint32_t*>(vrow0 + nt * 8 + tc);
      const uint32_t v1 = *reinterpret_cast<const uint32_t*>(vrow1 + nt * 8 + tc);
      const float d0 = bf16lo(v0) - acc[nt][0], d1 = bf16hi(v0) - acc[nt][1];
      const float d2 = bf16lo(v1) - acc[nt][2], d3 = bf16hi(v1) - acc[nt][3];
      e0 = fmaf(d0, d0, fmaf(d1, d1, e0));
      e1 = fmaf(d2, d2, fmaf(d3, d3, e1));
    }
    e0 += __shfl_xor_sync(0xffffffffu, e0, 1);
    e0 += __shfl_xor_sync(0xffffffffu, e0, 2);
    e1 += __shfl_xor_sync(0xffffffffu, e1, 1);
    e1 += __shfl_xor_sync(0xffffffffu, e1, 2);
    const int t0 = __shfl_sync(0xffffffffu, tok, gr), t1 = __shfl_sync(0xffffffffu, tok, gr + 8);
    if ((lane & 3) == 0) {
      const float nan = __int_as_float(0x7fc00000);
      if (j0 + gr < T) key[(int64_t)i * T + j0 + gr] = t0 >= 0 ? -e0 : nan;
      if (j0 + gr + 8 < T) key[(int64_t)i * T + j0 + gr + 8] = t1 >= 0 ? -e1 : nan;
    }
    __syncwarp();                        // the tile buffers are reused by the next gather
  }
  cp_wait<0>();
}

// Step 3 as a cache layout.  Head i keeps the K rows of all counts_i pool
// tokens at kstart_i = offsets_i + i * slack, the napprox_i approximated
// ones first (pool positions approx_pos[i, 0..napprox_i), ascending), then
// the exact ones in pool order; the V rows of the exact tokens go to
// vstart_i = offsets_i - approx_offsets_i + i * slack.  A warp takes 16
// output rows: lane r < 16 finds its row's token (the r-th exact position is
// r + m, m the number of approximated positions before it, found by binary
// search over the sorted approximated positions), then the warp copies the
// 16 K rows and the exact rows' V with 16-byte loads, 8 vectors in flight.
constexpr int kCompactThreads = 256;
constexpr int kCompactRows = (kCompactThreads / 32) * 16;     // output rows per CTA

__global__ void __launch_bounds__(kCompactThreads)
vector_compact_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v, int T,
                      const int32_t* __restrict__ kept_idx, const int32_t* __restrict__ counts,
                      const int64_t* __restrict__ offsets, const int32_t* __restrict__ apos,
                      const int32_t* __restrict__ acounts, const int64_t* __restrict__ aoffsets,
                      int slack, uint4* __restrict__ kc, int64_t kc_rows,
                      uint4* __restrict__ vc, int64_t vc_rows, int64_t* __restrict__ kstart,
                      int32_t* __restrict__ klen, int64_t* __restrict__ vstart,
                      int32_t* __restrict__ napprox, int* status) {
  constexpr int VPR = D * 2 / 16;                 // 16-byte vectors per bf16 row
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cnt = counts[i], na = acounts[i];
  const int64_t ks = offsets[i] + (int64_t)i * slack;
  const int64_t vs = offsets[i] - aoffsets[i] + (int64_t)i * slack;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    kstart[i] = ks;
    klen[i] = cnt;
    vstart[i] = vs;
    napprox[i] = na;
  }
  if (na < 0 || na > cnt || cnt > T) {
    if (threadIdx.x == 0 && blockIdx.x == 0) report(status, KVC_ERR_RANGE);
    return;
  }
  const int o0 = blockIdx.x * kCompactRows + warp * 16;
  if (o0 >= cnt) return;
  const int32_t* ap = apos + (int64_t)i * T;
  int64_t src = -1, kdst = -1, vdst = -1;
  const int o = o0 + lane;
  if (lane < 16 && o < cnt) {
    int j;
    int64_t vd = -1;
    if (o < na) {
      j = ap[o];
    } else {
      const int r = o - na;
      int lo = 0, hi = na;                        // smallest m with ap[m] > r + m (or m = na)
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (ap[mid] > r + mid) hi = mid; else lo = mid + 1;
      }
      j = r + lo;
      vd = vs + r;
    }
    const int t = (j >= 0 && j < cnt) ? kept_idx[(int64_t)i * T + j] : -1;
    const bool v_bad = o >= na && (vd < 0 || vd >= vc_rows);   // exact rows need a V row
    if (t < 0 || t >= T || ks + o < 0 || ks + o >= kc_rows || v_bad) {
      report(status, KVC_ERR_RANGE);
    } else {
      src = (int64_t)i * T + t;
      kdst = ks + o;
      vdst = vd;
    }
  }
  const int nrows = min(cnt - o0, 16);
  const int pairs = nrows * VPR;
  for (int p0 = 0; p0 < pairs; p0 += 32 * 8) {
    uint4 kv[8], vv[8];
    int64_t kd[8], vd[8];
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const int p = p0 + x * 32 + lane;
      const int row = (p / VPR) & 15, vec = p % VPR;
      const int64_t s_row = __shfl_sync(0xffffffffu, src, row);
      const int64_t k_row = __shfl_sync(0xffffffffu, kdst, row);
      const int64_t v_row = __shfl_sync(0xffffffffu, vdst, row);
      kd[x] = vd[x] = -1;
      if (p < pairs && s_row >= 0) {
        kv[x] = __ldg(k + s_row * VPR + vec);
        kd[x] = k_row * VPR + vec;
        if (v_row >= 0) {
          vv[x] = __ldg(v + s_row * VPR + vec);
          vd[x] = v_row * VPR + vec;
        }
      }
    }
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      if (kd[x] >= 0) kc[kd[x]] = kv[x];
      if (vd[x] >= 0) vc[vd[x]] = vv[x];
    }
  }
}

}  // namespace

int vector_residual_launch(const void* k, const void* v, const void* W, int U, int Hkv, int T,
                           const int32_t* kept_idx, const int32_t* counts, int n_sink,
                           int n_recent, float* key, const Dev& dev, cudaStream_t s) {
  const int n = U * Hkv;
  if (n == 0 || T == 0) return KVC_OK;
  const size_t smem = sizeof(ResidualSmem);
  static std::atomic<uint32_t> attr_done{0};
  const uint32_t bit = 1u << (dev.device & 31);
  if (!(attr_done.load() & bit)) {
    KVC_CUDA_TRY(cudaFuncSetAttribute(vector_residual_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr_done.fetch_or(bit);
  }
  if (int rc = prefer_max_shared(vector_residual_kernel, dev.device)) return rc;
  // about two CTAs per SM over all heads; each CTA stages its head's W once
  const int ntiles = (T + kTile - 1) / kTile;
  int per_head = (2 * dev.sms + n - 1) / n;
  if (per_head > ntiles) per_head = ntiles;
  if (per_head < 1) per_head = 1;
  return launch_pdl(vector_residual_kernel, dim3((unsigned)per_head, (unsigned)n),
                    dim3(kResWarps * 32), smem, s, static_cast<const uint16_t*>(k),
                    static_cast<const uint16_t*>(v), static_cast<const uint16_t*>(W), Hkv, T,
                    kept_idx, counts, n_sink, n_recent, key, dev.status);
}

int vector_compact_launch(const void* k, const void* v, int U, int Hkv, int T,
                          const int32_t* kept_idx, const int32_t* counts,
                          const int64_t* offsets, const int32_t* approx_pos,
                          const int32_t* approx_counts, const int64_t* approx_offsets, int slack,
                          void* kc, int64_t kc_rows, void* vc, int64_t vc_rows, int64_t* kstart,
                          int32_t* klen, int64_t* vstart, int32_t* napprox, const Dev& dev,
                          cudaStream_t s) {
  const int n = U * Hkv;
  if (n == 0 || T == 0) return KVC_OK;
  const dim3 grid((unsigned)((T + kCompactRows - 1) / kCompactRows), (unsigned)n);
  return launch_pdl(vector_compact_kernel, grid, dim3(kCompactThreads), 0, s,
                    static_cast<const uint4*>(k), static_cast<const uint4*>(v), T, kept_idx,
                    counts, offsets, approx_pos, approx_counts, approx_offsets, slack,
                    static_cast<uint4*>(kc), kc_rows, static_cast<uint4*>(vc), vc_rows, kstart,
                    klen, vstart, napprox, dev.status);
}

}  // namespace kvc
