// KVzip+ score (KVzap: Fast, Adaptive, and Faithful KV Cache Pruning, §2.1):
// the largest attention weight a token receives from the window rows, each
// weighted by the token's value contribution to the residual stream,
// ||W_O^h v_t||, over the row's hidden-state norm ||h_w||.
//
//   value_norm_kernel   ||W_O^h v_t|| = sqrt(v_t^T M_h v_t) for every query
//                       head h and token t, with M_h = W_O^h^T W_O^h the d x d
//                       Gram matrix of the output projection's slice for
//                       head h (part of the model's weights, formed offline):
//                       a d x d contraction per (head, token) on warp-level
//                       bf16 MMAs, M_h staged per head in shared memory;
//   then the scoring pass in its KVzip+ mode (per-head maxima of a_wt /
//   ||h_w||, times the value norm, maximum over heads): the tensor-core
//   scorer where each quarter of its pass-2 columns is one head's rows (the
//   row norm folds into the row normaliser, the value norm scales the
//   quarter's maximum), else the SIMT column pass.
#include <atomic>

#include "kvc_internal.cuh"
#include "mma_sync.cuh"

namespace kvc {
namespace {

using namespace ::kvc::mmasync;

constexpr int D = 128;
constexpr int RS = D + 8;            // padded smem row (bf16): conflict-free ldmatrix
constexpr int kWarps = 4;            // 16 tokens per warp
constexpr int kTokens = kWarps * 16;

struct NormSmem {
  uint16_t m[D * RS];                // M_h
  uint16_t vt[kWarps][16 * RS];      // each warp's 16 value rows
};

// grid (ceil(T / 64), U * Hkv); CTA: 64 tokens of one (unit, kv head), all G
// of its query heads
__global__ void __launch_bounds__(kWarps * 32)
value_norm_kernel(const uint16_t* __restrict__ v, const uint16_t* __restrict__ gram, int Hkv,
                  int G, int T, float* __restrict__ vnorm) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  NormSmem& sm = *reinterpret_cast<NormSmem*>(smem_raw);
  const int ug = blockIdx.y;
  const int u = ug / Hkv, g = ug - u * Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * kTokens + warp * 16;
  const uint32_t mb = smem_u32(sm.m), vb = smem_u32(sm.vt[warp]);
  pdl_wait();
  pdl_trigger();
  // this warp's 16 value rows (zero rows past T)
  for (int x = lane; x < 16 * (D / 8); x += 32) {
    const int r = x / (D / 8), ch = x - r * (D / 8);
    const bool ok = t0 + r < T;
    const int64_t off = ((int64_t)ug * T + (ok ? t0 + r : 0)) * D + ch * 8;
    cp_async16(vb + (uint32_t)(r * RS + ch * 8) * 2u, v + off, ok ? 16u : 0u);
  }
  cp_commit();
  const int j8 = lane >> 3, r8 = lane & 7;
  const uint32_t a_addr = vb + (uint32_t)(((j8 & 1) * 8 + r8) * RS + (j8 >> 1) * 8) * 2u;
  const uint32_t b_addr = mb + (uint32_t)(((j8 >> 1) * 8 + r8) * RS + (j8 & 1) * 8) * 2u;
  const int gr = lane >> 2, tc = (lane & 3) * 2;
  for (int hh = 0; hh < G; ++hh) {
    const int h = g * G + hh;
    __syncthreads();                       // every warp is done with the previous M_h
    const uint16_t* mh = gram + (int64_t)h * D * D;
    for (int x = threadIdx.x; x < D * (D / 8); x += kWarps * 32) {
      const int r = x / (D / 8), ch = x - r * (D / 8);
      cp_async16(mb + (uint32_t)(r * RS + ch * 8) * 2u, mh + r * D + ch * 8, 16u);
    }
    cp_commit();
    cp_wait<0>();
    __syncthreads();
    // R = V M_h (M_h symmetric: its rows serve as the N x K operand)
    float acc[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a[4];
      ldsm_x4(a_addr + kk * 32u, a);
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        uint32_t b[4];
        ldsm_x4(b_addr + (uint32_t)(np * 16 * RS) * 2u + kk * 32u, b);
        mma_bf16(acc[2 * np], a[0], a[1], a[2], a[3], b[0], b[1]);
        mma_bf16(acc[2 * np + 1], a[0], a[1], a[2], a[3], b[2], b[3]);
      }
    }
    // f^2 = v . R per row: rows gr (c0, c1) and gr + 8 (c2, c3)
    const uint16_t* v0 = sm.vt[warp] + gr * RS;
    const uint16_t* v1 = sm.vt[warp] + (gr + 8) * RS;
    float e0 = 0.f, e1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const uint32_t w0 = *reinterpret_cast<const uint32_t*>(v0 + nt * 8 + tc);
      const uint32_t w1 = *reinterpret_cast<const uint32_t*>(v1 + nt * 8 + tc);
      e0 = fmaf(bf16lo(w0), acc[nt][0], fmaf(bf16hi(w0), acc[nt][1], e0));
      e1 = fmaf(bf16lo(w1), acc[nt][2], fmaf(bf16hi(w1), acc[nt][3], e1));
    }
    e0 += __shfl_xor_sync(0xffffffffu, e0, 1);
    e0 += __shfl_xor_sync(0xffffffffu, e0, 2);
    e1 += __shfl_xor_sync(0xffffffffu, e1, 1);
    e1 += __shfl_xor_sync(0xffffffffu, e1, 2);
    if ((lane & 3) == 0) {
      float* out = vnorm + ((int64_t)u * Hkv * G + h) * T;
      if (t0 + gr < T) out[t0 + gr] = sqrtf(fmaxf(e0, 0.0f));
      if (t0 + gr + 8 < T) out[t0 + gr + 8] = sqrtf(fmaxf(e1, 0.0f));
    }
  }
  cp_wait<0>();
}

}  // namespace

namespace {
// the tensor-core scorer takes the KVzip+ mode when each quarter of its
// pass-2 columns lies inside one query head's rows
bool kvzip_tc(int Hq, int Hkv, int W) {
  const int R = (Hq / Hkv) * W;
  return score_attn_tc_supported(KVC_BF16, Hq, Hkv, W, 128) && W % (R / 4) == 0;
}
size_t vn_bytes(int U, int Hq, int T) {
  return (((size_t)U * Hq * T * sizeof(float)) + 255) & ~(size_t)255;
}
}  // namespace

size_t score_kvzip_plus_ws_bytes(int U, int Hq, int Hkv, int T, int W) {
  const size_t simt = score_attn_simt_ws(U, Hq, W);
  const size_t tc = kvzip_tc(Hq, Hkv, W) ? score_attn_tc_ws(Hq, Hkv, W) : 0;
  return vn_bytes(U, Hq, T) + (simt > tc ? simt : tc);
}

int score_kvzip_plus_launch(const void* q, const void* k, const void* v, const void* gram,
                            const float* hnorm, int U, int Hq, int Hkv, int T, int W,
                            float scale, const float* head_scale, int causal, float* scores,
                            void* workspace, const Dev& dev, cudaStream_t s) {
  if (U == 0 || T == 0) return KVC_OK;
  float* vnorm = static_cast<float*>(workspace);
  uint8_t* rest = static_cast<uint8_t*>(workspace) + vn_bytes(U, Hq, T);
  const size_t smem = sizeof(NormSmem);
  static std::atomic<uint32_t> attr_done{0};
  const uint32_t bit = 1u << (dev.device & 31);
  if (!(attr_done.load() & bit)) {
    KVC_CUDA_TRY(cudaFuncSetAttribute(value_norm_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr_done.fetch_or(bit);
  }
  const dim3 grid((unsigned)((T + kTokens - 1) / kTokens), (unsigned)(U * Hkv));
  if (int rc = launch_pdl(value_norm_kernel, grid, dim3(kWarps * 32), smem, s,
                          static_cast<const uint16_t*>(v), static_cast<const uint16_t*>(gram),
                          Hkv, Hq / Hkv, T, vnorm))
    return rc;
  const bool aligned = ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k)) & 15u) == 0;
  if (aligned && kvzip_tc(Hq, Hkv, W))
    return score_attn_tc(q, k, U, Hq, Hkv, T, W, scale, head_scale, causal, kAggKvzipPlus, scores,
                         rest, dev, s, hnorm, vnorm);
  return score_kvzip_plus_simt(q, k, U, Hq, Hkv, T, W, scale, head_scale, causal, hnorm, vnorm,
                               scores, reinterpret_cast<float*>(rest), dev, s);
}

}  // namespace kvc
