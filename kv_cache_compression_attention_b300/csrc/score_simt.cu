// Attention-mass scoring on the SIMT cores (fp32 inputs, and any shape the
// tensor-core kernel does not cover).
//
// Definition (KVSculpt §1 / §2B; KVzap §2.1): for unit u, kv head g, query
// head h in g and window row w, s[(h,w),t] = scale*f[u,h]*<q[u,h,w], k[u,g,t]>
// over t <= T-W+w (causal) and score[u,g,t] = sum_{h,w} softmax_t(s)[t].
//
// Two kernels:
//   row_lse   one warp per window row: the row's log-sum-exp over its tokens
//             (online max/sum per lane, merged across the warp);
//   col_mass  one thread per token: sum over the group's rows of
//             exp(s - lse_row), rows staged through shared memory.
// Accumulation and exponentials are fp32 (expf/logf), which keeps the
// fp32 path within 1e-4 relative of the float64 definition.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

template <typename Tin>
__device__ __forceinline__ void load_row(const Tin* p, int d, float* dst);

template <>
__device__ __forceinline__ void load_row<float>(const float* p, int d, float* dst) {
  const float4* p4 = reinterpret_cast<const float4*>(p);
  for (int x = 0; x < d / 4; ++x) {
    float4 v = __ldg(p4 + x);
    dst[4 * x] = v.x; dst[4 * x + 1] = v.y; dst[4 * x + 2] = v.z; dst[4 * x + 3] = v.w;
  }
}

template <>
__device__ __forceinline__ void load_row<uint16_t>(const uint16_t* p, int d, float* dst) {
  const uint4* p4 = reinterpret_cast<const uint4*>(p);
  for (int x = 0; x < d / 8; ++x) {
    uint4 v = __ldg(p4 + x);
    dst[8 * x + 0] = bf16lo(v.x); dst[8 * x + 1] = bf16hi(v.x);
    dst[8 * x + 2] = bf16lo(v.y); dst[8 * x + 3] = bf16hi(v.y);
    dst[8 * x + 4] = bf16lo(v.z); dst[8 * x + 5] = bf16hi(v.z);
    dst[8 * x + 6] = bf16lo(v.w); dst[8 * x + 7] = bf16hi(v.w);
  }
}

template <typename Tin>
__device__ __forceinline__ float load_elem(const Tin* p, int x);
template <>
__device__ __forceinline__ float load_elem<float>(const float* p, int x) { return __ldg(p + x); }
template <>
__device__ __forceinline__ float load_elem<uint16_t>(const uint16_t* p, int x) {
  return __uint_as_float(((uint32_t)__ldg(p + x)) << 16);
}

constexpr int kRowWarps = 8;

// lse[(u*Hq + h)*W + w] for every window row.
template <typename Tin, int D>
__global__ void __launch_bounds__(kRowWarps * 32)
row_lse_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, int U, int Hq, int Hkv,
               int T, int W, float scale, const float* __restrict__ head_scale, int causal,
               float* __restrict__ lse, int* status) {
  __shared__ float qs[kRowWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kRowWarps + warp;
  const int64_t rows = (int64_t)U * Hq * W;
  if (row >= rows) return;
  const int w = (int)(row % W);
  const int h = (int)((row / W) % Hq);
  const int u = (int)(row / ((int64_t)W * Hq));
  const int G = Hq / Hkv, g = h / G;
  const float f = head_scale ? head_scale[(int64_t)u * Hq + h] : 1.0f;
  if (lane == 0 && !(f > 0.0f && f < INFINITY)) report(status, KVC_ERR_INVALID);
  const float c = scale * f;
  for (int x = lane; x < D; x += 32) qs[warp][x] = load_elem<Tin>(q + row * D, x);
  __syncwarp();
  const int last = causal ? (T - W + w) : (T - 1);
  const Tin* kb = k + ((int64_t)u * Hkv + g) * (int64_t)T * D;
  float m = -INFINITY, l = 0.0f;
  for (int t = lane; t <= last; t += 32) {
    float kr[D];
    load_row<Tin>(kb + (int64_t)t * D, D, kr);
    float acc = 0.0f;
#pragma unroll
    for (int x = 0; x < D; ++x) acc = fmaf(qs[warp][x], kr[x], acc);
    const float s = c * acc;
    if (s > m) { l = l * expf(m - s) + 1.0f; m = s; }
    else       { l += expf(s - m); }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    float l2 = __shfl_xor_sync(0xffffffffu, l, off);
    float mn = fmaxf(m, m2);
    float a = (m == -INFINITY) ? 0.0f : l * expf(m - mn);
    float b = (m2 == -INFINITY) ? 0.0f : l2 * expf(m2 - mn);
    m = mn; l = a + b;
  }
  if (lane == 0) lse[row] = m + logf(l);
}

constexpr int kColThreads = 128;
constexpr int kRowChunk = 32;

// One thread per token t of (u, g): score = sum_r exp(c_r * <q_r, k_t> - lse_r).
template <typename Tin, int D>
__global__ void __launch_bounds__(kColThreads)
col_mass_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k, int U, int Hq, int Hkv,
                int T, int W, float scale, const float* __restrict__ head_scale, int causal,
                int agg_max, const float* __restrict__ lse, float* __restrict__ scores,
                const float* __restrict__ hnorm, const float* __restrict__ vnorm) {
  __shared__ float4 qs[kRowChunk][D / 4];
  __shared__ float cs[kRowChunk], ls[kRowChunk];
  const int ug = blockIdx.y;                 // u*Hkv + g
  const int u = ug / Hkv, g = ug % Hkv;
  const int G = Hq / Hkv, R = G * W;
  const int t = blockIdx.x * kColThreads + threadIdx.x;
  const bool valid = t < T;
  float kr[D];
  if (valid) load_row<Tin>(k + ((int64_t)ug * T + t) * D, D, kr);
  float sum = 0.0f;
  const int64_t row0 = ((int64_t)u * Hq + (int64_t)g * G) * W;   // first row of the group
  // KVzip+ (vnorm set): a head's largest weight over its rows, each divided
  // by the row's hidden-state norm (folded into the row's normaliser), times
  // the token's value contribution ||W_O^h v_t||; the maximum over heads
  const bool plus = vnorm != nullptr;
  int cur_h = 0;
  float hmax = 0.0f;
  for (int r0 = 0; r0 < R; r0 += kRowChunk) {
    const int nr = min(kRowChunk, R - r0);
    __syncthreads();
    for (int e = threadIdx.x; e < nr * D; e += kColThreads) {
      const int rr = e / D, x = e % D;
      reinterpret_cast<float*>(qs[rr])[x] = load_elem<Tin>(q + (row0 + r0 + rr) * D, x);
    }
    if (threadIdx.x < nr) {
      const int r = r0 + threadIdx.x;
      const int h = g * G + r / W;
      cs[threadIdx.x] = scale * (head_scale ? head_scale[(int64_t)u * Hq + h] : 1.0f);
      ls[threadIdx.x] = lse[row0 + r] + (plus ? logf(hnorm[(int64_t)u * W + r % W]) : 0.0f);
    }
    __syncthreads();
    if (valid) {
      for (int rr = 0; rr < nr; ++rr) {
        const int w = (r0 + rr) % W;
        if (plus && (r0 + rr) / W != cur_h) {
          sum = fmaxf(sum, hmax * vnorm[((int64_t)u * Hq + g * G + cur_h) * T + t]);
          hmax = 0.0f;
          cur_h = (r0 + rr) / W;
        }
        if (causal && t > T - W + w) continue;
        float acc = 0.0f;
#pragma unroll
        for (int x4 = 0; x4 < D / 4; ++x4) {
          const float4 qv = qs[rr][x4];
          acc = fmaf(qv.x, kr[4 * x4], acc);
          acc = fmaf(qv.y, kr[4 * x4 + 1], acc);
          acc = fmaf(qv.z, kr[4 * x4 + 2], acc);
          acc = fmaf(qv.w, kr[4 * x4 + 3], acc);
        }
        const float e = expf(cs[rr] * acc - ls[rr]);
        if (plus) hmax = fmaxf(hmax, e);
        else sum = agg_max ? fmaxf(sum, e) : sum + e;
      }
    }
  }
  if (valid && plus) sum = fmaxf(sum, hmax * vnorm[((int64_t)u * Hq + g * G + cur_h) * T + t]);
  if (valid) scores[(int64_t)ug * T + t] = sum;
}

template <typename Tin, int D>
int run(const void* q, const void* k, int U, int Hq, int Hkv, int T, int W, float scale,
        const float* hs, int causal, int agg, float* scores, float* lse, int* status,
        cudaStream_t s, const float* hnorm = nullptr, const float* vnorm = nullptr) {
  const int64_t rows = (int64_t)U * Hq * W;
  dim3 g1((unsigned)((rows + kRowWarps - 1) / kRowWarps));
  row_lse_kernel<Tin, D><<<g1, kRowWarps * 32, 0, s>>>(
      static_cast<const Tin*>(q), static_cast<const Tin*>(k), U, Hq, Hkv, T, W, scale, hs,
      causal, lse, status);
  dim3 g2((unsigned)((T + kColThreads - 1) / kColThreads), (unsigned)(U * Hkv));
  col_mass_kernel<Tin, D><<<g2, kColThreads, 0, s>>>(
      static_cast<const Tin*>(q), static_cast<const Tin*>(k), U, Hq, Hkv, T, W, scale, hs,
      causal, agg == KVC_AGG_MAX ? 1 : 0, lse, scores, hnorm, vnorm);
  return launch_status();
}

}  // namespace

int score_kvzip_plus_simt(const void* q, const void* k, int U, int Hq, int Hkv, int T, int W,
                          float scale, const float* head_scale, int causal, const float* hnorm,
                          const float* vnorm, float* scores, float* lse_ws, const Dev& dev,
                          cudaStream_t s) {
  return run<uint16_t, 128>(q, k, U, Hq, Hkv, T, W, scale, head_scale, causal, KVC_AGG_MAX,
                            scores, lse_ws, dev.status, s, hnorm, vnorm);
}

size_t score_attn_simt_ws(int U, int Hq, int W) {
  return (size_t)U * Hq * W * sizeof(float);
}

int score_attn_simt(const void* q, const void* k, int dtype, int U, int Hq, int Hkv, int T,
                    int W, int d, float scale, const float* head_scale, int causal, int agg,
                    float* scores, float* lse_ws, const Dev& dev, cudaStream_t s) {
  if (dtype == KVC_F32) {
    return d == 64 ? run<float, 64>(q, k, U, Hq, Hkv, T, W, scale, head_scale, causal, agg, scores, lse_ws, dev.status, s)
                   : run<float, 128>(q, k, U, Hq, Hkv, T, W, scale, head_scale, causal, agg, scores, lse_ws, dev.status, s);
  }
  return d == 64 ? run<uint16_t, 64>(q, k, U, Hq, Hkv, T, W, scale, head_scale, causal, agg, scores, lse_ws, dev.status, s)
                 : run<uint16_t, 128>(q, k, U, Hq, Hkv, T, W, scale, head_scale, causal, agg, scores, lse_ws, dev.status, s);
}

}  // namespace kvc
