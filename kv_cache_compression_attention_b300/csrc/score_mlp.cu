// Two-layer surrogate scorer (KVzap: Fast, Adaptive, and Faithful KV Cache
// Pruning, §2.2, the MLP variant: hidden width Dh / 8 with a GELU):
//   z[r, m]      = b1[m] + hidden[r, :] . W1[:, m]        (r = u * T + t)
//   score[u,g,t] = b2[g] + sum_m GELU(z[r, m]) W2[m, g]
//
// The first layer is a plain dense GEMM (131072 x 3584 x 448 on the 128k
// layer, 421 GFLOP): it runs as a cuBLAS bf16 GEMM with fp32 accumulation
// into a bf16 intermediate held in the caller's workspace.  The bias, the
// exact GELU and the second layer (Dm x Hkv, a few multiply-adds per
// element) run in one streaming pass over that intermediate: a warp per row,
// 16-byte loads, W2 and b1 in shared memory, the Hkv sums reduced by shuffles.
#include <cublas_v2.h>

#include <atomic>
#include <mutex>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxDm = 1024;
constexpr size_t kCublasWs = (size_t)32 << 20;     // cuBLAS scratch inside the workspace

template <int HK>
__global__ void __launch_bounds__(kThreads)
mlp_out_kernel(const uint16_t* __restrict__ pre, const float* __restrict__ b1,
               const uint16_t* __restrict__ w2, const float* __restrict__ b2, int64_t rows,
               int T, int Dm, float* __restrict__ scores) {
  __shared__ float w2s[kMaxDm * HK];
  __shared__ float b1s[kMaxDm];
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < Dm * HK; e += kThreads) w2s[e] = bf16lo(w2[e]);
  for (int e = threadIdx.x; e < Dm; e += kThreads) b1s[e] = b1 ? b1[e] : 0.0f;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int nch = Dm / 8;                        // 16-byte chunks per row
  const int64_t warp0 = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
  for (int64_t r = warp0; r < rows; r += nwarps) {
    const uint4* prow = reinterpret_cast<const uint4*>(pre + r * Dm);
    float acc[HK];
#pragma unroll
    for (int g = 0; g < HK; ++g) acc[g] = 0.0f;
    for (int c = lane; c < nch; c += 32) {
      const uint4 w = __ldg(prow + c);
      const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int m = c * 8 + e;
        const float z = ((e & 1) ? bf16hi(wv[e >> 1]) : bf16lo(wv[e >> 1])) + b1s[m];
        const float a = 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
#pragma unroll
        for (int g = 0; g < HK; ++g) acc[g] = fmaf(a, w2s[m * HK + g], acc[g]);
      }
    }
#pragma unroll
    for (int g = 0; g < HK; ++g) {
      float v = acc[g];
#pragma unroll
      for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      acc[g] = v;
    }
    if (lane < HK) {
      float v = 0.0f;
#pragma unroll
      for (int g = 0; g < HK; ++g) v = (lane == g) ? acc[g] : v;
      const int64_t u = r / T, t = r - u * T;
      scores[(u * HK + lane) * (int64_t)T + t] = v + (b2 ? b2[lane] : 0.0f);
    }
  }
}

// One cuBLAS handle per device, created on first use and kept for the
// process.  Setting its stream and workspace and enqueuing the GEMM happen
// under the same lock, so host threads sharing a device do not race on them.
std::mutex& handle_mutex() {
  static std::mutex mu;
  return mu;
}

cublasHandle_t handle_for(int device) {
  static cublasHandle_t handles[64] = {};
  cublasHandle_t& h = handles[device & 63];
  if (!h && cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) h = nullptr;
  return h;
}

template <int HK>
int launch_out(const uint16_t* pre, const float* b1, const uint16_t* w2, const float* b2,
               int64_t rows, int T, int Dm, float* scores, const Dev& dev, cudaStream_t s) {
  const int64_t want = (rows + kThreads / 32 - 1) / (kThreads / 32);
  const int64_t cap = (int64_t)dev.sms * 8;
  const unsigned blocks = (unsigned)(want < cap ? want : cap);
  return launch_pdl(mlp_out_kernel<HK>, dim3(blocks), dim3(kThreads), 0, s, pre, b1, w2, b2,
                    rows, T, Dm, scores);
}

}  // namespace

size_t score_mlp_ws_bytes(int U, int T, int Dm) {
  const size_t inter = (((size_t)U * T * Dm * 2) + 255) & ~(size_t)255;
  return inter + kCublasWs;
}

int score_mlp_launch(const void* hidden, const void* w1, const float* b1, const void* w2,
                     const float* b2, int U, int T, int Dh, int Dm, int Hkv, float* scores,
                     void* workspace, const Dev& dev, cudaStream_t s) {
  const int64_t rows = (int64_t)U * T;
  if (rows == 0) return KVC_OK;
  if (Dm > kMaxDm) return KVC_ERR_UNSUPPORTED;
  if (rows > 0x7fffffffLL) return KVC_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint16_t* pre = reinterpret_cast<uint16_t*>(ws);
  void* cws = ws + (score_mlp_ws_bytes(U, T, Dm) - kCublasWs);
  {
    std::lock_guard<std::mutex> lock(handle_mutex());
    cublasHandle_t h = handle_for(dev.device);
    if (!h) return KVC_ERR_CUDA;
    if (cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS) return KVC_ERR_CUDA;
    if (cublasSetWorkspace(h, cws, kCublasWs) != CUBLAS_STATUS_SUCCESS) return KVC_ERR_CUDA;
    // row-major pre [rows, Dm] = hidden [rows, Dh] . W1 [Dh, Dm], i.e. in the
    // column-major terms of cuBLAS pre^T (Dm x rows) = W1^T (Dm x Dh) . hidden^T
    const float one = 1.0f, zero = 0.0f;
    if (cublasGemmEx(h, CUBLAS_OP_N, CUBLAS_OP_N, Dm, (int)rows, Dh, &one, w1, CUDA_R_16BF, Dm,
                     hidden, CUDA_R_16BF, Dh, &zero, pre, CUDA_R_16BF, Dm, CUBLAS_COMPUTE_32F,
                     CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
      return KVC_ERR_CUDA;
  }
  const uint16_t* w2b = static_cast<const uint16_t*>(w2);
  switch (Hkv) {
    case 1: return launch_out<1>(pre, b1, w2b, b2, rows, T, Dm, scores, dev, s);
    case 2: return launch_out<2>(pre, b1, w2b, b2, rows, T, Dm, scores, dev, s);
    case 3: return launch_out<3>(pre, b1, w2b, b2, rows, T, Dm, scores, dev, s);
    case 4: return launch_out<4>(pre, b1, w2b, b2, rows, T, Dm, scores, dev, s);
    case 5: return launch_out<5>(pre, b1, w2b, b2, rows, T, Dm, scores, dev, s);
    case 6: return launch_out<6>(pre, b1, w2b, b2, rows, T, Dm, scores, dev, s);
    case 7: return launch_out<7>(pre, b1, w2b, b2, rows, T, Dm, scores, dev, s);
    case 8: return launch_out<8>(pre, b1, w2b, b2, rows, T, Dm, scores, dev, s);
  }
  return KVC_ERR_UNSUPPORTED;
}

}  // namespace kvc
