// Fidelity probe (KVSculpt §4: fidelity of a compressed cache is measured as
// a KL divergence) and the self-test of the bounded device waits.
//
//   rel_err[r] = ||out_comp[r] - out_full[r]||_2 / ||out_full[r]||_2
//   kl[r]      = lse_full[r] - lse_comp[r]  (= KL(p_comp || p_full) because
//                the compressed rows are a subset of the full rows)
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kThreads = 128;

template <typename Tin>
__device__ __forceinline__ float ld(const Tin* p, int64_t i);
template <>
__device__ __forceinline__ float ld<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld<uint16_t>(const uint16_t* p, int64_t i) {
  return __uint_as_float(((uint32_t)p[i]) << 16);
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
fidelity_kernel(const Tin* __restrict__ oc, const Tin* __restrict__ of,
                const float* __restrict__ lc, const float* __restrict__ lf, int d,
                float* __restrict__ rel, float* __restrict__ kl) {
  __shared__ float red[2][kThreads / 32];
  const int64_t r = blockIdx.x;
  float num = 0.0f, den = 0.0f;
  for (int x = threadIdx.x; x < d; x += kThreads) {
    const float a = ld(oc, r * d + x), b = ld(of, r * d + x);
    num = fmaf(a - b, a - b, num);
    den = fmaf(b, b, den);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    num += __shfl_xor_sync(0xffffffffu, num, off);
    den += __shfl_xor_sync(0xffffffffu, den, off);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { red[0][warp] = num; red[1][warp] = den; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float n = 0.0f, dd = 0.0f;
    for (int w = 0; w < kThreads / 32; ++w) { n += red[0][w]; dd += red[1][w]; }
    rel[r] = dd > 0.0f ? sqrtf(n / dd) : sqrtf(n);
    kl[r] = lf[r] - lc[r];
  }
}

// Waits on an mbarrier that nothing will ever complete; the bounded wait
// gives up after timeout_ns and records KVC_ERR_TIMEOUT.
__global__ void wait_selftest_kernel(uint64_t timeout_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
  }
  __syncthreads();
  mbar_wait(&bar, 0, status, &abort_flag, timeout_ns);
  __syncthreads();
}

}  // namespace

int fidelity_launch(const void* oc, const void* of, const float* lc, const float* lf,
                    int dtype, int n, int d, float* rel, float* kl, const Dev& dev,
                    cudaStream_t s) {
  (void)dev;
  if (dtype == KVC_F32)
    fidelity_kernel<float><<<n, kThreads, 0, s>>>(static_cast<const float*>(oc),
                                                  static_cast<const float*>(of), lc, lf, d, rel, kl);
  else
    fidelity_kernel<uint16_t><<<n, kThreads, 0, s>>>(static_cast<const uint16_t*>(oc),
                                                     static_cast<const uint16_t*>(of), lc, lf, d,
                                                     rel, kl);
  return launch_status();
}

int selftest_wait_launch(uint64_t timeout_ns, const Dev& dev, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(timeout_ns, dev.status);
  return launch_status();
}

}  // namespace kvc
