// Linear surrogate scorer (KVzap §2.2): score[u,g,t] = bias[g] + h[u,t,:] . W[:,g].
//
// A streaming GEMV-like pass: every hidden row (Dh = 3584 bf16 = 7 KiB) is
// read once from HBM with 16-byte coalesced loads and dotted with the Hkv
// weight columns held in shared memory.  Work is 2*Hkv flops per hidden
// element (8 per 16 bytes at Hkv = 4): bandwidth bound, so the kernel is
// SIMT FFMA, not a tensor-core GEMM.
//
// Mapping: a warp owns 4 consecutive rows and reads 1 KiB of each per
// iteration (two 512-byte column blocks: lane L takes the 16-byte chunks L
// and L + 32 of the pair); for each chunk it loads the matching weight slice
// once from shared memory (laid out chunk-interleaved so a warp's 32 loads
// hit 32 consecutive 16-byte words) and applies it to all 4 rows.  Each lane
// streams its 16-byte pieces of the next three iterations into a private
// shared-memory ring with cp.async, so 12 warps keep ~144 KB of reads per SM
// in flight without holding them in registers.  (1 KiB per row and
// iteration measured 1-2 % faster than 512 bytes for 8 rows, 2 KiB for 2
// rows slower.)  The 4 x Hkv partial sums are reduced across the warp with
// xor-shuffles at the end.
#include <atomic>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kCPR = 2;         // 512-byte column blocks of a row per iteration
constexpr int kRows = 8 / kCPR; // rows per warp task
constexpr int kWarps = 12;      // one block per SM
constexpr int kStages = 3;      // column blocks in flight per warp
constexpr int kBlockBytes = 32 * 16;   // one row's column block: 32 lanes x 16 bytes

template <typename Tin> struct Vec;
template <> struct Vec<uint16_t> { static constexpr int E = 8; };
template <> struct Vec<float> { static constexpr int E = 4; };

__device__ __forceinline__ void unpack(const uint4& v, float* x, uint16_t) {
  x[0] = bf16lo(v.x); x[1] = bf16hi(v.x); x[2] = bf16lo(v.y); x[3] = bf16hi(v.y);
  x[4] = bf16lo(v.z); x[5] = bf16hi(v.z); x[6] = bf16lo(v.w); x[7] = bf16hi(v.w);
}
__device__ __forceinline__ void unpack(const uint4& v, float* x, float) {
  x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
  x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
}

__device__ __forceinline__ float to_f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }
__device__ __forceinline__ float to_f(float f) { return f; }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}

template <typename Tin, int HK>
__global__ void __launch_bounds__(kWarps * 32, 1)
linear_kernel(const Tin* __restrict__ hidden, const Tin* __restrict__ weight,
              const float* __restrict__ bias, int64_t rows, int T, int Dh,
              float* __restrict__ scores) {
  constexpr int E = Vec<Tin>::E;          // hidden elements per 16-byte chunk
  constexpr int F4 = E * HK / 4;          // float4 words of weight per chunk
  extern __shared__ __align__(128) uint8_t smem_lin[];
  pdl_wait();
  pdl_trigger();
  const int NC = Dh / E;
  const int NIT = (NC + 32 * kCPR - 1) / (32 * kCPR);   // iterations per row
  float4* wsm = reinterpret_cast<float4*>(smem_lin);                    // [F4][NC]
  uint8_t* ring = smem_lin + (((size_t)F4 * NC * 16 + 127) & ~size_t(127));
  // stage the weight: chunk c, element jj, head g -> float (jj*HK + g) of chunk c
  for (int e = threadIdx.x; e < Dh * HK; e += blockDim.x) {
    const int j = e / HK, g = e % HK;
    const int c = j / E, jj = j % E;
    const int f = jj * HK + g;
    reinterpret_cast<float*>(&wsm[(f / 4) * NC + c])[f % 4] = to_f(weight[(int64_t)j * HK + g]);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t warp_global = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t warps_total = (int64_t)gridDim.x * kWarps;
  const int64_t tasks = (rows + kRows - 1) / kRows;
  const int64_t my_tasks =
      (warp_global < tasks) ? (tasks - warp_global + warps_total - 1) / warps_total : 0;
  const int64_t nq = my_tasks * NIT;      // this warp's (task, column block) iterations
  // lane's 16 bytes of row r in ring slot `slot` (each lane reads back only
  // what it copied itself, so its own cp.async wait is enough)
  const uint32_t lane_ring =
      smem_u32(ring) + (uint32_t)((warp * kStages * kRows * kCPR) * kBlockBytes + lane * 16);
  // iteration cursors, advanced without divisions: (task, column block, slot)
  struct Cursor {
    int64_t task;
    int k, slot;
  };
  auto advance = [&](Cursor& cu) {
    if (++cu.k == NIT) { cu.k = 0; cu.task += warps_total; }
    if (++cu.slot == kStages) cu.slot = 0;
  };
  auto issue = [&](const Cursor& cu) {
    const int64_t r0 = cu.task * kRows;
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int h = 0; h < kCPR; ++h) {
        const int c = (cu.k * kCPR + h) * 32 + lane;
        const bool ok = c < NC && r0 + r < rows;
        cp_async16(lane_ring + (uint32_t)(((cu.slot * kRows + r) * kCPR + h) * kBlockBytes),
                   ok ? hidden + (r0 + r) * (int64_t)Dh + (int64_t)c * E : hidden, ok ? 16u : 0u);
      }
  };
  Cursor ahead{warp_global, 0, 0};          // the next iteration to fetch
#pragma unroll
  for (int x = 0; x < kStages; ++x) {
    if (x < nq) { issue(ahead); advance(ahead); }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  Cursor cur{warp_global, 0, 0};            // the iteration being multiplied
  float acc[kRows][HK];
#pragma unroll
  for (int r = 0; r < kRows; ++r)
#pragma unroll
    for (int g = 0; g < HK; ++g) acc[r][g] = 0.0f;
  for (int64_t q = 0; q < nq; ++q) {
    const int k = cur.k;
    const int slot = cur.slot;
    const int64_t r0 = cur.task * kRows;
    asm volatile("cp.async.wait_group %0;" ::"n"(kStages - 1) : "memory");
    uint4 hv[kRows][kCPR];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
      for (int h = 0; h < kCPR; ++h) {
        const uint32_t a = lane_ring + (uint32_t)(((slot * kRows + r) * kCPR + h) * kBlockBytes);
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(hv[r][h].x), "=r"(hv[r][h].y), "=r"(hv[r][h].z), "=r"(hv[r][h].w)
                     : "r"(a));
      }
    // the slot is now in registers: refill it with iteration q + kStages
    if (q + kStages < nq) { issue(ahead); advance(ahead); }
    asm volatile("cp.async.commit_group;" ::: "memory");
#pragma unroll
    for (int h = 0; h < kCPR; ++h) {
      const int c = (k * kCPR + h) * 32 + lane;
      if (c < NC) {
        float wv[E * HK];
#pragma unroll
        for (int f4 = 0; f4 < F4; ++f4) {
          const float4 w4 = wsm[f4 * NC + c];
          wv[4 * f4] = w4.x; wv[4 * f4 + 1] = w4.y; wv[4 * f4 + 2] = w4.z; wv[4 * f4 + 3] = w4.w;
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          float x[E];
          unpack(hv[r][h], x, Tin());
#pragma unroll
          for (int jj = 0; jj < E; ++jj)
#pragma unroll
            for (int g = 0; g < HK; ++g) acc[r][g] = fmaf(x[jj], wv[jj * HK + g], acc[r][g]);
        }
      }
    }
    if (k == NIT - 1) {
#pragma unroll
      for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int g = 0; g < HK; ++g) {
          float v = acc[r][g];
#pragma unroll
          for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
          acc[r][g] = v;
        }
      // lane (r*HK + g) mod 32 writes (row r, head g); one division per task
      const int64_t u0 = r0 / T;
      int64_t uu = u0, tt = r0 - u0 * T;
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        if (r > 0 && ++tt == T) { tt = 0; ++uu; }
#pragma unroll
        for (int g = 0; g < HK; ++g)
          if (lane == ((r * HK + g) & 31) && r0 + r < rows)
            scores[(uu * HK + g) * (int64_t)T + tt] = acc[r][g] + (bias ? bias[g] : 0.0f);
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int g = 0; g < HK; ++g) acc[r][g] = 0.0f;
    }
    advance(cur);
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Few rows (a decode step scores one new token per sequence), or a weight
// too large for shared memory: one CTA per hidden row, the weight read from
// L2 (every CTA reads the same Dh x HK values).  Thread x takes the 16-byte
// chunks x, x + 512, ... of the row (one chunk per thread up to Dh = 4096
// bf16, so each thread's loads are all in flight at once); partial sums are
// reduced by shuffles and across the sixteen warps in shared memory.
constexpr int kRowThreads = 512;
constexpr int64_t kFewRows = 1024;   // up to this many rows: one CTA per row

template <typename Tin, int HK, bool kVecW>
__global__ void __launch_bounds__(kRowThreads, 1)
linear_row_kernel(const Tin* __restrict__ hidden, const Tin* __restrict__ weight,
                  const float* __restrict__ bias, int T, int Dh, float* __restrict__ scores) {
  constexpr int E = Vec<Tin>::E;
  __shared__ float part[kRowThreads / 32][HK];
  // The row and the weights are read before waiting on the previous kernel
  // of the stream (no kernel of this library writes hidden states, weights or
  // biases), so that this work overlaps its tail; the scores are written
  // after the wait (the previous kernel may still read the last ones).
  pdl_trigger();
  const int64_t row = blockIdx.x;
  const int NC = Dh / E;
  const uint4* hrow = reinterpret_cast<const uint4*>(hidden + row * (int64_t)Dh);
  float acc[HK];
#pragma unroll
  for (int g = 0; g < HK; ++g) acc[g] = 0.0f;
  // chunk c's weights (E rows of HK values) are HK 16-byte words at
  // weight + c * E * HK, loaded as vectors when the weight is 16-byte aligned
  const uint4* wvec = reinterpret_cast<const uint4*>(weight);
  for (int c = threadIdx.x; c < NC; c += kRowThreads) {
    float x[E];
    unpack(__ldg(hrow + c), x, Tin());
    if (kVecW) {
      float wv[E * HK];
#pragma unroll
      for (int k = 0; k < HK; ++k) unpack(__ldg(wvec + (int64_t)c * HK + k), wv + k * E, Tin());
#pragma unroll
      for (int jj = 0; jj < E; ++jj)
#pragma unroll
        for (int g = 0; g < HK; ++g) acc[g] = fmaf(x[jj], wv[jj * HK + g], acc[g]);
    } else {
      const Tin* wrow = weight + (int64_t)c * E * HK;
#pragma unroll
      for (int jj = 0; jj < E; ++jj)
#pragma unroll
        for (int g = 0; g < HK; ++g) acc[g] = fmaf(x[jj], to_f(__ldg(wrow + jj * HK + g)), acc[g]);
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int g = 0; g < HK; ++g) {
    float v = acc[g];
#pragma unroll
    for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) part[warp][g] = v;
  }
  __syncthreads();
  pdl_wait();
  if (threadIdx.x < HK) {
    const int g = threadIdx.x;
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kRowThreads / 32; ++w) v += part[w][g];
    const int64_t u = row / T, t = row - u * T;
    scores[(u * HK + g) * (int64_t)T + t] = v + (bias ? bias[g] : 0.0f);
  }
}

template <typename Tin, int HK>
size_t smem_bytes(int Dh) {
  const int NC = Dh / Vec<Tin>::E;
  const size_t wbytes = (((size_t)(Vec<Tin>::E * HK / 4) * NC * 16) + 127) & ~size_t(127);
  return wbytes + (size_t)kWarps * kStages * kRows * kCPR * kBlockBytes;
}

template <typename Tin, int HK>
int run(const void* hidden, const void* weight, const float* bias, int U, int T, int Dh,
        float* scores, const Dev& dev, cudaStream_t s) {
  const size_t smem = smem_bytes<Tin, HK>(Dh);
  const int64_t rows = (int64_t)U * T;
  if (rows <= kFewRows || smem > (size_t)dev.max_smem_optin) {
    if (rows > 0x7fffffffLL) return KVC_ERR_UNSUPPORTED;
    auto rk = (reinterpret_cast<uintptr_t>(weight) & 15u) ? linear_row_kernel<Tin, HK, false>
                                                          : linear_row_kernel<Tin, HK, true>;
    return launch_pdl(rk, dim3((unsigned)rows), dim3(kRowThreads), 0, s,
                      static_cast<const Tin*>(hidden), static_cast<const Tin*>(weight), bias, T,
                      Dh, scores);
  }
  auto kern = linear_kernel<Tin, HK>;
  // raise the kernel's dynamic shared-memory limit when a call needs more
  // than any earlier one on this device
  static std::atomic<int> attr_bytes[64];
  if ((int)smem > attr_bytes[dev.device & 63].load()) {
    KVC_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr_bytes[dev.device & 63].store((int)smem);
  }
  const int64_t tasks = (rows + kRows - 1) / kRows;
  int64_t blocks = dev.sms;
  const int64_t need = (tasks + kWarps - 1) / kWarps;
  if (blocks > need) blocks = need;
  if (int rc = prefer_max_shared(kern, dev.device)) return rc;
  return launch_pdl(kern, dim3((unsigned)blocks), dim3(kWarps * 32), smem, s,
                    static_cast<const Tin*>(hidden), static_cast<const Tin*>(weight), bias, rows,
                    T, Dh, scores);
}

template <typename Tin>
int dispatch(const void* h, const void* w, const float* b, int U, int T, int Dh, int Hkv,
             float* sc, const Dev& dev, cudaStream_t s) {
  switch (Hkv) {
    case 1: return run<Tin, 1>(h, w, b, U, T, Dh, sc, dev, s);
    case 2: return run<Tin, 2>(h, w, b, U, T, Dh, sc, dev, s);
    case 3: return run<Tin, 3>(h, w, b, U, T, Dh, sc, dev, s);
    case 4: return run<Tin, 4>(h, w, b, U, T, Dh, sc, dev, s);
    case 5: return run<Tin, 5>(h, w, b, U, T, Dh, sc, dev, s);
    case 6: return run<Tin, 6>(h, w, b, U, T, Dh, sc, dev, s);
    case 7: return run<Tin, 7>(h, w, b, U, T, Dh, sc, dev, s);
    case 8: return run<Tin, 8>(h, w, b, U, T, Dh, sc, dev, s);
  }
  return KVC_ERR_UNSUPPORTED;
}

}  // namespace

int score_linear_launch(const void* hidden, const void* weight, const float* bias, int dtype,
                        int U, int T, int Dh, int Hkv, float* scores, const Dev& dev,
                        cudaStream_t s) {
  if (dtype == KVC_F32) {
    if (Dh % 4) return KVC_ERR_UNSUPPORTED;
    return dispatch<float>(hidden, weight, bias, U, T, Dh, Hkv, scores, dev, s);
  }
  return dispatch<uint16_t>(hidden, weight, bias, U, T, Dh, Hkv, scores, dev, s);
}

}  // namespace kvc
