// Internal helpers shared by the kernels of libkvc (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <set>
#include <utility>

#include "kvc.h"

namespace kvc {

// ------------------------------------------------------------ host side
struct Dev {
  int device = 0;
  int sms = 0;
  int max_smem_optin = 0;
  int* status = nullptr;        // device address of this device's status word
};

// Per-device properties and the status word address (cached, thread-safe).
int device_info(Dev* out);

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

#define KVC_CUDA_TRY(expr)                                  \
  do {                                                      \
    cudaError_t e_ = (expr);                                \
    if (e_ != cudaSuccess) { (void)cudaGetLastError(); return KVC_ERR_CUDA; } \
  } while (0)

inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

inline size_t elt_size(int dtype) { return dtype == KVC_F32 ? 4 : 2; }

// Launch attribute for programmatic dependent launch: the kernel may start
// while the previous kernel of the stream still runs (its prologue overlaps
// that kernel's tail); every such kernel calls pdl_wait() before it touches
// memory the previous kernel reads or writes.
inline cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// Launches `kernel` with programmatic dependent launch enabled.
template <typename... P, typename... A>
inline int launch_pdl(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                      A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1] = {pdl_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  KVC_CUDA_TRY(cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...));
  return KVC_OK;
}

// Asks for the largest shared-memory carve-out for a kernel, once per
// device, so that back-to-back launches of the library's shared-memory
// kernels (score -> select, decode partial -> combine) need no
// reconfiguration of the SMs in between.  The gather-compaction keeps the
// default split: its streams run faster with the larger L1.
template <typename K>
inline int prefer_max_shared(K* kernel, int device) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), device);
  if (done.count(key)) return KVC_OK;
  KVC_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                    (int)cudaSharedmemCarveoutMaxShared));
  done.insert(key);
  return KVC_OK;
}

// Launchers (one per translation unit).  Arguments are already validated.
int score_attn_simt(const void* q, const void* k, int dtype, int U, int Hq, int Hkv, int T,
                    int W, int d, float scale, const float* head_scale, int causal, int agg,
                    float* scores, float* lse_ws, const Dev& dev, cudaStream_t s);
size_t score_attn_simt_ws(int U, int Hq, int W);

bool score_attn_tc_supported(int dtype, int Hq, int Hkv, int W, int d);
size_t score_attn_tc_ws(int Hq, int Hkv, int W);
// Aggregation code of the KVzip+ score inside the library (not an ABI value).
constexpr int kAggKvzipPlus = 2;
int score_attn_tc(const void* q, const void* k, int U, int Hq, int Hkv, int T, int W,
                  float scale, const float* head_scale, int causal, int agg, float* scores,
                  void* ws, const Dev& dev, cudaStream_t s, const float* hnorm = nullptr,
                  const float* vnorm = nullptr);

int score_linear_launch(const void* hidden, const void* weight, const float* bias, int dtype,
                        int U, int T, int Dh, int Hkv, float* scores, const Dev& dev,
                        cudaStream_t s);

int select_launch(const float* scores, int U, int Hkv, int T, int mode, int64_t need_global,
                  float tau, const int32_t* head_budget, int n_sink, int n_recent,
                  int32_t* kept_idx, int32_t* counts, int64_t* offsets, const Dev& dev,
                  cudaStream_t s);

// Global top-k of `need` keys per unit in which head i's candidates are its
// positions t < lens[i] (no protected set); the cluster kernel only.
int select_lens_launch(const float* keys, int U, int Hkv, int T, const int32_t* lens,
                       int64_t need, int32_t* kept_idx, int32_t* counts, int64_t* offsets,
                       const Dev& dev, cudaStream_t s);

// kvc_select followed by kvc_compact; a launch with one selection pool
// hands the select's decision to a kernel that emits and copies in one go.
size_t select_compact_ws(int U, int Hkv, int T, int mode);
int select_compact_launch(const float* scores, int U, int Hkv, int T, int mode,
                          int64_t need_global, float tau, const int32_t* head_budget, int n_sink,
                          int n_recent, const void* k, const void* v, int row_bytes, int slack,
                          void* kc, void* vc, int64_t capacity_rows, int32_t* kept_idx,
                          int32_t* counts, int64_t* offsets, int64_t* start, int32_t* len,
                          void* ws, size_t ws_bytes, const Dev& dev, cudaStream_t s);

int select_stream_launch(const float* scores, int U, int Hkv, int T, int mode,
                         int64_t need_global, float tau, const int32_t* head_budget, int n_sink,
                         int n_recent, int nP, int32_t* kept_idx, int32_t* counts,
                         int64_t* offsets, bool offsets_in_kernel, const Dev& dev,
                         cudaStream_t s);

int compact_launch(const void* k, const void* v, int row_bytes, int U, int Hkv, int T,
                   const int32_t* kept_idx, const int32_t* counts, const int64_t* offsets,
                   int slack, void* kc, void* vc, int64_t capacity_rows, int64_t* start,
                   int32_t* len, const Dev& dev, cudaStream_t s);

size_t decode_ws_bytes(int U, int Hq, int Hkv, int d, int max_len);
int decode_launch(const void* q, void* kc, void* vc, const int64_t* start, int32_t* len,
                  const void* k_new, const void* v_new, int dtype, int U, int Hq, int Hkv,
                  int d, int max_len, float scale, void* out, float* lse, float* ws,
                  const Dev& dev, cudaStream_t s);

int decode_q8_launch(const void* q, uint8_t* kq, void* kp, uint8_t* vq, void* vp,
                     const int64_t* start, int32_t* len, const void* k_new, const void* v_new,
                     int U, int Hq, int Hkv, int max_len, float scale, void* out, float* lse,
                     float* ws, const Dev& dev, cudaStream_t s);
int quantize_rows_launch(const void* x, int64_t rows, int d, uint8_t* codes, void* params,
                         const Dev& dev, cudaStream_t s);

int decode_prune_launch(void* const* pools, const int* row_bytes, int n_pools, float* rscore,
                        const int64_t* start, int32_t* len, const float* s_new, int n_heads,
                        int window, int n_sink, float tau, int64_t capacity_rows, const Dev& dev,
                        cudaStream_t s);
int decode_prune_ring_launch(void* const* pools, const int* row_bytes, int n_pools,
                             float* rscore, const int64_t* start, int32_t* len, int32_t* ring,
                             int64_t t_new, const float* s_new, int n_heads, int window,
                             int n_sink, float tau, int64_t capacity_rows, const Dev& dev,
                             cudaStream_t s);
int prune_ring_init_launch(const int32_t* len, int n_heads, int window, int64_t t_next,
                           int32_t* ring, const Dev& dev, cudaStream_t s);
int gather_scores_launch(const float* scores, int U, int Hkv, int T, const int32_t* kept_idx,
                         const int32_t* counts, const int64_t* start, float* rscore,
                         int64_t capacity_rows, const Dev& dev, cudaStream_t s);

int score_kvzip_plus_simt(const void* q, const void* k, int U, int Hq, int Hkv, int T, int W,
                          float scale, const float* head_scale, int causal, const float* hnorm,
                          const float* vnorm, float* scores, float* lse_ws, const Dev& dev,
                          cudaStream_t s);
size_t score_kvzip_plus_ws_bytes(int U, int Hq, int Hkv, int T, int W);
int score_kvzip_plus_launch(const void* q, const void* k, const void* v, const void* gram,
                            const float* hnorm, int U, int Hq, int Hkv, int T, int W,
                            float scale, const float* head_scale, int causal, float* scores,
                            void* workspace, const Dev& dev, cudaStream_t s);
size_t score_mlp_ws_bytes(int Dh, int Dm);
int score_mlp_launch(const void* hidden, const void* w1, const float* b1, const void* w2,
                     const float* b2, int U, int T, int Dh, int Dm, int Hkv, float* scores,
                     void* workspace, const Dev& dev, cudaStream_t s);
int vector_residual_launch(const void* k, const void* v, const void* W, int U, int Hkv, int T,
                           const int32_t* kept_idx, const int32_t* counts, int n_sink,
                           int n_recent, float* key, const Dev& dev, cudaStream_t s);
int vector_compact_launch(const void* k, const void* v, int U, int Hkv, int T,
                          const int32_t* kept_idx, const int32_t* counts,
                          const int64_t* offsets, const int32_t* approx_pos,
                          const int32_t* approx_counts, const int64_t* approx_offsets, int slack,
                          void* kc, int64_t kc_rows, void* vc, int64_t vc_rows, int64_t* kstart,
                          int32_t* klen, int64_t* vstart, int32_t* napprox, const Dev& dev,
                          cudaStream_t s);
size_t decode_vector_ws_bytes(int U, int Hq, int Hkv, int d, int max_len);
int decode_vector_launch(const void* q, void* kc, void* vc, const int64_t* kstart,
                         int32_t* klen, const int64_t* vstart, const int32_t* napprox,
                         const void* W, const void* k_new, const void* v_new, int U, int Hq,
                         int Hkv, int max_len, float scale, void* out, float* lse, float* ws,
                         const Dev& dev, cudaStream_t s);

int fidelity_launch(const void* oc, const void* of, const float* lc, const float* lf,
                    int dtype, int n, int d, float* rel, float* kl, const Dev& dev,
                    cudaStream_t s);

int selftest_wait_launch(uint64_t timeout_ns, const Dev& dev, cudaStream_t s);

}  // namespace kvc

// ---------------------------------------------------------- device side
#ifdef __CUDACC__

namespace kvc {

// Default bound on every spin-wait in the kernels: 2 s of wall time.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

__device__ __forceinline__ void report(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Programmatic dependent launch, device side: pdl_wait() returns once the
// previous kernel of the stream has completed and its memory is visible (at
// once when the kernel was launched without the attribute); pdl_trigger()
// lets the next kernel's CTAs be scheduled before this one ends.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// bf16 <-> fp32.  bf16 -> fp32 is exact (the bf16 bits are the top half).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// fp32 -> bf16 with round-to-nearest-even (NaN kept quiet).
__device__ __forceinline__ uint16_t f2bf16_rne(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((b >> 16) | 0x0040u);
  uint32_t lsb = (b >> 16) & 1u;
  b += 0x7fffu + lsb;
  return (uint16_t)(b >> 16);
}

// Order-preserving map of fp32 onto uint32 for selection: larger score ->
// larger key; -0 and +0 share one key; every NaN maps to 1 (below -inf);
// key 0 is reserved for "protected, not a candidate".
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7fffffffu) > 0x7f800000u) return 1u;     // NaN
  if ((b << 1) == 0u) b = 0u;                          // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase.  On timeout the status word records
// KVC_ERR_TIMEOUT, *abort is raised (if given) and false is returned; the
// caller carries on as if the phase had completed so that the kernel ends.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                                          volatile int* abort_flag,
                                          uint64_t timeout_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (abort_flag && *abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        report(status, KVC_ERR_TIMEOUT);
        if (abort_flag) *abort_flag = 1;
        return false;
      }
    }
  }
}

}  // namespace kvc

#endif  // __CUDACC__
