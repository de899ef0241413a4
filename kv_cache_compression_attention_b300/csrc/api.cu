// C ABI entry points: host-side validation, workspace sizing and dispatch.
#include <math.h>
#include <mutex>

#include "kvc_internal.cuh"

namespace {

__device__ int g_status_word;   // one per device that loads the library

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
kvc::Dev g_devs[kMaxDevices];
bool g_dev_ready[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A source the compaction kernels may read in place: device (or managed)
// memory, or pinned host memory that the device sees at the same address
// (page-locked with the mapped property, which unified addressing gives
// cudaHostAlloc memory).  Anything else would fault on the device, so it is
// refused here.
int device_readable(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return KVC_ERR_INVALID;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return KVC_OK;
  if (a.type == cudaMemoryTypeHost && a.devicePointer == p) return KVC_OK;
  return KVC_ERR_INVALID;
}

}  // namespace

namespace kvc {

int device_info(Dev* out) {
  int dev = 0;
  KVC_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return KVC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (!g_dev_ready[dev]) {
    Dev d;
    d.device = dev;
    KVC_CUDA_TRY(cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev));
    KVC_CUDA_TRY(cudaDeviceGetAttribute(&d.max_smem_optin,
                                        cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
    void* p = nullptr;
    KVC_CUDA_TRY(cudaGetSymbolAddress(&p, g_status_word));
    d.status = static_cast<int*>(p);
    g_devs[dev] = d;
    g_dev_ready[dev] = true;
  }
  *out = g_devs[dev];
  return KVC_OK;
}

}  // namespace kvc

using kvc::Dev;

extern "C" {

int kvc_version(void) { return 100; }

const char* kvc_status_string(int status) {
  switch (status) {
    case KVC_OK: return "ok";
    case KVC_ERR_INVALID: return "invalid argument";
    case KVC_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case KVC_ERR_WORKSPACE: return "workspace too small";
    case KVC_ERR_CUDA: return "CUDA error";
    case KVC_ERR_TIMEOUT: return "device wait timed out";
    case KVC_ERR_RANGE: return "device index outside the stated capacity";
    default: return "unknown status";
  }
}

int kvc_device_status(void* stream) {
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  KVC_CUDA_TRY(cudaStreamSynchronize(kvc::as_stream(stream)));
  int v = 0;
  KVC_CUDA_TRY(cudaMemcpy(&v, dev.status, sizeof(int), cudaMemcpyDeviceToHost));
  int zero = 0;
  KVC_CUDA_TRY(cudaMemcpy(dev.status, &zero, sizeof(int), cudaMemcpyHostToDevice));
  return v;
}

// ------------------------------------------------------------------ score
namespace kvc {
size_t kvc_score_ws_need(bool tc, int U, int Hq, int Hkv, int W) {
  return tc ? score_attn_tc_ws(Hq, Hkv, W) : score_attn_simt_ws(U, Hq, W);
}
}  // namespace kvc

size_t kvc_score_attn_workspace(int U, int Hq, int Hkv, int T, int W, int d, int dtype) {
  if (U <= 0 || Hq <= 0 || W <= 0) return 0;
  if (kvc::score_attn_tc_supported(dtype, Hq, Hkv, W, d)) return kvc::score_attn_tc_ws(Hq, Hkv, W);
  return kvc::score_attn_simt_ws(U, Hq, W);
}

int kvc_score_attn_agg(const void* q_win, const void* k, int dtype, int U, int Hq, int Hkv,
                       int T, int W, int d, float scale, const float* head_scale, int causal,
                       int aggregation, float* scores, void* workspace, size_t workspace_bytes,
                       void* stream) {
  if (!q_win || !k || !scores) return KVC_ERR_INVALID;
  if (dtype != KVC_F32 && dtype != KVC_BF16) return KVC_ERR_INVALID;
  if (aggregation != KVC_AGG_SUM && aggregation != KVC_AGG_MAX) return KVC_ERR_INVALID;
  if (U <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || W <= 0 || Hq % Hkv) return KVC_ERR_INVALID;
  if (W > T || !(scale > 0.0f) || !isfinite(scale)) return KVC_ERR_INVALID;
  if (d != 64 && d != 128) return KVC_ERR_UNSUPPORTED;
  if ((int64_t)U * Hkv > 65535 || (int64_t)U * Hq * W > (1ll << 31)) return KVC_ERR_UNSUPPORTED;
  const bool tc = kvc::score_attn_tc_supported(dtype, Hq, Hkv, W, d);
  size_t need = kvc::kvc_score_ws_need(tc, U, Hq, Hkv, W);
  if (workspace_bytes < need || (need && !workspace)) return KVC_ERR_WORKSPACE;
  if (tc && (!aligned16(q_win) || !aligned16(k) || !aligned16(workspace)))
    return KVC_ERR_UNSUPPORTED;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  if (tc)
    return kvc::score_attn_tc(q_win, k, U, Hq, Hkv, T, W, scale, head_scale, causal, aggregation,
                              scores, workspace, dev, kvc::as_stream(stream));
  return kvc::score_attn_simt(q_win, k, dtype, U, Hq, Hkv, T, W, d, scale, head_scale, causal,
                              aggregation, scores, static_cast<float*>(workspace), dev,
                              kvc::as_stream(stream));
}

int kvc_score_attn(const void* q_win, const void* k, int dtype, int U, int Hq, int Hkv,
                   int T, int W, int d, float scale, const float* head_scale, int causal,
                   float* scores, void* workspace, size_t workspace_bytes, void* stream) {
  return kvc_score_attn_agg(q_win, k, dtype, U, Hq, Hkv, T, W, d, scale, head_scale, causal,
                            KVC_AGG_SUM, scores, workspace, workspace_bytes, stream);
}

int kvc_score_linear(const void* hidden, const void* weight, const float* bias, int dtype,
                     int U, int T, int Dh, int Hkv, float* scores, void* stream) {
  if (!hidden || !weight || !scores) return KVC_ERR_INVALID;
  if (dtype != KVC_F32 && dtype != KVC_BF16) return KVC_ERR_INVALID;
  if (U <= 0 || T <= 0 || Dh <= 0 || Hkv <= 0) return KVC_ERR_INVALID;
  if (Dh % 8 || Hkv > 8 || !aligned16(hidden)) return KVC_ERR_UNSUPPORTED;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::score_linear_launch(hidden, weight, bias, dtype, U, T, Dh, Hkv, scores, dev,
                                  kvc::as_stream(stream));
}

// ----------------------------------------------------------------- select
size_t kvc_select_workspace(int U, int Hkv, int T, int mode) { return 0; }

namespace {

// kvc_select's argument rules; on success *need_out is the non-protected
// budget, *ns_out / *nr_out the clamped sink and recent counts.
int select_args(const float* scores, int U, int Hkv, int T, int mode, double keep_ratio,
                const int32_t* head_budget, int n_sink, int n_recent, const int32_t* kept_idx,
                const int32_t* counts, const int64_t* offsets, int64_t* need_out, int* ns_out,
                int* nr_out) {
  if (!scores || !kept_idx || !counts || !offsets) return KVC_ERR_INVALID;
  if (U <= 0 || Hkv <= 0 || T <= 0 || n_sink < 0 || n_recent < 0) return KVC_ERR_INVALID;
  if (mode != KVC_SEL_GLOBAL_TOPK && mode != KVC_SEL_THRESHOLD && mode != KVC_SEL_PER_HEAD)
    return KVC_ERR_INVALID;
  if (mode == KVC_SEL_GLOBAL_TOPK && !(keep_ratio >= 0.0 && keep_ratio <= 1.0))
    return KVC_ERR_INVALID;
  if (mode == KVC_SEL_PER_HEAD && !head_budget) return KVC_ERR_INVALID;
  int64_t pool = (mode == KVC_SEL_GLOBAL_TOPK) ? (int64_t)Hkv * T : (int64_t)T;
  if (pool > (1ll << 24) || (int64_t)U * Hkv > (1ll << 24)) return KVC_ERR_UNSUPPORTED;
  if (mode == KVC_SEL_GLOBAL_TOPK && Hkv > 512) return KVC_ERR_UNSUPPORTED;   // heads per pool
  // protected set size |P| (the two ranges may overlap when T is small)
  int64_t ns = n_sink < T ? n_sink : T;
  int64_t rs = T - (int64_t)n_recent;           // first recent token
  if (rs < 0) rs = 0;
  int64_t nP = ns + (T - rs) - (rs < ns ? ns - rs : 0);
  int64_t need = 0;
  if (mode == KVC_SEL_GLOBAL_TOPK) {
    int64_t total = (int64_t)Hkv * T;
    int64_t B = (int64_t)floor(keep_ratio * (double)total);
    int64_t Beff = B < Hkv * nP ? Hkv * nP : B;
    if (Beff > total) Beff = total;
    need = Beff - Hkv * nP;
  }
  *need_out = need;
  *ns_out = (int)ns;
  *nr_out = (int)(T - rs);
  return KVC_OK;
}

}  // namespace

int kvc_select(const float* scores, int U, int Hkv, int T, int mode, double keep_ratio,
               float tau, const int32_t* head_budget, int n_sink, int n_recent,
               int32_t* kept_idx, int32_t* counts, int64_t* offsets, void* workspace,
               size_t workspace_bytes, void* stream) {
  int64_t need = 0;
  int ns = 0, nr = 0;
  if (int rc = select_args(scores, U, Hkv, T, mode, keep_ratio, head_budget, n_sink, n_recent,
                           kept_idx, counts, offsets, &need, &ns, &nr))
    return rc;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::select_launch(scores, U, Hkv, T, mode, need, tau, head_budget, ns, nr, kept_idx,
                            counts, offsets, dev, kvc::as_stream(stream));
}

size_t kvc_select_compact_workspace(int U, int Hkv, int T, int mode) {
  if (U <= 0 || Hkv <= 0 || T <= 0) return 0;
  return kvc::select_compact_ws(U, Hkv, T, mode);
}

int kvc_select_compact(const float* scores, int U, int Hkv, int T, int mode, double keep_ratio,
                       float tau, const int32_t* head_budget, int n_sink, int n_recent,
                       const void* k, const void* v, int dtype, int d, int slack_per_head,
                       void* kc, void* vc, int64_t capacity_rows, int32_t* kept_idx,
                       int32_t* counts, int64_t* offsets, int64_t* start, int32_t* len,
                       void* workspace, size_t workspace_bytes, void* stream) {
  int64_t need = 0;
  int ns = 0, nr = 0;
  if (int rc = select_args(scores, U, Hkv, T, mode, keep_ratio, head_budget, n_sink, n_recent,
                           kept_idx, counts, offsets, &need, &ns, &nr))
    return rc;
  if (!k || !v || !kc || !vc || !start || !len) return KVC_ERR_INVALID;
  if (dtype != KVC_F32 && dtype != KVC_BF16) return KVC_ERR_INVALID;
  if (d <= 0 || slack_per_head < 0 || capacity_rows < 0) return KVC_ERR_INVALID;
  int64_t row_bytes = (int64_t)d * (int64_t)kvc::elt_size(dtype);
  if (row_bytes % 16 || row_bytes > 4096) return KVC_ERR_UNSUPPORTED;
  if (!aligned16(k) || !aligned16(v) || !aligned16(kc) || !aligned16(vc))
    return KVC_ERR_UNSUPPORTED;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  if ((rc = device_readable(k)) || (rc = device_readable(v))) return rc;
  return kvc::select_compact_launch(scores, U, Hkv, T, mode, need, tau, head_budget, ns, nr, k,
                                    v, (int)row_bytes, slack_per_head, kc, vc, capacity_rows,
                                    kept_idx, counts, offsets, start, len, workspace,
                                    workspace ? workspace_bytes : 0, dev,
                                    kvc::as_stream(stream));
}

// ---------------------------------------------------------------- compact
int kvc_compact(const void* k, const void* v, int dtype, int U, int Hkv, int T, int d,
                const int32_t* kept_idx, const int32_t* counts, const int64_t* offsets,
                int slack_per_head, void* kc, void* vc, int64_t capacity_rows,
                int64_t* start, int32_t* len, void* stream) {
  if (!k || !v || !kept_idx || !counts || !offsets || !kc || !vc || !start || !len)
    return KVC_ERR_INVALID;
  if (dtype != KVC_F32 && dtype != KVC_BF16) return KVC_ERR_INVALID;
  if (U <= 0 || Hkv <= 0 || T <= 0 || d <= 0 || slack_per_head < 0 || capacity_rows < 0)
    return KVC_ERR_INVALID;
  int64_t row_bytes = (int64_t)d * (int64_t)kvc::elt_size(dtype);
  if (row_bytes % 16 || row_bytes > 4096) return KVC_ERR_UNSUPPORTED;
  if (!aligned16(k) || !aligned16(v) || !aligned16(kc) || !aligned16(vc))
    return KVC_ERR_UNSUPPORTED;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  if ((rc = device_readable(k)) || (rc = device_readable(v))) return rc;
  return kvc::compact_launch(k, v, (int)row_bytes, U, Hkv, T, kept_idx, counts, offsets,
                             slack_per_head, kc, vc, capacity_rows, start, len, dev,
                             kvc::as_stream(stream));
}

// ----------------------------------------------------------------- decode
size_t kvc_decode_workspace(int U, int Hq, int Hkv, int d, int max_len, int dtype) {
  if (U <= 0 || Hq <= 0 || Hkv <= 0 || max_len < 0) return 0;
  return kvc::decode_ws_bytes(U, Hq, Hkv, d, max_len);
}

int kvc_decode_attn(const void* q, void* kc, void* vc, const int64_t* start, int32_t* len,
                    const void* k_new, const void* v_new, int dtype, int U, int Hq, int Hkv,
                    int d, int max_len, float scale, void* out, float* lse, void* workspace,
                    size_t workspace_bytes, void* stream) {
  if (!q || !kc || !vc || !start || !len || !out) return KVC_ERR_INVALID;
  if ((k_new == nullptr) != (v_new == nullptr)) return KVC_ERR_INVALID;
  if (dtype != KVC_F32 && dtype != KVC_BF16) return KVC_ERR_INVALID;
  if (U <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || max_len < 0 || !isfinite(scale))
    return KVC_ERR_INVALID;
  if (d != 64 && d != 128) return KVC_ERR_UNSUPPORTED;
  if (Hq / Hkv > 8 || (int64_t)U * Hkv > 65535) return KVC_ERR_UNSUPPORTED;
  if (!aligned16(kc) || !aligned16(vc) || !aligned16(q)) return KVC_ERR_UNSUPPORTED;
  size_t need = kvc::decode_ws_bytes(U, Hq, Hkv, d, max_len);
  if (workspace_bytes < need || (need && !workspace)) return KVC_ERR_WORKSPACE;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::decode_launch(q, kc, vc, start, len, k_new, v_new, dtype, U, Hq, Hkv, d, max_len,
                            scale, out, lse, static_cast<float*>(workspace), dev,
                            kvc::as_stream(stream));
}

int kvc_quantize_rows(const void* x, int dtype, int64_t rows, int d, uint8_t* codes,
                      void* params, void* stream) {
  if (!x || !codes || !params) return KVC_ERR_INVALID;
  if (dtype != KVC_F32 && dtype != KVC_BF16) return KVC_ERR_INVALID;
  if (rows < 0) return KVC_ERR_INVALID;
  if (dtype != KVC_BF16 || (d != 64 && d != 128)) return KVC_ERR_UNSUPPORTED;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::quantize_rows_launch(x, rows, d, codes, params, dev, kvc::as_stream(stream));
}

int kvc_decode_attn_q8(const void* q, uint8_t* kq, void* kp, uint8_t* vq, void* vp,
                       const int64_t* start, int32_t* len, const void* k_new, const void* v_new,
                       int dtype, int U, int Hq, int Hkv, int d, int max_len, float scale,
                       void* out, float* lse, void* workspace, size_t workspace_bytes,
                       void* stream) {
  if (!q || !kq || !kp || !vq || !vp || !start || !len || !out) return KVC_ERR_INVALID;
  if ((k_new == nullptr) != (v_new == nullptr)) return KVC_ERR_INVALID;
  if (dtype != KVC_F32 && dtype != KVC_BF16) return KVC_ERR_INVALID;
  if (U <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || max_len < 0 || !isfinite(scale))
    return KVC_ERR_INVALID;
  if (dtype != KVC_BF16 || d != 128) return KVC_ERR_UNSUPPORTED;
  if (Hq / Hkv > 8 || (int64_t)U * Hkv > 65535) return KVC_ERR_UNSUPPORTED;
  if (!aligned16(kq) || !aligned16(vq) || !aligned16(kp) || !aligned16(vp) || !aligned16(q))
    return KVC_ERR_UNSUPPORTED;
  size_t need = kvc::decode_ws_bytes(U, Hq, Hkv, d, max_len);
  if (workspace_bytes < need || (need && !workspace)) return KVC_ERR_WORKSPACE;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::decode_q8_launch(q, kq, kp, vq, vp, start, len, k_new, v_new, U, Hq, Hkv, max_len,
                               scale, out, lse, static_cast<float*>(workspace), dev,
                               kvc::as_stream(stream));
}

int kvc_gather_scores(const float* scores, int U, int Hkv, int T, const int32_t* kept_idx,
                      const int32_t* counts, const int64_t* start, float* rscore,
                      int64_t capacity_rows, void* stream) {
  if (!scores || !kept_idx || !counts || !start || !rscore) return KVC_ERR_INVALID;
  if (U < 0 || Hkv < 0 || T < 0 || capacity_rows < 0) return KVC_ERR_INVALID;
  if ((int64_t)U * Hkv > 65535) return KVC_ERR_UNSUPPORTED;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::gather_scores_launch(scores, U, Hkv, T, kept_idx, counts, start, rscore,
                                   capacity_rows, dev, kvc::as_stream(stream));
}

int kvc_decode_prune(void* const* pools, const int* row_bytes, int n_pools, float* rscore,
                     const int64_t* start, int32_t* len, const float* s_new, int n_heads,
                     int window, int n_sink, float tau, int64_t capacity_rows, void* stream) {
  if (!pools || !row_bytes || !rscore || !start || !len || !s_new) return KVC_ERR_INVALID;
  if (n_pools < 1 || n_pools > KVC_PRUNE_MAX_POOLS) return KVC_ERR_INVALID;
  if (n_heads < 0 || window < 1 || n_sink < 0 || capacity_rows < 0 || isnan(tau))
    return KVC_ERR_INVALID;
  for (int p = 0; p < n_pools; ++p) {
    if (!pools[p] || row_bytes[p] <= 0) return KVC_ERR_INVALID;
    if (row_bytes[p] % 16 || row_bytes[p] > 65536 || !aligned16(pools[p]))
      return KVC_ERR_UNSUPPORTED;
  }
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::decode_prune_launch(pools, row_bytes, n_pools, rscore, start, len, s_new, n_heads,
                                  window, n_sink, tau, capacity_rows, dev,
                                  kvc::as_stream(stream));
}

int kvc_prune_ring_init(const int32_t* len, int n_heads, int window, int64_t t_next,
                        int32_t* ring, void* stream) {
  if (!len || !ring) return KVC_ERR_INVALID;
  if (n_heads < 0 || window < 1 || t_next < 0) return KVC_ERR_INVALID;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::prune_ring_init_launch(len, n_heads, window, t_next, ring, dev,
                                     kvc::as_stream(stream));
}

int kvc_decode_prune_ring(void* const* pools, const int* row_bytes, int n_pools, float* rscore,
                          const int64_t* start, int32_t* len, int32_t* ring, int64_t t_new,
                          const float* s_new, int n_heads, int window, int n_sink, float tau,
                          int64_t capacity_rows, void* stream) {
  if (!pools || !row_bytes || !rscore || !start || !len || !ring || !s_new) return KVC_ERR_INVALID;
  if (n_pools < 1 || n_pools > KVC_PRUNE_MAX_POOLS) return KVC_ERR_INVALID;
  if (n_heads < 0 || window < 1 || n_sink < 0 || capacity_rows < 0 || t_new < 0 || isnan(tau))
    return KVC_ERR_INVALID;
  for (int p = 0; p < n_pools; ++p) {
    if (!pools[p] || row_bytes[p] <= 0) return KVC_ERR_INVALID;
    if (row_bytes[p] % 16 || row_bytes[p] > 65536 || !aligned16(pools[p]))
      return KVC_ERR_UNSUPPORTED;
  }
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::decode_prune_ring_launch(pools, row_bytes, n_pools, rscore, start, len, ring, t_new,
                                       s_new, n_heads, window, n_sink, tau, capacity_rows, dev,
                                       kvc::as_stream(stream));
}

size_t kvc_score_kvzip_plus_workspace(int U, int Hq, int Hkv, int T, int W) {
  if (U < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || T < 0 || W <= 0) return 0;
  return kvc::score_kvzip_plus_ws_bytes(U, Hq, Hkv, T, W);
}

int kvc_score_kvzip_plus(const void* q_win, const void* k, const void* v, const void* gram,
                         const float* hnorm, int dtype, int U, int Hq, int Hkv, int T, int W,
                         int d, float scale, const float* head_scale, int causal, float* scores,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (!q_win || !k || !v || !gram || !hnorm || !scores) return KVC_ERR_INVALID;
  if (dtype != KVC_F32 && dtype != KVC_BF16) return KVC_ERR_INVALID;
  if (U <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || T <= 0 || W <= 0 || W > T || d <= 0)
    return KVC_ERR_INVALID;
  if (!(scale > 0.0f) || !isfinite(scale)) return KVC_ERR_INVALID;
  if (dtype != KVC_BF16 || d != 128) return KVC_ERR_UNSUPPORTED;
  if ((int64_t)U * Hkv > 65535 || !aligned16(v) || !aligned16(gram)) return KVC_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KVC_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < kvc::score_kvzip_plus_ws_bytes(U, Hq, Hkv, T, W))
    return KVC_ERR_WORKSPACE;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::score_kvzip_plus_launch(q_win, k, v, gram, hnorm, U, Hq, Hkv, T, W, scale,
                                      head_scale, causal ? 1 : 0, scores, workspace, dev,
                                      kvc::as_stream(stream));
}

size_t kvc_score_mlp_workspace(int Dh, int Dm) {
  if (Dh <= 0 || Dm <= 0) return 0;
  return kvc::score_mlp_ws_bytes(Dh, Dm);
}

int kvc_score_mlp(const void* hidden, const void* w1, const float* b1, const void* w2,
                  const float* b2, int dtype, int U, int T, int Dh, int Dm, int Hkv,
                  float* scores, void* workspace, size_t workspace_bytes, void* stream) {
  if (!hidden || !w1 || !w2 || !scores) return KVC_ERR_INVALID;
  if (dtype != KVC_F32 && dtype != KVC_BF16) return KVC_ERR_INVALID;
  if (U <= 0 || T <= 0 || Dh <= 0 || Dm <= 0 || Hkv <= 0) return KVC_ERR_INVALID;
  if (dtype != KVC_BF16 || Dh % 8 || Dm % 8 || Dm > 1024 || Hkv > 8) return KVC_ERR_UNSUPPORTED;
  if (!aligned16(hidden) || !aligned16(w1)) return KVC_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KVC_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < kvc::score_mlp_ws_bytes(Dh, Dm)) return KVC_ERR_WORKSPACE;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::score_mlp_launch(hidden, w1, b1, w2, b2, U, T, Dh, Dm, Hkv, scores, workspace, dev,
                               kvc::as_stream(stream));
}

int kvc_vector_residual(const void* k, const void* v, const void* W, int dtype, int U, int Hkv,
                        int T, int d, const int32_t* kept_idx, const int32_t* counts,
                        int n_sink, int n_recent, float* key, void* stream) {
  if (!k || !v || !W || !kept_idx || !counts || !key) return KVC_ERR_INVALID;
  if (dtype != KVC_F32 && dtype != KVC_BF16) return KVC_ERR_INVALID;
  if (U < 0 || Hkv <= 0 || T < 0 || d <= 0 || n_sink < 0 || n_recent < 0) return KVC_ERR_INVALID;
  if (dtype != KVC_BF16 || d != 128) return KVC_ERR_UNSUPPORTED;
  if ((int64_t)U * Hkv > 65535 || !aligned16(k) || !aligned16(v) || !aligned16(W))
    return KVC_ERR_UNSUPPORTED;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::vector_residual_launch(k, v, W, U, Hkv, T, kept_idx, counts, n_sink, n_recent, key,
                                     dev, kvc::as_stream(stream));
}

int kvc_vector_select(const float* key, int U, int Hkv, int T, const int32_t* counts,
                      int64_t n_approx, int32_t* approx_pos, int32_t* approx_counts,
                      int64_t* approx_offsets, void* stream) {
  if (!key || !counts || !approx_pos || !approx_counts || !approx_offsets) return KVC_ERR_INVALID;
  if (U <= 0 || Hkv <= 0 || T <= 0 || n_approx < 0 || n_approx > (int64_t)Hkv * T)
    return KVC_ERR_INVALID;
  if ((int64_t)Hkv * T > (1ll << 24) || (int64_t)U * Hkv > (1ll << 24)) return KVC_ERR_UNSUPPORTED;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::select_lens_launch(key, U, Hkv, T, counts, n_approx, approx_pos, approx_counts,
                                 approx_offsets, dev, kvc::as_stream(stream));
}

int kvc_vector_compact(const void* k, const void* v, int dtype, int U, int Hkv, int T, int d,
                       const int32_t* kept_idx, const int32_t* counts, const int64_t* offsets,
                       const int32_t* approx_pos, const int32_t* approx_counts,
                       const int64_t* approx_offsets, int slack_per_head, void* kc,
                       int64_t kc_rows, void* vc, int64_t vc_rows, int64_t* kstart,
                       int32_t* klen, int64_t* vstart, int32_t* napprox, void* stream) {
  if (!k || !v || !kept_idx || !counts || !offsets || !approx_pos || !approx_counts ||
      !approx_offsets || !kc || !vc || !kstart || !klen || !vstart || !napprox)
    return KVC_ERR_INVALID;
  if (dtype != KVC_F32 && dtype != KVC_BF16) return KVC_ERR_INVALID;
  if (U < 0 || Hkv <= 0 || T < 0 || d <= 0 || slack_per_head < 0 || kc_rows < 0 || vc_rows < 0)
    return KVC_ERR_INVALID;
  if (dtype != KVC_BF16 || d != 128) return KVC_ERR_UNSUPPORTED;
  if ((int64_t)U * Hkv > 65535 || !aligned16(k) || !aligned16(v) || !aligned16(kc) ||
      !aligned16(vc))
    return KVC_ERR_UNSUPPORTED;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::vector_compact_launch(k, v, U, Hkv, T, kept_idx, counts, offsets, approx_pos,
                                    approx_counts, approx_offsets, slack_per_head, kc, kc_rows,
                                    vc, vc_rows, kstart, klen, vstart, napprox, dev,
                                    kvc::as_stream(stream));
}

size_t kvc_decode_vector_workspace(int U, int Hq, int Hkv, int d, int max_len) {
  if (U <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || max_len < 0) return 0;
  return kvc::decode_vector_ws_bytes(U, Hq, Hkv, d, max_len);
}

int kvc_decode_attn_vector(const void* q, void* kc, void* vc, const int64_t* kstart,
                           int32_t* klen, const int64_t* vstart, const int32_t* napprox,
                           const void* W, const void* k_new, const void* v_new, int dtype, int U,
                           int Hq, int Hkv, int d, int max_len, float scale, void* out,
                           float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !kc || !vc || !kstart || !klen || !vstart || !napprox || !W || !out)
    return KVC_ERR_INVALID;
  if ((k_new == nullptr) != (v_new == nullptr)) return KVC_ERR_INVALID;
  if (dtype != KVC_F32 && dtype != KVC_BF16) return KVC_ERR_INVALID;
  if (U <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || max_len < 0 || !isfinite(scale))
    return KVC_ERR_INVALID;
  if (dtype != KVC_BF16 || d != 128) return KVC_ERR_UNSUPPORTED;
  if (Hq / Hkv > 8 || (int64_t)U * Hkv > 65535) return KVC_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(kc) || !aligned16(vc) || !aligned16(W))
    return KVC_ERR_UNSUPPORTED;
  size_t need = kvc::decode_vector_ws_bytes(U, Hq, Hkv, d, max_len);
  if (workspace_bytes < need || (need && !workspace)) return KVC_ERR_WORKSPACE;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::decode_vector_launch(q, kc, vc, kstart, klen, vstart, napprox, W, k_new, v_new, U,
                                   Hq, Hkv, max_len, scale, out, lse,
                                   static_cast<float*>(workspace), dev, kvc::as_stream(stream));
}

int kvc_fidelity(const void* out_comp, const void* out_full, const float* lse_comp,
                 const float* lse_full, int dtype, int n, int d, float* rel_err, float* kl,
                 void* stream) {
  if (!out_comp || !out_full || !lse_comp || !lse_full || !rel_err || !kl)
    return KVC_ERR_INVALID;
  if (dtype != KVC_F32 && dtype != KVC_BF16) return KVC_ERR_INVALID;
  if (n <= 0 || d <= 0 || d > 1024) return KVC_ERR_INVALID;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::fidelity_launch(out_comp, out_full, lse_comp, lse_full, dtype, n, d, rel_err, kl,
                              dev, kvc::as_stream(stream));
}

int kvc_selftest_wait_timeout(uint64_t timeout_ns, void* stream) {
  if (timeout_ns > 10000000000ull) return KVC_ERR_INVALID;
  Dev dev;
  int rc = kvc::device_info(&dev);
  if (rc) return rc;
  return kvc::selftest_wait_launch(timeout_ns, dev, kvc::as_stream(stream));
}

}  // extern "C"
