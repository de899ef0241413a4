// kvc_decode_attn_noalloc: one decode step over a compressed cache for
// callers that cannot allocate device memory.
//
// kvc_decode_attn takes its split-K scratch (one (acc[d], max, sum) record
// per q head and 1024-row chunk) from a workspace the caller allocates.  Some
// callers have no way to do that: a plug-in loaded into a host engine that
// owns every device allocation and hands its plug-ins no allocator and no
// workspace, or a caller whose device-memory budget is fixed at start-up and
// must not grow (or stall the device, which cudaMalloc may do) in the middle
// of serving.  This entry point serves them: its scratch is a fixed array in
// the library's own device memory, held on each GPU where the library's
// device code is loaded until the process exits.
//
// Nothing here allocates: no cudaMalloc, no cudaFree, no allocating library
// routine.  The first call on a device looks up the array's device address
// with cudaGetSymbolAddress (in host code the array's name is only a host
// stand-in, not a device address) and caches it.  Under CUDA's lazy module
// loading (the default) that lookup is what loads the module on the device,
// so the array is reserved inside the first call, which then fails with
// KVC_ERR_CUDA if the device has no memory left: make that first call at
// start-up, before the caller commits its device memory and before any
// stream capture.  Every call on a device shares the one array, so calls
// whose kernels overlap on the GPU (different streams, no ordering between
// them) race on it; serialise them.  The array keeps the last call's
// contents, and nothing in it has to start at zero: every record the step
// reads is written earlier in the same step.
#include <mutex>

#include "kvc_internal.cuh"

namespace {

constexpr size_t kScratchBytes = KVC_DECODE_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) float g_decode_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of this device's copy of the scratch array (set up once per
// device, with that device current).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { (void)cudaGetLastError(); return KVC_ERR_CUDA; }
  if (dev < 0 || dev >= kMaxDevices) return KVC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return KVC_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KVC_OK;
}

}  // namespace

extern "C" size_t kvc_decode_noalloc_scratch_bytes(void) { return kScratchBytes; }

extern "C" int kvc_decode_attn_noalloc(const void* q, void* kc, void* vc, const int64_t* start,
                                       int32_t* len, const void* k_new, const void* v_new,
                                       int dtype, int U, int Hq, int Hkv, int d, int max_len,
                                       float scale, void* out, float* lse, void* stream) {
  if (!q || !kc || !vc || !start || !len || !out) return KVC_ERR_INVALID;
  if (U <= 0 || Hq <= 0 || Hkv <= 0 || max_len < 0) return KVC_ERR_INVALID;
  // sizes whose split-K records do not fit the fixed scratch are refused
  // before any CUDA call
  if (kvc_decode_workspace(U, Hq, Hkv, d, max_len, dtype) > kScratchBytes)
    return KVC_ERR_WORKSPACE;
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc) return rc;
  return kvc_decode_attn(q, kc, vc, start, len, k_new, v_new, dtype, U, Hq, Hkv, d, max_len,
                         scale, out, lse, scratch, kScratchBytes, stream);
}
