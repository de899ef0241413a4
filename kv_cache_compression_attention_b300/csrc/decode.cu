// Varlen split-K decode attention over a compressed cache, with append.
//
// Definition (KVSculpt §2B: attention output and its log-sum-exp; KVzap
// §2.3: pruning sits after attention and also runs while decoding): for
// head i = u*Hkv + g with rows j < L of the pool starting at start_i, and
// each of its G query heads h,
//   lse_h = log sum_j exp(scale <q_h, k_j>),  o_h = sum_j exp(scale <q_h,k_j> - lse_h) v_j.
//
// The step streams every cached K/V row once from HBM (bandwidth bound; the
// G query heads of a kv head share each row, 4*d flops per 2*d bytes at
// G = 4), so it runs on the SIMT cores:
//   partial  grid (chunks of 1024 rows, heads): each CTA's 4 warps take
//            16-row groups; K rows are read by 8-lane teams (16-byte
//            coalesced loads), the 8 partial dot products are reduced by
//            xor-shuffles, an online softmax (base 2) keeps (m, l) per head,
//            and each lane accumulates d/32 output columns of all G heads
//            from the V rows.  The 4 warps merge through shared memory and
//            the CTA writes (m, l, acc[d]) per query head to the workspace.
//   combine  one CTA per kv head: merges the chunks by their maxima, adds
//            the appended token (from k_new / v_new, not from the pool, so
//            no CTA of this step reads a row another one writes), writes out
//            and lse, then appends k_new / v_new at row start_i + L and
//            bumps len.
#include <cuda_fp16.h>

#include <atomic>

#include "kvc_internal.cuh"
#include "mma_sync.cuh"

namespace kvc {
namespace {

constexpr int kChunk = 1024;    // rows per partial CTA (512 measured 3 % slower on the batch-64 step)
constexpr int kQ8Chunk = 2048;  // rows per partial CTA over a quantised pool
constexpr int kWarps = 4;       // compute warps per partial CTA
constexpr int kStageRows = 32;  // rows per shared-memory stage (8 per compute warp)
constexpr int kStages = 4;
constexpr int kStagedChunks = 256;  // chunks whose statistics the combine stages in smem
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename Tin> struct Elt;
template <> struct Elt<float> {
  static __device__ __forceinline__ float get(const float* p, int x) { return p[x]; }
  static __device__ __forceinline__ void put(float* p, int x, float v) { p[x] = v; }
};
template <> struct Elt<uint16_t> {
  static __device__ __forceinline__ float get(const uint16_t* p, int x) {
    return __uint_as_float(((uint32_t)p[x]) << 16);
  }
  static __device__ __forceinline__ void put(uint16_t* p, int x, float v) { p[x] = f2bf16_rne(v); }
};

// N consecutive elements held packed in registers (bf16: two per word) and
// loaded with 16/8/4-byte vector loads through the read-only path.
template <typename Tin, int N>
struct Raw {
  static constexpr int kWords = N * (int)sizeof(Tin) / 4;
  uint32_t w[kWords];
  __device__ __forceinline__ void load(const Tin* p) {
    if constexpr (kWords % 4 == 0) {
#pragma unroll
      for (int i = 0; i < kWords / 4; ++i) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p) + i);
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
      }
    } else if constexpr (kWords == 2) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
      w[0] = v.x; w[1] = v.y;
    } else {
      static_assert(kWords == 1, "vector width");
      w[0] = __ldg(reinterpret_cast<const uint32_t*>(p));
    }
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < kWords; ++i) w[i] = 0u;
  }
  __device__ __forceinline__ float operator[](int x) const {
    if constexpr (sizeof(Tin) == 2) return (x & 1) ? bf16hi(w[x >> 1]) : bf16lo(w[x >> 1]);
    else return __uint_as_float(w[x]);
  }
};

// N consecutive elements of a shared-memory row, loaded with 16/8/4-byte
// vector loads.
template <typename Tin, int N>
struct SRaw {
  static constexpr int kWords = N * (int)sizeof(Tin) / 4;
  uint32_t w[kWords];
  __device__ __forceinline__ void load(const Tin* p) {
    if constexpr (kWords % 4 == 0) {
#pragma unroll
      for (int i = 0; i < kWords / 4; ++i) {
        const uint4 v = reinterpret_cast<const uint4*>(p)[i];
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
      }
    } else if constexpr (kWords == 2) {
      const uint2 v = *reinterpret_cast<const uint2*>(p);
      w[0] = v.x; w[1] = v.y;
    } else {
      static_assert(kWords == 1, "vector width");
      w[0] = *reinterpret_cast<const uint32_t*>(p);
    }
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < kWords; ++i) w[i] = 0u;
  }
  __device__ __forceinline__ float operator[](int x) const {
    if constexpr (sizeof(Tin) == 2) return (x & 1) ? bf16hi(w[x >> 1]) : bf16lo(w[x >> 1]);
    else return __uint_as_float(w[x]);
  }
};

// Bulk asynchronous copy global -> shared, completing on an mbarrier
// (addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

template <typename Tin, int D>
constexpr size_t partial_smem_bytes() {
  return 2ull * kStages * kStageRows * D * sizeof(Tin);
}

// One CTA per (kv head, 1024-row chunk).  A producer warp streams the chunk's
// K and V rows (contiguous in the pool) into a 4-stage shared-memory ring
// with bulk asynchronous copies; four compute warps take 8 rows of every
// stage each.
template <typename Tin, int D, int G>
__global__ void __launch_bounds__((kWarps + 1) * 32)
decode_partial_kernel(const Tin* __restrict__ q, const Tin* __restrict__ kc,
                      const Tin* __restrict__ vc, const int64_t* __restrict__ start,
                      const int32_t* __restrict__ len, int Hkv, int max_chunks, float scale_log2,
                      float* __restrict__ ws, int* status) {
  constexpr int DPL = D / 8;     // q.k dims per lane (8 lanes per row)
  constexpr int VPL = D / 32;    // output dims per lane
  constexpr int RPW = kStageRows / kWarps;   // rows per warp and stage
  constexpr uint32_t RB = D * sizeof(Tin);   // bytes per row
  extern __shared__ __align__(128) uint8_t smem_dec[];
  Tin* ks = reinterpret_cast<Tin*>(smem_dec);
  Tin* vs = ks + kStages * kStageRows * D;
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ float p_sm[kWarps][RPW][G];
  __shared__ float m_sm[kWarps][G], l_sm[kWarps][G];
  __shared__ float acc_sm[kWarps][G][D];
  pdl_wait();
  pdl_trigger();

  const int i = blockIdx.y, c = blockIdx.x;
  const int L = len[i];
  const int rb = c * kChunk;
  if (rb >= L) return;
  const int nrows = min(L, rb + kChunk) - rb;
  const int nst = (nrows + kStageRows - 1) / kStageRows;
  const int u = i / Hkv, g = i - u * Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], kWarps); }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const Tin* kb = kc + (start[i] + rb) * D;
      const Tin* vb = vc + (start[i] + rb) * D;
      for (int st = 0; st < nst; ++st) {
        const int slot = st % kStages;
        if (st >= kStages) mbar_wait(&empty[slot], ((st / kStages) - 1) & 1, status, nullptr);
        const int n = min(kStageRows, nrows - st * kStageRows);
        const uint32_t bytes = (uint32_t)n * RB;
        mbar_arrive_expect_tx(&full[slot], 2u * bytes);
        bulk_g2s(smem_u32(ks + (size_t)slot * kStageRows * D), kb + (size_t)st * kStageRows * D,
                 bytes, &full[slot]);
        bulk_g2s(smem_u32(vs + (size_t)slot * kStageRows * D), vb + (size_t)st * kStageRows * D,
                 bytes, &full[slot]);
      }
    }
    return;
  }

  // -------------------------------------------------------------- compute
  const int r8 = lane >> 3, sub = lane & 7;
  float qr[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    Raw<Tin, DPL> rq;
    rq.load(q + ((int64_t)u * Hkv * G + (int64_t)g * G + h) * D + sub * DPL);
#pragma unroll
    for (int x = 0; x < DPL; ++x) qr[h][x] = rq[x];
  }
  float m[G], l[G], acc[G][VPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY; l[h] = 0.0f;
#pragma unroll
    for (int x = 0; x < VPL; ++x) acc[h][x] = 0.0f;
  }
  const int r0 = warp * RPW;                   // this warp's rows inside a stage
  for (int st = 0; st < nst; ++st) {
    const int slot = st % kStages;
    mbar_wait(&full[slot], (st / kStages) & 1, status, nullptr);
    const int n = min(kStageRows, nrows - st * kStageRows);
    const Tin* kst = ks + ((size_t)slot * kStageRows + r0) * D;
    const Tin* vst = vs + ((size_t)slot * kStageRows + r0) * D;
    // K rows by 8-lane teams (pass p covers rows 4p + r8), V rows by the
    // whole warp (lane owns d/32 columns)
    SRaw<Tin, DPL> kr[RPW / 4];
    SRaw<Tin, VPL> vr[RPW];
#pragma unroll
    for (int pp = 0; pp < RPW / 4; ++pp) {
      const int row = 4 * pp + r8;
      if (r0 + row < n) kr[pp].load(kst + row * D + sub * DPL);
      else kr[pp].zero();
    }
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
      if (r0 + rr < n) vr[rr].load(vst + rr * D + lane * VPL);
      else vr[rr].zero();
    }
    float sc[RPW / 4][G];
#pragma unroll
    for (int pp = 0; pp < RPW / 4; ++pp) {
      const int row = 4 * pp + r8;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float a = 0.0f;
#pragma unroll
        for (int x = 0; x < DPL; ++x) a = fmaf(qr[h][x], kr[pp][x], a);
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        a += __shfl_xor_sync(0xffffffffu, a, 4);
        sc[pp][h] = (r0 + row < n) ? a * scale_log2 : -INFINITY;
      }
    }
    // online softmax update (base 2), identical in all lanes
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float mx = sc[0][h];
#pragma unroll
      for (int pp = 1; pp < RPW / 4; ++pp) mx = fmaxf(mx, sc[pp][h]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float mn = fmaxf(m[h], mx);
      const float alpha = (mn == -INFINITY) ? 1.0f : exp2f(m[h] - mn);   // m = -inf -> 0
      m[h] = mn;
      l[h] *= alpha;
#pragma unroll
      for (int x = 0; x < VPL; ++x) acc[h][x] *= alpha;
#pragma unroll
      for (int pp = 0; pp < RPW / 4; ++pp) {
        const float e = (mn == -INFINITY) ? 0.0f : exp2f(sc[pp][h] - mn);
        l[h] += e;                               // summed over the 4 row teams at the end
        if (sub == 0) p_sm[warp][4 * pp + r8][h] = e;
      }
    }
    __syncwarp();
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
      // rows past the end carry p = 0 and zeroed V
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pw = p_sm[warp][rr][h];
#pragma unroll
        for (int x = 0; x < VPL; ++x) acc[h][x] = fmaf(pw, vr[rr][x], acc[h][x]);
      }
    }
    // every lane has consumed its shared-memory reads of this stage
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  // l: each 8-lane team summed its own rows -> add the 4 teams
#pragma unroll
  for (int h = 0; h < G; ++h) {
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 8);
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 16);
  }
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) { m_sm[warp][h] = m[h]; l_sm[warp][h] = l[h]; }
  }
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int x = 0; x < VPL; ++x) acc_sm[warp][h][lane * VPL + x] = acc[h][x];
  asm volatile("bar.sync 1, %0;" ::"r"(kWarps * 32) : "memory");   // compute warps only
  // merge the warps: thread -> (h, column block)
  float* out = ws + ((int64_t)i * max_chunks + c) * G * (D + 2);
  for (int e = threadIdx.x; e < G * D; e += kWarps * 32) {
    const int h = e / D, x = e - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, m_sm[w][h]);
    float a = 0.0f, lsum = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = (m_sm[w][h] == -INFINITY) ? 0.0f : exp2f(m_sm[w][h] - M);
      a += acc_sm[w][h][x] * f;
      lsum += l_sm[w][h] * f;
    }
    out[h * (D + 2) + x] = a;
    if (x == 0) { out[h * (D + 2) + D] = M; out[h * (D + 2) + D + 1] = lsum; }
  }
}

// Group quantisation of one element per lane of a warp that holds one group
// of 32 ([KVTC] §2B: groups share a scale and an offset): lo = fp16(min),
// scale = fp16((max - lo) / 255), code = clamp(rint((x - lo) / scale), 0, 255)
// (0 when scale is 0), all in IEEE fp32.  Lane 0 writes (scale, lo) as an
// fp16 pair.
__device__ __forceinline__ void quantize_elem(float v, int lane, uint8_t* code, uint32_t* param) {
  float mn = v, mx = v;
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  const __half lo16 = __float2half_rn(mn);
  const float lo = __half2float(lo16);
  const __half sc16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, lo), 255.0f));
  const float sc = __half2float(sc16);
  float c = 0.0f;
  if (sc != 0.0f) c = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(v, lo), sc)), 0.0f), 255.0f);
  *code = (uint8_t)c;
  if (lane == 0)
    *param = (uint32_t)__half_as_ushort(sc16) | ((uint32_t)__half_as_ushort(lo16) << 16);
}

// Group-quantised copy of bf16 rows of D elements: one warp per row, lane l
// holds element l of every group.
template <int D>
__global__ void __launch_bounds__(256)
quantize_rows_kernel(const uint16_t* __restrict__ x, int64_t rows, uint8_t* __restrict__ codes,
                     uint32_t* __restrict__ params) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  for (int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); row < rows;
       row += (int64_t)gridDim.x * 8) {
#pragma unroll
    for (int g = 0; g < D / 32; ++g) {
      const float v = bf16lo((uint32_t)x[row * D + g * 32 + lane]);
      quantize_elem(v, lane, codes + row * D + g * 32 + lane, params + row * (D / 32) + g);
    }
  }
}

template <typename Tin, int D, int G>
__global__ void __launch_bounds__(D)
decode_combine_kernel(const Tin* __restrict__ q, Tin* __restrict__ kc, Tin* __restrict__ vc,
                      const int64_t* __restrict__ start, int32_t* __restrict__ len,
                      const Tin* __restrict__ k_new, const Tin* __restrict__ v_new, int n_heads,
                      int Hkv, int max_chunks, float scale_log2, const float* __restrict__ ws,
                      Tin* __restrict__ out, float* __restrict__ lse, int* status,
                      uint8_t* __restrict__ kq, uint32_t* __restrict__ kp,
                      uint8_t* __restrict__ vq, uint32_t* __restrict__ vp, int chunk) {
  __shared__ float red[D / 32][G];
  const int i = blockIdx.x;
  const int u = i / Hkv, g = i - u * Hkv;
  const int x = threadIdx.x, lane = x & 31, warp = x >> 5;
  const bool append = k_new != nullptr;
  const int64_t nrow = (int64_t)u * Hkv + g;
  // The step's own inputs (q, k_new, v_new: no kernel writes them) are read
  // and the appended token's scores formed before waiting on the partial
  // kernel, so that this work overlaps its tail.
  const float kn = append ? Elt<Tin>::get(k_new + nrow * D, x) : 0.0f;
  const float vn = append ? Elt<Tin>::get(v_new + nrow * D, x) : 0.0f;
  // appended-token scores for the G heads
  float snew[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float a = append ? Elt<Tin>::get(q + (nrow * G + h) * D, x) * kn : 0.0f;
#pragma unroll
    for (int off = 16; off; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
    if (lane == 0) red[warp][h] = a;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float a = 0.0f;
#pragma unroll
    for (int w = 0; w < D / 32; ++w) a += red[w][h];
    snew[h] = a * scale_log2;
  }
  // the head's length too: the previous kernels that write it (this
  // library's appends and prunes of earlier steps) completed before the
  // partial kernel let this one start, so it is final (read from L2, past
  // any line an earlier kernel left in this SM's L1)
  const int L = __ldcg(len + i);
  int nch = (L + chunk - 1) / chunk;
  if (nch > max_chunks) { if (x == 0) report(status, KVC_ERR_RANGE); nch = max_chunks; }
  bool room = append;
  if (append && i + 1 < n_heads && __ldcg(start + i) + L >= __ldcg(start + i + 1)) {
    if (x == 0) report(status, KVC_ERR_RANGE);
    room = false;
  }
  pdl_wait();
  pdl_trigger();
  const float* base = ws + (int64_t)i * max_chunks * G * (D + 2);
  if (nch <= kStagedChunks) {
    // every chunk's (max, sum) of every head into shared memory (all loads
    // in flight), one warp per head for the maxima and the normalisers, then
    // each thread sums its column over the chunks with the staged weights
    __shared__ float s_w[kStagedChunks * G], s_l[kStagedChunks * G];
    __shared__ float s_M[G], s_L[G];
    for (int e = x; e < nch * G; e += D) {
      const float* pc = base + (int64_t)e * (D + 2);
      s_w[e] = pc[D];
      s_l[e] = pc[D + 1];
    }
    // column x of the first kEarly chunks, in flight with the statistics
    constexpr int kEarly = 8;
    float pe[kEarly][G];
#pragma unroll
    for (int c = 0; c < kEarly; ++c)
#pragma unroll
      for (int h = 0; h < G; ++h)
        pe[c][h] = c < nch ? base[(int64_t)(c * G + h) * (D + 2) + x] : 0.0f;
    __syncthreads();
    for (int h = warp; h < G; h += D / 32) {
      float M = append ? snew[h] : -INFINITY;
      for (int c = lane; c < nch; c += 32) M = fmaxf(M, s_w[c * G + h]);
#pragma unroll
      for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
      if (lane == 0) s_M[h] = M;
    }
    __syncthreads();
    for (int e = x; e < nch * G; e += D) {
      const float mc = s_w[e];
      s_w[e] = (mc == -INFINITY) ? 0.0f : exp2f(mc - s_M[e % G]);
    }
    __syncthreads();
    for (int h = warp; h < G; h += D / 32) {
      float Ls = 0.0f;
      for (int c = lane; c < nch; c += 32) Ls += s_w[c * G + h] * s_l[c * G + h];
#pragma unroll
      for (int off = 16; off; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
      if (lane == 0) s_L[h] = Ls;
    }
    __syncthreads();
    // column x of every chunk and head: chunks outer, heads inner, so that
    // 4 x G loads are in flight per thread
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.0f;
#pragma unroll
    for (int c = 0; c < kEarly; ++c)
      if (c < nch) {
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] = fmaf(s_w[c * G + h], pe[c][h], acc[h]);
      }
#pragma unroll 4
    for (int c = kEarly; c < nch; ++c) {
      float pv[G];
#pragma unroll
      for (int h = 0; h < G; ++h) pv[h] = base[(int64_t)(c * G + h) * (D + 2) + x];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = fmaf(s_w[c * G + h], pv[h], acc[h]);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float M = s_M[h];
      float a = acc[h], lsum = s_L[h];
      if (append) {
        const float f = exp2f(snew[h] - M);
        a += vn * f;
        lsum += f;
      }
      const int64_t orow = nrow * G + h;
      Elt<Tin>::put(out + orow * D, x, lsum > 0.0f ? a / lsum : 0.0f);
      if (lse && x == 0) lse[orow] = lsum > 0.0f ? (M + log2f(lsum)) * kLn2 : -INFINITY;
    }
  } else {
    // more chunks than the staging holds: per head, a pass for the maximum
    // and a pass for the weighted sums
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float M = append ? snew[h] : -INFINITY;
      for (int c = 0; c < nch; ++c) M = fmaxf(M, base[(int64_t)(c * G + h) * (D + 2) + D]);
      float a = 0.0f, lsum = 0.0f;
      for (int c = 0; c < nch; ++c) {
        const float* pc = base + (int64_t)(c * G + h) * (D + 2);
        const float mc = pc[D];
        const float f = (mc == -INFINITY) ? 0.0f : exp2f(mc - M);
        a += pc[x] * f;
        lsum += pc[D + 1] * f;
      }
      if (append) {
        const float f = exp2f(snew[h] - M);
        a += vn * f;
        lsum += f;
      }
      const int64_t orow = nrow * G + h;
      Elt<Tin>::put(out + orow * D, x, lsum > 0.0f ? a / lsum : 0.0f);
      if (lse && x == 0) lse[orow] = lsum > 0.0f ? (M + log2f(lsum)) * kLn2 : -INFINITY;
    }
  }
  __syncthreads();                      // every thread has read len[i] and the pool
  if (room && kq) {
    // group-quantised pool: the new row's codes and (scale, offset) per
    // group of 32 (warp w holds group w)
    const int64_t row = start[i] + L;
    quantize_elem(kn, lane, kq + row * D + x, kp + row * (D / 32) + warp);
    quantize_elem(vn, lane, vq + row * D + x, vp + row * (D / 32) + warp);
    if (x == 0) len[i] = L + 1;
  } else if (room) {
    const int64_t row = start[i] + L;
    if (sizeof(Tin) == 2) {
      reinterpret_cast<uint16_t*>(kc)[row * D + x] = reinterpret_cast<const uint16_t*>(k_new)[nrow * D + x];
      reinterpret_cast<uint16_t*>(vc)[row * D + x] = reinterpret_cast<const uint16_t*>(v_new)[nrow * D + x];
    } else {
      reinterpret_cast<float*>(kc)[row * D + x] = reinterpret_cast<const float*>(k_new)[nrow * D + x];
      reinterpret_cast<float*>(vc)[row * D + x] = reinterpret_cast<const float*>(v_new)[nrow * D + x];
    }
    if (x == 0) len[i] = L + 1;
  }
}

// Merge for a VECTOR cache: the chunks of the approximated rows hold
// sum_j p_j k_j (their K tile stood in for V), the others sum_j p_j v_j.  With
// both under one maximum and one normaliser, the output is
//   o = (sum_exact p_j v_j + W_g (sum_approx p_j k_j)) / l,
// i.e. every approximated value W_g k_j is rebuilt by one d x d product per
// query head instead of one per row (the reconstruction is linear).  The new
// token is appended as an exact row.
constexpr int kVecStaged = 64;   // chunks staged by the VECTOR merge (W takes most of its smem)

template <int D, int G>
__global__ void __launch_bounds__(D)
decode_combine_vector_kernel(const uint16_t* __restrict__ q, uint16_t* __restrict__ kc,
                             uint16_t* __restrict__ vc, const int64_t* __restrict__ kstart,
                             int32_t* __restrict__ klen, const int64_t* __restrict__ vstart,
                             const int32_t* __restrict__ napprox, const uint16_t* __restrict__ W,
                             const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                             int n_heads, int Hkv, int max_chunks, float scale_log2,
                             const float* __restrict__ ws, uint16_t* __restrict__ out,
                             float* __restrict__ lse, int* status) {
  constexpr int WS = D + 8;                // padded W row: 16-byte row reads spread over banks
  __shared__ float red[D / 32][G];
  __shared__ float ak_sm[G][D];
  __shared__ __align__(16) uint16_t w_sm[D * WS];
  const int i = blockIdx.x;
  const int u = i / Hkv, g = i - u * Hkv;
  const int x = threadIdx.x, lane = x & 31, warp = x >> 5;
  // W_g does not depend on the partial kernel: fetch it while that kernel drains
  for (int e = x; e < D * (D / 8); e += D) {
    const int r = e / (D / 8), ch = e - r * (D / 8);
    mmasync::cp_async16(smem_u32(w_sm + r * WS + ch * 8), W + ((int64_t)g * D + r) * D + ch * 8, 16u);
  }
  mmasync::cp_commit();
  // nor do the step's inputs (q, k_new, v_new) or the head's lengths: the
  // kernels that write klen (appends of earlier steps) completed before the
  // partial kernel let this one start (read from L2, past any line an
  // earlier kernel left in this SM's L1)
  const int L = __ldcg(klen + i);
  int na = __ldcg(napprox + i);
  if (na < 0 || na > L) { if (x == 0) report(status, KVC_ERR_RANGE); na = na < 0 ? 0 : L; }
  const int ne = L - na;
  const int cha = (na + 2 * kChunk - 1) / (2 * kChunk);    // chunks of 2048 approximated rows
  int nch = cha + (ne + kChunk - 1) / kChunk;
  if (nch > max_chunks) { if (x == 0) report(status, KVC_ERR_RANGE); nch = max_chunks; }
  const bool append = k_new != nullptr;
  bool room = append;
  if (append && i + 1 < n_heads &&
      (__ldcg(kstart + i) + L >= __ldcg(kstart + i + 1) ||
       __ldcg(vstart + i) + ne >= __ldcg(vstart + i + 1))) {
    if (x == 0) report(status, KVC_ERR_RANGE);
    room = false;
  }
  const int64_t nrow = (int64_t)u * Hkv + g;
  const float kn = append ? Elt<uint16_t>::get(k_new + nrow * D, x) : 0.0f;
  const float vn = append ? Elt<uint16_t>::get(v_new + nrow * D, x) : 0.0f;
  float snew[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float a = append ? Elt<uint16_t>::get(q + (nrow * G + h) * D, x) * kn : 0.0f;
#pragma unroll
    for (int off = 16; off; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
    if (lane == 0) red[warp][h] = a;
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float a = 0.0f;
#pragma unroll
    for (int w = 0; w < D / 32; ++w) a += red[w][h];
    snew[h] = a * scale_log2;
  }
  pdl_wait();
  pdl_trigger();
  const float* base = ws + (int64_t)i * max_chunks * G * (D + 2);
  float av[G], M[G], lsum[G];
  if (nch <= kVecStaged) {
    // as in decode_combine_kernel: every chunk's (max, sum) staged in shared
    // memory, one warp per head for the maxima and normalisers
    __shared__ float s_w[kVecStaged * G], s_l[kVecStaged * G];
    __shared__ float s_M[G], s_L[G];
    for (int e = x; e < nch * G; e += D) {
      const float* pc = base + (int64_t)e * (D + 2);
      s_w[e] = pc[D];
      s_l[e] = pc[D + 1];
    }
    __syncthreads();
    for (int h = warp; h < G; h += D / 32) {
      float m = append ? snew[h] : -INFINITY;
      for (int c = lane; c < nch; c += 32) m = fmaxf(m, s_w[c * G + h]);
#pragma unroll
      for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) s_M[h] = m;
    }
    __syncthreads();
    for (int e = x; e < nch * G; e += D) {
      const float mc = s_w[e];
      s_w[e] = (mc == -INFINITY) ? 0.0f : exp2f(mc - s_M[e % G]);
    }
    __syncthreads();
    for (int h = warp; h < G; h += D / 32) {
      float ls = 0.0f;
      for (int c = lane; c < nch; c += 32) ls += s_w[c * G + h] * s_l[c * G + h];
#pragma unroll
      for (int off = 16; off; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
      if (lane == 0) s_L[h] = ls;
    }
    __syncthreads();
    // chunks outer, heads inner: 4 x G loads in flight per thread
    float acc_k[G], acc_v[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc_k[h] = acc_v[h] = 0.0f;
#pragma unroll 4
    for (int c = 0; c < cha; ++c) {
      float pv[G];
#pragma unroll
      for (int h = 0; h < G; ++h) pv[h] = base[(int64_t)(c * G + h) * (D + 2) + x];
#pragma unroll
      for (int h = 0; h < G; ++h) acc_k[h] = fmaf(s_w[c * G + h], pv[h], acc_k[h]);
    }
#pragma unroll 4
    for (int c = cha; c < nch; ++c) {
      float pv[G];
#pragma unroll
      for (int h = 0; h < G; ++h) pv[h] = base[(int64_t)(c * G + h) * (D + 2) + x];
#pragma unroll
      for (int h = 0; h < G; ++h) acc_v[h] = fmaf(s_w[c * G + h], pv[h], acc_v[h]);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float a = acc_v[h], ak = acc_k[h];
      M[h] = s_M[h];
      lsum[h] = s_L[h];
      if (append) {
        const float f = exp2f(snew[h] - M[h]);
        a += vn * f;
        lsum[h] += f;
      }
      ak_sm[h][x] = ak;
      av[h] = a;
    }
  } else {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float m = append ? snew[h] : -INFINITY;
      for (int c = 0; c < nch; ++c) m = fmaxf(m, base[(int64_t)(c * G + h) * (D + 2) + D]);
      float a = 0.0f, ak = 0.0f, ls = 0.0f;
      for (int c = 0; c < nch; ++c) {
        const float* pc = base + (int64_t)(c * G + h) * (D + 2);
        const float mc = pc[D];
        const float f = (mc == -INFINITY) ? 0.0f : exp2f(mc - m);
        if (c < cha) ak += pc[x] * f; else a += pc[x] * f;
        ls += pc[D + 1] * f;
      }
      if (append) {
        const float f = exp2f(snew[h] - m);
        a += vn * f;
        ls += f;
      }
      ak_sm[h][x] = ak;
      av[h] = a;
      M[h] = m;
      lsum[h] = ls;
    }
  }
  mmasync::cp_wait<0>();
  __syncthreads();
  // out dimension x: sum_y W[g][x][y] * ak[h][y], the row read as 16-byte words
  float rec[G];
#pragma unroll
  for (int h = 0; h < G; ++h) rec[h] = 0.0f;
  const uint4* wrow = reinterpret_cast<const uint4*>(w_sm + x * WS);
#pragma unroll 4
  for (int ch = 0; ch < D / 8; ++ch) {
    const uint4 w4 = wrow[ch];
    const float wf[8] = {bf16lo(w4.x), bf16hi(w4.x), bf16lo(w4.y), bf16hi(w4.y),
                         bf16lo(w4.z), bf16hi(w4.z), bf16lo(w4.w), bf16hi(w4.w)};
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 8; ++e) rec[h] = fmaf(wf[e], ak_sm[h][ch * 8 + e], rec[h]);
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const int64_t orow = nrow * G + h;
    Elt<uint16_t>::put(out + orow * D, x, lsum[h] > 0.0f ? (av[h] + rec[h]) / lsum[h] : 0.0f);
    if (lse && x == 0) lse[orow] = lsum[h] > 0.0f ? (M[h] + log2f(lsum[h])) * kLn2 : -INFINITY;
  }
  __syncthreads();                      // every thread has read klen[i] and the pool
  if (room) {
    kc[(kstart[i] + L) * D + x] = k_new[nrow * D + x];
    vc[(vstart[i] + ne) * D + x] = v_new[nrow * D + x];
    if (x == 0) klen[i] = L + 1;
  }
}

// ---------------------------------------------------------------------------
// bf16 partial kernel on the tensor cores.  Per row of the cache the G query
// heads need G * d multiply-adds for q.k and again for p.v; done on the SIMT
// cores that is ~50-100 instructions per 512-byte row, which caps the kernel
// below the HBM rate.  Warp-level bf16 MMAs (m16n8k16, fp32 accumulate) do
// the same work in ~4 instructions per row: S = Q . K^T with the (<= 8)
// query heads as the M rows and 8 tokens per N tile, then O += P . V with P
// taken straight from the S accumulators.  The contraction is tiny (M = G
// padded to 16), so the warp-level MMA is the right size; the rows stream
// through a 3-stage cp.async ring whose 16-byte-padded rows make every
// ldmatrix conflict-free.
namespace mma {

using namespace ::kvc::mmasync;

constexpr int kRows = 64;      // rows per stage (16 per warp)
constexpr int kStg = 3;

// bf16 path: kStg stages of (K tile, V tile), kRows x (D + 8) bf16 each.
template <int D>
constexpr size_t smem_bytes() { return (size_t)kStg * 2 * kRows * (D + 8) * 2; }
// Quantised path: kQ8Stg stages of (K codes, V codes, K pairs, V pairs),
// code rows padded to D + 16 bytes; three CTAs fit an SM.
constexpr int kQ8Stg = 3;
template <int D>
constexpr int q8_row_bytes() { return D + 16; }
template <int D>
constexpr size_t q8_smem_bytes() {
  return (size_t)kQ8Stg * (2 * kRows * q8_row_bytes<D>() + 2 * kRows * (D / 8));
}

// D = A (16x16 f16, row) . B (16x8 f16, col) + C, fp32 accumulators.
__device__ __forceinline__ void mma_f16x4(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// The same with rows 8-15 of A zero.
__device__ __forceinline__ void mma_f16(float* d, uint32_t a0, uint32_t a2, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Two codes of w (the bytes `sel` picks into the low byte of each half) ->
// f16x2 code * scale + lo.  A code under the exponent byte 0x64 is the fp16
// 1024 + code (exact); 1024 is subtracted exactly, then one fused
// multiply-add rounds the value once to fp16.
__device__ __forceinline__ uint32_t deq2(uint32_t w, uint32_t sel, uint32_t sc2, uint32_t lo2) {
  const uint32_t h = __byte_perm(w, 0x64646464u, sel);
  uint32_t c, x;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(c) : "r"(h), "r"(0x64006400u));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(x) : "r"(c), "r"(sc2), "r"(lo2));
  return x;
}

}  // namespace mma

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32, 2)
decode_partial_mma_kernel(const uint16_t* __restrict__ q, const void* __restrict__ kc,
                          const void* __restrict__ vc, const int64_t* __restrict__ start,
                          const int32_t* __restrict__ len, int Hkv, int max_chunks,
                          float scale_log2, float* __restrict__ ws,
                          const int64_t* __restrict__ vstart, const int32_t* __restrict__ napprox) {
  static_assert(G <= 8, "query heads per kv head");
  constexpr int RS = D + 8;                  // padded row stride (elements)
  constexpr int CPR = D * 2 / 16;            // 16-byte chunks per row
  constexpr int NT = D / 8;                  // 8-wide output tiles
  extern __shared__ __align__(128) uint16_t smem_m[];
  __shared__ float m_sm[kWarps][G], l_sm[kWarps][G];
  __shared__ float acc_sm[kWarps][G][D];
  constexpr int STG = mma::kStg;             // stages in flight
  pdl_wait();
  pdl_trigger();

  const int i = blockIdx.y, c = blockIdx.x;
  const int L = len[i];
  // the chunk's rows: c * kChunk.. of the head, or (a VECTOR cache, napprox
  // set) the chunks of the napprox approximated rows first, whose values are
  // rebuilt from their keys later (the K tile stands in for the V tile), then
  // the chunks of the exact rows, whose values start at vstart[i]
  int rb = c * kChunk, seg = L;
  int64_t row0 = start[i] + rb, vrow0 = row0;
  bool k_as_v = false;
  if (napprox != nullptr) {
    // approximated rows stream K only: twice the rows per chunk and per stage
    // (the stage's V tile holds the next 64 keys), the same bytes as a chunk
    // of exact rows
    const int na = napprox[i];
    const int cha = (na + 2 * kChunk - 1) / (2 * kChunk);
    if (c < cha) {
      rb = c * 2 * kChunk;
      row0 = start[i] + rb;
      seg = na;
      k_as_v = true;
    } else {
      rb = (c - cha) * kChunk;
      seg = L - na;
      row0 = start[i] + na + rb;
      vrow0 = vstart[i] + rb;
    }
  }
  if (rb >= seg) return;
  const int SR = k_as_v ? 2 * mma::kRows : mma::kRows;      // rows per stage
  const int nrows = min(seg, rb + (k_as_v ? 2 * kChunk : kChunk)) - rb;
  const int nst = (nrows + SR - 1) / SR;
  const int u = i / Hkv, g = i - u * Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t sbase = smem_u32(smem_m);

  // stage st -> slot: K rows then V rows, each kRows x RS elements (bf16)
  auto issue = [&](int st) {
    const int slot = st % STG;
    const int r0 = st * mma::kRows;
    const uint16_t* kb = static_cast<const uint16_t*>(kc) + row0 * D;
    const uint16_t* vb = static_cast<const uint16_t*>(vc) + vrow0 * D;
    const uint32_t ks = sbase + (uint32_t)(slot * 2 * mma::kRows * RS) * 2u;
    const uint32_t vs = ks + (uint32_t)(mma::kRows * RS) * 2u;
    if (k_as_v) {
      // 128 keys: rows 64..127 land in the V tile, which follows the K tile
      const int r0k = st * 2 * mma::kRows;
      for (int x = tid; x < 2 * mma::kRows * CPR; x += kWarps * 32) {
        const int r = x / CPR, ch = x - r * CPR;
        const bool ok = r0k + r < nrows;
        const size_t off = (size_t)(ok ? r0k + r : 0) * D + ch * 8;
        mma::cp_async16(ks + (uint32_t)(r * RS + ch * 8) * 2u, kb + off, ok ? 16u : 0u);
      }
    } else {
      for (int x = tid; x < mma::kRows * CPR; x += kWarps * 32) {
        const int r = x / CPR, ch = x - r * CPR;
        const bool ok = r0 + r < nrows;
        const size_t off = (size_t)(ok ? r0 + r : 0) * D + ch * 8;
        const uint32_t so = (uint32_t)(r * RS + ch * 8) * 2u;
        mma::cp_async16(ks + so, kb + off, ok ? 16u : 0u);     // zero-fill past the end
        mma::cp_async16(vs + so, vb + off, ok ? 16u : 0u);
      }
    }
  };
  for (int st = 0; st < STG - 1; ++st) {
    if (st < nst) issue(st);
    mma::cp_commit();
  }

  // Q as the A operand: rows = query heads (lane / 4), 8 dims per register pair
  uint32_t qa[D / 16][2];
  {
    const int h = lane >> 2;
    const int d0 = (lane & 3) * 2;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      if (h < G) {
        const uint16_t* qp = q + ((int64_t)u * Hkv * G + (int64_t)g * G + h) * D + kk * 16 + d0;
        qa[kk][0] = *reinterpret_cast<const uint32_t*>(qp);
        qa[kk][1] = *reinterpret_cast<const uint32_t*>(qp + 8);
      } else {
        qa[kk][0] = qa[kk][1] = 0u;
      }
    }
  }
  float o[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.0f;
  float m = -INFINITY, l = 0.0f;                  // for head lane / 4 (lanes of a quad agree)

  for (int st = 0; st < nst; ++st) {
    mma::cp_wait<STG - 2>();
    __syncthreads();                              // stage st landed; slot st-1 is free
    if (st + STG - 1 < nst) issue(st + STG - 1);
    mma::cp_commit();
    const int slot = st % STG;
    const uint32_t ks = sbase + (uint32_t)(slot * 2 * mma::kRows * RS) * 2u;
    const uint32_t vs = ks + (uint32_t)(mma::kRows * RS) * 2u;
    auto tile_step = [&](uint32_t ks, uint32_t vs, int base) {
      const int wr = warp * 16;                     // this warp's 16 rows of the stage
      // ---- S = Q . K^T for 16 tokens (two 8-token tiles)
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int j = lane >> 3, r = lane & 7;
        const uint32_t rowaddr = ks + (uint32_t)((wr + (j >> 1) * 8 + r) * RS + (j & 1) * 8) * 2u;
  #pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t b[4];
          mma::ldsm_x4(rowaddr + kk * 32u, b);
          mma::mma_bf16(s0, qa[kk][0], 0u, qa[kk][1], 0u, b[0], b[1]);
          mma::mma_bf16(s1, qa[kk][0], 0u, qa[kk][1], 0u, b[2], b[3]);
        }
      }
      // ---- online softmax in base 2 over the 16 tokens (row = head lane / 4)
      const int tcol = (lane & 3) * 2;
      const int base_row = base + wr;
      float x0 = (base_row + tcol < nrows) ? s0[0] * scale_log2 : -INFINITY;
      float x1 = (base_row + tcol + 1 < nrows) ? s0[1] * scale_log2 : -INFINITY;
      float x2 = (base_row + 8 + tcol < nrows) ? s1[0] * scale_log2 : -INFINITY;
      float x3 = (base_row + 8 + tcol + 1 < nrows) ? s1[1] * scale_log2 : -INFINITY;
      float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mn = fmaxf(m, mx);
      float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
      if (mn != -INFINITY) {
        const float alpha = mma::ex2(m - mn);        // m = -inf -> 0
        l *= alpha;
  #pragma unroll
        for (int nt = 0; nt < NT; ++nt) { o[nt][0] *= alpha; o[nt][1] *= alpha; }
        p0 = mma::ex2(x0 - mn); p1 = mma::ex2(x1 - mn); p2 = mma::ex2(x2 - mn); p3 = mma::ex2(x3 - mn);
        l += (p0 + p1) + (p2 + p3);
        m = mn;
      }
      // ---- O += P . V: P (heads x 16 tokens) is the A operand
      const uint32_t pa0 = mma::pack_bf16(p0, p1), pa2 = mma::pack_bf16(p2, p3);
      {
        const int j = lane >> 3, r = lane & 7;
        const uint32_t rowaddr = vs + (uint32_t)((wr + (j & 1) * 8 + r) * RS + (j >> 1) * 8) * 2u;
  #pragma unroll
        for (int dn = 0; dn < D / 16; ++dn) {
          uint32_t b[4];
          mma::ldsm_x4_t(rowaddr + dn * 32u, b);
          mma::mma_bf16(o[2 * dn], pa0, 0u, pa2, 0u, b[0], b[1]);
          mma::mma_bf16(o[2 * dn + 1], pa0, 0u, pa2, 0u, b[2], b[3]);
        }
      }
    };
    if (k_as_v) {
      tile_step(ks, ks, st * 2 * mma::kRows);
      tile_step(ks + (uint32_t)(mma::kRows * RS) * 2u, ks + (uint32_t)(mma::kRows * RS) * 2u,
                st * 2 * mma::kRows + mma::kRows);
    } else {
      tile_step(ks, vs, st * mma::kRows);
    }
  }
  mma::cp_wait<0>();
  // quad sum of l, then per-warp partials to shared memory
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  const int h = lane >> 2;
  if (h < G) {
    if ((lane & 3) == 0) { m_sm[warp][h] = m; l_sm[warp][h] = l; }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      acc_sm[warp][h][nt * 8 + (lane & 3) * 2] = o[nt][0];
      acc_sm[warp][h][nt * 8 + (lane & 3) * 2 + 1] = o[nt][1];
    }
  }
  __syncthreads();
  float* out = ws + ((int64_t)i * max_chunks + c) * G * (D + 2);
  for (int e = tid; e < G * D; e += kWarps * 32) {
    const int hh = e / D, x = e - hh * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, m_sm[w][hh]);
    float a = 0.0f, lsum = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = (m_sm[w][hh] == -INFINITY) ? 0.0f : exp2f(m_sm[w][hh] - M);
      a += acc_sm[w][hh][x] * f;
      lsum += l_sm[w][hh] * f;
    }
    out[hh * (D + 2) + x] = a;
    if (x == 0) { out[hh * (D + 2) + D] = M; out[hh * (D + 2) + D + 1] = lsum; }
  }
}

// Partial kernel over a group-quantised pool (codes [rows, D] uint8, fp16
// (scale, lo) pairs [rows, D / 32]).  The raw codes and pairs stream through
// a cp.async ring (code rows padded to D + 16 bytes, so ldmatrix is
// conflict-free; rows past the chunk zero-filled, so they read as 0) and
// every warp dequantises its 16 rows of a stage straight into MMA operand
// registers (no bf16 tile, one barrier per stage):
//  * S = Q . K^T: ldmatrix hands a lane 4 consecutive codes (dims 16kk + 4t
//    .. +3) of token lane / 4; the contraction takes a k-step's 16 dims in
//    that order (the query fragment is loaded to match), so the 4 codes are
//    the lane's two B registers.
//  * O^T += V^T . P^T: ldmatrix.trans hands a lane the codes of tokens 2t,
//    2t+1 at dims 2g, 2g+1 of a 16-dim chunk, which are exactly the A
//    fragment of the chunk with its even dims as rows 0-7 and its odd dims as
//    rows 8-15; P from the S accumulators is the B fragment as it stands.
// Dequantisation is code * scale + lo rounded once to fp16 (three
// instructions per two codes); queries and probabilities enter the MMAs as
// fp16, products accumulate in fp32.  The accumulators are rescaled only when
// a head's running maximum moves.
template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32, 3)
decode_partial_q8_kernel(const uint16_t* __restrict__ q, const uint8_t* __restrict__ kq,
                         const uint8_t* __restrict__ vq, const uint32_t* __restrict__ kp,
                         const uint32_t* __restrict__ vp, const int64_t* __restrict__ start,
                         const int32_t* __restrict__ len, int Hkv, int max_chunks,
                         float scale_log2, float* __restrict__ ws) {
  static_assert(D == 128 && G <= 8, "shape");
  constexpr int RSB = mma::q8_row_bytes<D>();
  constexpr int PB = D / 8;                        // pair bytes per row (4 per 32 dims)
  constexpr int STG = mma::kQ8Stg;
  constexpr int MT = D / 16;                       // 16-dim output chunks
  constexpr uint32_t kCodeB = (uint32_t)(mma::kRows * RSB);
  constexpr uint32_t kParB = (uint32_t)(mma::kRows * PB);
  constexpr uint32_t kStageB = 2 * kCodeB + 2 * kParB;
  extern __shared__ __align__(128) uint8_t smem_q8[];
  __shared__ float m_sm[kWarps][G], l_sm[kWarps][G];
  pdl_wait();
  pdl_trigger();

  const int i = blockIdx.y, c = blockIdx.x;
  const int L = len[i];
  const int rb = c * kQ8Chunk;
  if (rb >= L) return;
  const int nrows = min(L, rb + kQ8Chunk) - rb;
  const int nst = (nrows + mma::kRows - 1) / mma::kRows;
  const int u = i / Hkv, g = i - u * Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t sbase = smem_u32(smem_q8);
  const int64_t row0 = start[i] + rb;

  // stage st -> slot: K codes, V codes, K pairs, V pairs
  auto issue = [&](int st) {
    const int slot = st % STG;
    const int r0 = st * mma::kRows;
    const uint32_t sk = sbase + (uint32_t)slot * kStageB, sv = sk + kCodeB;
    const uint32_t spk = sv + kCodeB, spv = spk + kParB;
    const uint8_t* kb = kq + row0 * D;
    const uint8_t* vb = vq + row0 * D;
    constexpr int CB = D / 16;                     // 16-byte code chunks per row
    for (int x = tid; x < mma::kRows * CB; x += kWarps * 32) {
      const int r = x / CB, ch = x - r * CB;
      const bool ok = r0 + r < nrows;
      const size_t off = (size_t)(ok ? r0 + r : 0) * D + ch * 16;
      const uint32_t so = (uint32_t)(r * RSB + ch * 16);
      mma::cp_async16(sk + so, kb + off, ok ? 16u : 0u);     // zero-fill past the end
      mma::cp_async16(sv + so, vb + off, ok ? 16u : 0u);
    }
    for (int r = tid; r < mma::kRows; r += kWarps * 32) {
      const bool ok = r0 + r < nrows;
      const size_t off = (size_t)(row0 + (ok ? r0 + r : 0)) * (D / 32);
      mma::cp_async16(spk + (uint32_t)(r * PB), kp + off, ok ? 16u : 0u);
      mma::cp_async16(spv + (uint32_t)(r * PB), vp + off, ok ? 16u : 0u);
    }
  };
  for (int st = 0; st < STG - 1; ++st) {
    if (st < nst) issue(st);
    mma::cp_commit();
  }

  // Q as the A operand (rows = query heads lane / 4), fp16, dims of k-step kk
  // in the order the K codes arrive: 16kk + 4t, +1 | 16kk + 4t + 2, +3
  const int t4 = lane & 3, gi = lane >> 2;
  uint32_t qa[D / 16][2];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    if (gi < G) {
      const uint16_t* qp = q + ((int64_t)u * Hkv * G + (int64_t)g * G + gi) * D + kk * 16 + 4 * t4;
      const uint2 w = *reinterpret_cast<const uint2*>(qp);
      qa[kk][0] = mma::pack_f16(bf16lo(w.x), bf16hi(w.x));
      qa[kk][1] = mma::pack_f16(bf16lo(w.y), bf16hi(w.y));
    } else {
      qa[kk][0] = qa[kk][1] = 0u;
    }
  }
  // o[s]: heads 2t, 2t+1 (columns) at dims 16s + 2g (c0, c1) and 16s + 2g + 1
  // (c2, c3), g = lane / 4
  float o[MT][4];
#pragma unroll
  for (int x = 0; x < MT; ++x) o[x][0] = o[x][1] = o[x][2] = o[x][3] = 0.0f;
  float m = -INFINITY, l = 0.0f;                  // for head lane / 4 (lanes of a quad agree)
  const int r8 = lane & 7, mi = lane >> 3;        // ldmatrix: row r8 of matrix mi

  for (int st = 0; st < nst; ++st) {
    mma::cp_wait<STG - 2>();
    __syncthreads();                              // stage st landed; slot st-1 is free
    if (st + STG - 1 < nst) issue(st + STG - 1);
    mma::cp_commit();
    const int slot = st % STG;
    const uint32_t sk = sbase + (uint32_t)slot * kStageB, sv = sk + kCodeB;
    const uint32_t spk = sv + kCodeB, spv = spk + kParB;
    const int wr = warp * 16;                     // this warp's 16 rows of the stage
    const int valid = nrows - st * mma::kRows - wr;   // rows of the 16 that exist

    // ---- S = Q . K^T for 16 tokens (two 8-token tiles)
    float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint4 pw = mma::lds128(spk + (uint32_t)((wr + 8 * nt + gi) * PB));   // token's pairs
      uint32_t sc2[4], lo2[4];
      sc2[0] = __byte_perm(pw.x, 0u, 0x1010u); lo2[0] = __byte_perm(pw.x, 0u, 0x3232u);
      sc2[1] = __byte_perm(pw.y, 0u, 0x1010u); lo2[1] = __byte_perm(pw.y, 0u, 0x3232u);
      sc2[2] = __byte_perm(pw.z, 0u, 0x1010u); lo2[2] = __byte_perm(pw.z, 0u, 0x3232u);
      sc2[3] = __byte_perm(pw.w, 0u, 0x1010u); lo2[3] = __byte_perm(pw.w, 0u, 0x3232u);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t b[4];
        mma::ldsm_x4(sk + (uint32_t)((wr + 8 * nt + r8) * RSB + (4 * half + mi) * 16), b);
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
          const int kk = 4 * half + m4;
          mma::mma_f16(sacc[nt], qa[kk][0], qa[kk][1],
                       mma::deq2(b[m4], 0x5140u, sc2[kk >> 1], lo2[kk >> 1]),
                       mma::deq2(b[m4], 0x5342u, sc2[kk >> 1], lo2[kk >> 1]));
        }
      }
    }
    // ---- online softmax in base 2 over the 16 tokens (row = head lane / 4)
    const int tcol = t4 * 2;
    const float x0 = (tcol < valid) ? sacc[0][0] * scale_log2 : -INFINITY;
    const float x1 = (tcol + 1 < valid) ? sacc[0][1] * scale_log2 : -INFINITY;
    const float x2 = (8 + tcol < valid) ? sacc[1][0] * scale_log2 : -INFINITY;
    const float x3 = (8 + tcol + 1 < valid) ? sacc[1][1] * scale_log2 : -INFINITY;
    float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(m, mx);
    float alpha = 1.0f, p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
    if (mn != -INFINITY) {
      if (mn > m) alpha = mma::ex2(m - mn);       // m = -inf -> 0
      p0 = mma::ex2(x0 - mn); p1 = mma::ex2(x1 - mn); p2 = mma::ex2(x2 - mn); p3 = mma::ex2(x3 - mn);
      l = l * alpha + ((p0 + p1) + (p2 + p3));
      m = mn;
    }
    if (__any_sync(0xffffffffu, alpha != 1.0f)) {
      // this lane's output columns are heads 2t and 2t+1
      const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * t4);
      const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * t4 + 4);
#pragma unroll
      for (int x = 0; x < MT; ++x) {
        o[x][0] *= a0; o[x][1] *= a1; o[x][2] *= a0; o[x][3] *= a1;
      }
    }
    // ---- O^T += V^T . P^T: P (16 tokens x heads) is the B operand
    const uint32_t pb0 = mma::pack_f16(p0, p1), pb1 = mma::pack_f16(p2, p3);
    {
      // pairs of tokens 2t, 2t+1 (k 2t, 2t+1) and 2t+8, 2t+9 (k 2t+8, 2t+9)
      const uint4 wa4 = mma::lds128(spv + (uint32_t)((wr + 2 * t4) * PB));
      const uint4 wb4 = mma::lds128(spv + (uint32_t)((wr + 2 * t4 + 1) * PB));
      const uint4 wc4 = mma::lds128(spv + (uint32_t)((wr + 8 + 2 * t4) * PB));
      const uint4 wd4 = mma::lds128(spv + (uint32_t)((wr + 9 + 2 * t4) * PB));
      // matrix mi: tokens wr + 8 (mi & 1) + r8 of chunk 2sp + (mi >> 1)
      const uint32_t vrow = sv + (uint32_t)((wr + 8 * (mi & 1) + r8) * RSB + (mi >> 1) * 16);
#pragma unroll
      for (int sp = 0; sp < D / 32; ++sp) {        // chunks 2sp, 2sp+1 share pair group sp
        uint32_t b[4];
        mma::ldsm_x4_t(vrow + (uint32_t)(sp * 32), b);
        const uint32_t wa = sp == 0 ? wa4.x : sp == 1 ? wa4.y : sp == 2 ? wa4.z : wa4.w;
        const uint32_t wb = sp == 0 ? wb4.x : sp == 1 ? wb4.y : sp == 2 ? wb4.z : wb4.w;
        const uint32_t wc = sp == 0 ? wc4.x : sp == 1 ? wc4.y : sp == 2 ? wc4.z : wc4.w;
        const uint32_t wd = sp == 0 ? wd4.x : sp == 1 ? wd4.y : sp == 2 ? wd4.z : wd4.w;
        const uint32_t sc_a = __byte_perm(wa, wb, 0x5410u), lo_a = __byte_perm(wa, wb, 0x7632u);
        const uint32_t sc_b = __byte_perm(wc, wd, 0x5410u), lo_b = __byte_perm(wc, wd, 0x7632u);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const uint32_t r0 = b[2 * cc], r1 = b[2 * cc + 1];   // tokens 0-7 / 8-15
          mma::mma_f16x4(o[2 * sp + cc],
                         mma::deq2(r0, 0x5240u, sc_a, lo_a),     // rows 0-7: even dims
                         mma::deq2(r0, 0x5341u, sc_a, lo_a),     // rows 8-15: odd dims
                         mma::deq2(r1, 0x5240u, sc_b, lo_b),
                         mma::deq2(r1, 0x5341u, sc_b, lo_b), pb0, pb1);
        }
      }
    }
  }
  mma::cp_wait<0>();
  __syncthreads();                                // every warp is done with the stages
  // quad sum of l, then per-warp partials to shared memory (the stage area)
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  float (*acc_sm)[G][D] = reinterpret_cast<float (*)[G][D]>(smem_q8);
  if (gi < G && t4 == 0) { m_sm[warp][gi] = m; l_sm[warp][gi] = l; }
  {
    const int h0 = 2 * t4, h1 = 2 * t4 + 1;
#pragma unroll
    for (int x = 0; x < MT; ++x) {
      const int dm = 16 * x + 2 * gi;
      if (h0 < G) { acc_sm[warp][h0][dm] = o[x][0]; acc_sm[warp][h0][dm + 1] = o[x][2]; }
      if (h1 < G) { acc_sm[warp][h1][dm] = o[x][1]; acc_sm[warp][h1][dm + 1] = o[x][3]; }
    }
  }
  __syncthreads();
  float* out = ws + ((int64_t)i * max_chunks + c) * G * (D + 2);
  for (int e = tid; e < G * D; e += kWarps * 32) {
    const int hh = e / D, x = e - hh * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, m_sm[w][hh]);
    float a = 0.0f, lsum = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = (m_sm[w][hh] == -INFINITY) ? 0.0f : exp2f(m_sm[w][hh] - M);
      a += acc_sm[w][hh][x] * f;
      lsum += l_sm[w][hh] * f;
    }
    out[hh * (D + 2) + x] = a;
    if (x == 0) { out[hh * (D + 2) + D] = M; out[hh * (D + 2) + D + 1] = lsum; }
  }
}

// A group-quantised pool (codes and fp16 (scale, offset) pairs per group of
// 32); all null for a bf16 / fp32 pool.
struct QPool {
  uint8_t* kq = nullptr;
  uint32_t* kp = nullptr;
  uint8_t* vq = nullptr;
  uint32_t* vp = nullptr;
};

template <typename Tin, int D, int G>
int run(const void* q, void* kc, void* vc, const QPool& qz, const int64_t* start, int32_t* len,
        const void* k_new, const void* v_new, int U, int Hkv, int max_len, float scale, void* out,
        float* lse, float* ws, const Dev& dev, cudaStream_t s) {
  const int n = U * Hkv;
  const int chunk = qz.kq ? kQ8Chunk : kChunk;
  const int max_chunks = (max_len + chunk - 1) / chunk;
  const float sl2 = scale * kLog2e;
  if (max_chunks > 0) {
    dim3 grid((unsigned)max_chunks, (unsigned)n);
    static std::atomic<uint64_t> attr_done{0};          // one bit per device and variant
    const uint64_t bit = 1ull << (dev.device & 31);
    if constexpr (sizeof(Tin) == 2 && G <= 8) {
      if (qz.kq) {
        if constexpr (D == 128) {
          const size_t smem = mma::q8_smem_bytes<D>();
          auto kern = decode_partial_q8_kernel<D, G>;
          if (!(attr_done.load() & (bit << 32))) {
            KVC_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
            attr_done.fetch_or(bit << 32);
          }
          if (int rc = prefer_max_shared(kern, dev.device)) return rc;
          if (int rc = launch_pdl(kern, grid, dim3(kWarps * 32), smem, s,
                                  static_cast<const uint16_t*>(q), (const uint8_t*)qz.kq,
                                  (const uint8_t*)qz.vq, (const uint32_t*)qz.kp,
                                  (const uint32_t*)qz.vp, start, (const int32_t*)len, Hkv,
                                  max_chunks, sl2, ws))
            return rc;
        } else {
          return KVC_ERR_UNSUPPORTED;
        }
      } else {
        const size_t smem = mma::smem_bytes<D>();
        auto kern = decode_partial_mma_kernel<D, G>;
        if (!(attr_done.load() & bit)) {
          KVC_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
          attr_done.fetch_or(bit);
        }
        if (int rc = prefer_max_shared(kern, dev.device)) return rc;
        if (int rc = launch_pdl(kern, grid, dim3(kWarps * 32), smem, s,
                                static_cast<const uint16_t*>(q), (const void*)kc, (const void*)vc,
                                start, (const int32_t*)len, Hkv, max_chunks, sl2, ws,
                                (const int64_t*)nullptr, (const int32_t*)nullptr))
          return rc;
      }
    } else {
      if (qz.kq) return KVC_ERR_UNSUPPORTED;
      const size_t smem = partial_smem_bytes<Tin, D>();
      auto kern = decode_partial_kernel<Tin, D, G>;
      if (!(attr_done.load() & bit)) {
        KVC_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        attr_done.fetch_or(bit);
      }
      if (int rc = prefer_max_shared(kern, dev.device)) return rc;
      if (int rc = launch_pdl(kern, grid, dim3((kWarps + 1) * 32), smem, s,
                              static_cast<const Tin*>(q), static_cast<const Tin*>(kc),
                              static_cast<const Tin*>(vc), start, (const int32_t*)len, Hkv,
                              max_chunks, sl2, ws, dev.status))
        return rc;
    }
  }
  if (int rc = prefer_max_shared(decode_combine_kernel<Tin, D, G>, dev.device)) return rc;
  return launch_pdl(decode_combine_kernel<Tin, D, G>, dim3((unsigned)n), dim3(D), 0, s,
                    static_cast<const Tin*>(q), static_cast<Tin*>(kc), static_cast<Tin*>(vc),
                    start, len, static_cast<const Tin*>(k_new), static_cast<const Tin*>(v_new),
                    n, Hkv, max_chunks, sl2, (const float*)ws, static_cast<Tin*>(out), lse,
                    dev.status, qz.kq, qz.kp, qz.vq, qz.vp, chunk);
}

template <typename Tin, int D>
int dispatch_g(int G, const void* q, void* kc, void* vc, const QPool& qz, const int64_t* start,
               int32_t* len, const void* kn, const void* vn, int U, int Hkv, int max_len,
               float scale, void* out, float* lse, float* ws, const Dev& dev, cudaStream_t s) {
  switch (G) {
#define KVC_G(GG) \
    case GG: return run<Tin, D, GG>(q, kc, vc, qz, start, len, kn, vn, U, Hkv, max_len, scale, out, lse, ws, dev, s);
    KVC_G(1) KVC_G(2) KVC_G(3) KVC_G(4) KVC_G(5) KVC_G(6) KVC_G(7) KVC_G(8)
#undef KVC_G
  }
  return KVC_ERR_UNSUPPORTED;
}

template <int G>
int run_vector(const void* q, void* kc, void* vc, const int64_t* kstart, int32_t* klen,
               const int64_t* vstart, const int32_t* napprox, const void* W, const void* k_new,
               const void* v_new, int U, int Hkv, int max_len, float scale, void* out,
               float* lse, float* ws, const Dev& dev, cudaStream_t s) {
  constexpr int D = 128;
  const int n = U * Hkv;
  // approximated and exact rows are chunked apart: one chunk more at most
  const int max_chunks = (max_len + kChunk - 1) / kChunk + 1;
  const float sl2 = scale * kLog2e;
  const size_t smem = mma::smem_bytes<D>();
  auto kern = decode_partial_mma_kernel<D, G>;
  static std::atomic<uint32_t> attr_done{0};            // one bit per device
  const uint32_t bit = 1u << (dev.device & 31);
  if (!(attr_done.load() & bit)) {
    KVC_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    attr_done.fetch_or(bit);
  }
  if (int rc = prefer_max_shared(kern, dev.device)) return rc;
  if (int rc = launch_pdl(kern, dim3((unsigned)max_chunks, (unsigned)n), dim3(kWarps * 32), smem,
                          s, static_cast<const uint16_t*>(q), (const void*)kc, (const void*)vc,
                          kstart, (const int32_t*)klen, Hkv, max_chunks, sl2, ws, vstart, napprox))
    return rc;
  auto comb = decode_combine_vector_kernel<D, G>;
  if (int rc = prefer_max_shared(comb, dev.device)) return rc;
  return launch_pdl(comb, dim3((unsigned)n), dim3(D), 0, s, static_cast<const uint16_t*>(q),
                    static_cast<uint16_t*>(kc), static_cast<uint16_t*>(vc), kstart, klen, vstart,
                    napprox, static_cast<const uint16_t*>(W),
                    static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new), n,
                    Hkv, max_chunks, sl2, (const float*)ws, static_cast<uint16_t*>(out), lse,
                    dev.status);
}

}  // namespace

size_t decode_vector_ws_bytes(int U, int Hq, int Hkv, int d, int max_len) {
  const int64_t chunks = (max_len + kChunk - 1) / kChunk + 1;
  return (size_t)U * Hkv * chunks * (Hq / Hkv) * (d + 2) * sizeof(float);
}

int decode_vector_launch(const void* q, void* kc, void* vc, const int64_t* kstart,
                         int32_t* klen, const int64_t* vstart, const int32_t* napprox,
                         const void* W, const void* k_new, const void* v_new, int U, int Hq,
                         int Hkv, int max_len, float scale, void* out, float* lse, float* ws,
                         const Dev& dev, cudaStream_t s) {
  switch (Hq / Hkv) {
#define KVC_G(GG) \
    case GG: return run_vector<GG>(q, kc, vc, kstart, klen, vstart, napprox, W, k_new, v_new, U, Hkv, max_len, scale, out, lse, ws, dev, s);
    KVC_G(1) KVC_G(2) KVC_G(3) KVC_G(4) KVC_G(5) KVC_G(6) KVC_G(7) KVC_G(8)
#undef KVC_G
  }
  return KVC_ERR_UNSUPPORTED;
}

size_t decode_ws_bytes(int U, int Hq, int Hkv, int d, int max_len) {
  const int64_t chunks = (max_len + kChunk - 1) / kChunk;
  return (size_t)U * Hkv * chunks * (Hq / Hkv) * (d + 2) * sizeof(float);
}

int decode_launch(const void* q, void* kc, void* vc, const int64_t* start, int32_t* len,
                  const void* k_new, const void* v_new, int dtype, int U, int Hq, int Hkv,
                  int d, int max_len, float scale, void* out, float* lse, float* ws,
                  const Dev& dev, cudaStream_t s) {
  const int G = Hq / Hkv;
  const QPool none;
  if (dtype == KVC_F32)
    return d == 64 ? dispatch_g<float, 64>(G, q, kc, vc, none, start, len, k_new, v_new, U, Hkv, max_len, scale, out, lse, ws, dev, s)
                   : dispatch_g<float, 128>(G, q, kc, vc, none, start, len, k_new, v_new, U, Hkv, max_len, scale, out, lse, ws, dev, s);
  return d == 64 ? dispatch_g<uint16_t, 64>(G, q, kc, vc, none, start, len, k_new, v_new, U, Hkv, max_len, scale, out, lse, ws, dev, s)
                 : dispatch_g<uint16_t, 128>(G, q, kc, vc, none, start, len, k_new, v_new, U, Hkv, max_len, scale, out, lse, ws, dev, s);
}

int decode_q8_launch(const void* q, uint8_t* kq, void* kp, uint8_t* vq, void* vp,
                     const int64_t* start, int32_t* len, const void* k_new, const void* v_new,
                     int U, int Hq, int Hkv, int max_len, float scale, void* out, float* lse,
                     float* ws, const Dev& dev, cudaStream_t s) {
  QPool qz;
  qz.kq = kq; qz.kp = static_cast<uint32_t*>(kp);
  qz.vq = vq; qz.vp = static_cast<uint32_t*>(vp);
  return dispatch_g<uint16_t, 128>(Hq / Hkv, q, nullptr, nullptr, qz, start, len, k_new, v_new,
                                   U, Hkv, max_len, scale, out, lse, ws, dev, s);
}

int quantize_rows_launch(const void* x, int64_t rows, int d, uint8_t* codes, void* params,
                         const Dev& dev, cudaStream_t s) {
  if (rows <= 0) return KVC_OK;
  const int64_t want = (rows + 7) / 8;
  const unsigned blocks = (unsigned)(want < (int64_t)dev.sms * 8 ? want : (int64_t)dev.sms * 8);
  auto kern = d == 64 ? quantize_rows_kernel<64> : quantize_rows_kernel<128>;
  return launch_pdl(kern, dim3(blocks), dim3(256), 0, s, static_cast<const uint16_t*>(x), rows,
                    codes, static_cast<uint32_t*>(params));
}

}  // namespace kvc
