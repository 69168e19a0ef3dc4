// Small kernels of the SwiGLU projections and the gathered-expert MoE:
//  * the split-K reduce that applies SwiGLU ("Flagship dramatic-speedup plan --
//    the full stackable tuning set", section "Axis 4 -- kernel micro-opts": the
//    fused SwiGLU MLP), optionally scaled per row and expert segment by the
//    routing weights;
//  * MoE routing and grouping (same page, section "Baseline byte model": routed
//    experts through gather_qmm, top-8 of 256).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "moe_route.cuh"
#include "sdv_device.cuh"
#include "sdv_kernels.h"

namespace sdv {

namespace {

// h[s][c] = fp16(SiLU(g) * u [* row_w[s][c / seg]]), g and u summed over the
// split-K partials in split order; SiLU(t) = t / (1 + exp(-t)).
__global__ void swiglu_reduce_kernel(const float* __restrict__ part, int splits, long pstride, int ldp, long u_off,
                                     int S, int n, __half* __restrict__ h, int ldh,
                                     const float* __restrict__ row_w, int ldw, int seg,
                                     const int* __restrict__ n_dev) {
  griddep_wait();
  griddep_launch_dependents();
  const int ncols = (n_dev != nullptr) ? min(n, *n_dev * seg) : n;
  const long count = (long)S * ncols;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += (long)gridDim.x * blockDim.x) {
    const int s = (int)(i / ncols), c = (int)(i - (long)s * ncols);
    const float* const ps = part + (long)s * ldp + c;
    // the splits' loads in batches of 8 (independent, one L2 round trip per
    // batch), the sums in split order
    float g = 0.f, u = 0.f;
    for (int sp0 = 0; sp0 < splits; sp0 += 8) {
      float bg[8], bu[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int sp = sp0 + j;
        bg[j] = sp < splits ? __ldcg(ps + (long)sp * pstride) : 0.f;
        bu[j] = sp < splits ? __ldcg(ps + (long)sp * pstride + u_off) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (sp0 + j >= splits) break;
        g = (sp0 + j == 0) ? bg[j] : g + bg[j];
        u = (sp0 + j == 0) ? bu[j] : u + bu[j];
      }
    }
    float v = g / (1.f + expf(-g)) * u;
    if (row_w != nullptr) v *= row_w[(long)s * ldw + c / seg];
    h[(long)s * ldh + c] = __float2half_rn(v);
  }
}

// Exclusive prefix sum over the block (blockDim.x == 1024); returns the
// exclusive sum of thread tid's value and writes the total to *total.
__device__ int block_excl_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int t = wsum[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += o;
    }
    wsum[lane] = t;
  }
  __syncthreads();
  const int excl = incl - v + (warp > 0 ? wsum[warp - 1] : 0);
  *total = wsum[31];
  return excl;
}

constexpr int kRouteThreads = 1024;
constexpr int kMaxExperts = 1024;
constexpr int kMaxRows = 32;
constexpr int kMaxTopK = 32;

// One block.  Warp s routes row s (route_row: larger logit first, ties to the
// lower id, softmax-renormalised weights).  Each selection then counts its
// expert and marks its row in the expert's row mask.  The block scans the packed (count, hit) pairs of all
// experts at once; a selection's place among its expert's rows is the number of
// lower rows in the mask.
template <int SLOTS>
__global__ void __launch_bounds__(kRouteThreads) moe_route_kernel(
    const float* __restrict__ logits, int S, int E, int top_k, int32_t* __restrict__ ids,
    float* __restrict__ w, int32_t* __restrict__ offsets, int32_t* __restrict__ pair_rows,
    int32_t* __restrict__ n_hit, int32_t* __restrict__ hit, float* __restrict__ row_w, int n_cap) {
  __shared__ int s_ids[kMaxRows][kMaxTopK];
  __shared__ float s_w[kMaxRows][kMaxTopK];
  __shared__ int cnt[kMaxExperts];
  __shared__ uint32_t rowmask[kMaxExperts];
  __shared__ int s_off[kMaxExperts];
  __shared__ int s_slot[kMaxExperts];
  __shared__ int wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  griddep_wait();
  griddep_launch_dependents();  // the GEMM that follows may take the other SMs now
  for (int e = tid; e < kMaxExperts; e += blockDim.x) {
    cnt[e] = 0;
    rowmask[e] = 0u;
  }
  __syncthreads();

  // ---- route ----
  if (warp < S) {
    route_row<SLOTS>(logits + (long)warp * E, E, top_k, lane, s_ids[warp], s_w[warp]);
    if (lane < top_k) {
      const int e = s_ids[warp][lane];
      const float wt = s_w[warp][lane];
      ids[warp * top_k + lane] = e;
      w[warp * top_k + lane] = wt;
      atomicAdd(&cnt[e], 1);
      atomicOr(&rowmask[e], 1u << warp);
    }
  }
  __syncthreads();

  // ---- group: one scan of (count << 16 | hit) over the experts ----
  const int c = (tid < E) ? cnt[tid] : 0;
  int total = 0;
  const int packed = block_excl_scan((c << 16) | (c > 0 ? 1 : 0), wsum, &total);
  if (tid < E) {
    const int off = packed >> 16, sl = packed & 0xFFFF;
    s_off[tid] = off;
    s_slot[tid] = sl;
    offsets[tid] = off;
    if (c > 0) hit[sl] = tid;
  }
  if (tid == 0) {
    offsets[E] = total >> 16;
    *n_hit = total & 0xFFFF;
  }
  if (row_w != nullptr)
    for (int v = tid; v < S * n_cap; v += blockDim.x) row_w[v] = 0.f;
  __syncthreads();
  const int pairs = S * top_k;
  for (int pidx = tid; pidx < pairs; pidx += blockDim.x) {
    const int s = pidx / top_k, i = pidx - s * top_k;
    const int e = s_ids[s][i];
    pair_rows[s_off[e] + __popc(rowmask[e] & ((1u << s) - 1u))] = s;
    if (row_w != nullptr) row_w[s * n_cap + s_slot[e]] = s_w[s][i];
  }
}

}  // namespace

cudaError_t launch_swiglu_reduce(const float* part, int splits, long pstride, int ldp, long u_off, int S, int n,
                                 __half* h, int ldh, const float* row_w, int ldw, int seg, const int* n_dev,
                                 cudaStream_t st) {
  long grid = ((long)S * n + 255) / 256;
  if (grid > 4096) grid = 4096;
  if (grid < 1) grid = 1;
  return launch_pdl(swiglu_reduce_kernel, dim3((unsigned)grid), dim3(256), 0, st, part, splits, pstride, ldp, u_off,
                    S, n, h, ldh, row_w, ldw, seg > 0 ? seg : 1, n_dev);
}

cudaError_t launch_moe_route(const float* logits, int S, int E, int top_k, int32_t* ids, float* w,
                             int32_t* offsets, int32_t* pair_rows, int32_t* n_hit, int32_t* hit, float* row_w,
                             int n_cap, cudaStream_t st) {
  if (S < 1 || S > kMaxRows || E < 1 || E > kMaxExperts || top_k < 1 || top_k > kMaxTopK || top_k > E)
    return cudaErrorInvalidValue;
  if (E <= 256)
    return launch_pdl(moe_route_kernel<8>, dim3(1), dim3(kRouteThreads), 0, st, logits, S, E, top_k, ids, w,
                      offsets, pair_rows, n_hit, hit, row_w, n_cap);
  return launch_pdl(moe_route_kernel<kMaxExperts / 32>, dim3(1), dim3(kRouteThreads), 0, st, logits, S, E, top_k,
                    ids, w, offsets, pair_rows, n_hit, hit, row_w, n_cap);
}

}  // namespace sdv
