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
    float g = ps[0], u = ps[u_off];
    for (int sp = 1; sp < splits; ++sp) {
      g += ps[sp * pstride];
      u += ps[sp * pstride + u_off];
    }
    float v = g / (1.f + expf(-g)) * u;
    if (row_w != nullptr) v *= row_w[(long)s * ldw + c / seg];
    h[(long)s * ldh + c] = __float2half_rn(v);
  }
}

// (value, id) order of the routing: larger logit first, ties to the lower id.
__device__ __forceinline__ bool route_better(float v, int e, float bv, int be) {
  return v > bv || (v == bv && e < be);
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
  __syncthreads();
  return excl;
}

constexpr int kRouteThreads = 1024;
constexpr int kMaxExperts = 1024;
constexpr int kMaxRows = 32;
constexpr int kMaxTopK = 32;

// One block: warp s routes row s; then the block groups the selections.
// SLOTS = logits per lane (E <= 32 * SLOTS), kept in registers.
template <int SLOTS>
__global__ void __launch_bounds__(kRouteThreads) moe_route_kernel(
    const float* __restrict__ logits, int S, int E, int top_k, int32_t* __restrict__ ids,
    float* __restrict__ w, int32_t* __restrict__ offsets, int32_t* __restrict__ pair_rows,
    int32_t* __restrict__ n_hit, int32_t* __restrict__ hit, float* __restrict__ row_w, int n_cap) {
  __shared__ int s_ids[kMaxRows][kMaxTopK];
  __shared__ float s_val[kMaxRows][kMaxTopK];
  __shared__ int cnt[kMaxExperts];
  __shared__ int slot[kMaxExperts];
  __shared__ int wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  griddep_wait();
  griddep_launch_dependents();  // the GEMM that follows may take the other SMs now
  for (int e = tid; e < kMaxExperts; e += blockDim.x) cnt[e] = 0;
  __syncthreads();

  // ---- route: top_k by repeated warp argmax over the unselected experts ----
  // lane holds experts lane + 32 m in registers; bit m of `taken` marks a selection
  if (warp < S) {
    const float* const row = logits + (long)warp * E;
    constexpr int kSlots = SLOTS;
    float lv[kSlots];
#pragma unroll
    for (int m = 0; m < kSlots; ++m) {
      const int e = lane + 32 * m;
      lv[m] = (e < E) ? row[e] : 0.f;
    }
    uint32_t taken = 0u;
    float first = 0.f, sum = 0.f;
    for (int i = 0; i < top_k; ++i) {
      float bv = -__int_as_float(0x7f800000);  // -inf
      int be = INT32_MAX;
#pragma unroll
      for (int m = 0; m < kSlots; ++m) {
        const int e = lane + 32 * m;
        if (e < E && !((taken >> m) & 1u) && route_better(lv[m], e, bv, be)) {
          bv = lv[m];
          be = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oe = __shfl_xor_sync(0xffffffffu, be, off);
        if (route_better(ov, oe, bv, be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (lane == 0) {
        s_ids[warp][i] = be;
        s_val[warp][i] = bv;
      }
      if (i == 0) first = bv;
    }
    __syncwarp();  // lane 0's writes, visible to the whole warp
    // softmax over the selection (the first selected logit is the largest)
    for (int i = 0; i < top_k; ++i) sum += expf(s_val[warp][i] - first);
    if (lane < top_k) {
      ids[warp * top_k + lane] = s_ids[warp][lane];
      w[warp * top_k + lane] = expf(s_val[warp][lane] - first) / sum;
    }
  }
  __syncthreads();

  // ---- group: per-expert counts, offsets, hit slots ----
  const int pairs = S * top_k;
  for (int pidx = tid; pidx < pairs; pidx += blockDim.x) atomicAdd(&cnt[s_ids[pidx / top_k][pidx % top_k]], 1);
  __syncthreads();
  int total = 0;
  const int c = (tid < E) ? cnt[tid] : 0;
  const int off = block_excl_scan(c, wsum, &total);
  if (tid < E) offsets[tid] = off;
  if (tid == 0) offsets[E] = total;
  int nh = 0;
  const int f = (c > 0) ? 1 : 0;
  const int sl = block_excl_scan(f, wsum, &nh);
  if (tid < E) {
    slot[tid] = sl;
    if (f) hit[sl] = tid;
  }
  if (tid == 0) *n_hit = nh;
  // zero the routing-weight table, then fill it and the per-expert row lists
  if (row_w != nullptr)
    for (int v = tid; v < S * n_cap; v += blockDim.x) row_w[v] = 0.f;
  for (int e = tid; e < kMaxExperts; e += blockDim.x) cnt[e] = (e < E) ? offsets[e] : 0;
  __syncthreads();
  for (int pidx = tid; pidx < pairs; pidx += blockDim.x) {
    const int s = pidx / top_k, i = pidx - s * top_k;
    const int e = s_ids[s][i];
    // rows before s that also selected e (each row selects an expert at most once)
    int before = 0;
    for (int s2 = 0; s2 < s; ++s2)
      for (int i2 = 0; i2 < top_k; ++i2) before += (s_ids[s2][i2] == e) ? 1 : 0;
    pair_rows[cnt[e] + before] = s;
    if (row_w != nullptr) row_w[s * n_cap + slot[e]] = w[pidx];
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
