// Small kernels of the verify path: the per-block-32 quantiser, the
// stand-alone greedy and tree accepts, and the tail of the split-reduction head.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cstdint>

#include "sdv_device.cuh"
#include "sdv_kernels.h"

namespace sdv {

namespace {

// One warp per block of 32 weights ("Riding Apple's pipelined GPU engine",
// section "Quantization on the GPU delegate": per-block-32 absmax symmetric).
// s32 = max|w| / Q (IEEE fp32 division), s16 = fp16(s32) round-to-nearest-even,
// q = clamp(rint(w / s16), -Q, Q) with rint ties-to-even; s16 == 0 gives q = 0.
// QB = 2: FP4 (E2M1) codes -- Q = 6, r = w / s16 rounded to the nearest E2M1
// magnitude (0, 0.5, 1, 1.5, 2, 3, 4, 6) with ties to the even mantissa bit,
// saturating; sign bit 8 for r < 0 unless the magnitude is 0.
template <int QB>
__global__ void quantize_block32_kernel(const float* __restrict__ w, long nblocks, int k,
                                        uint8_t* __restrict__ codes, __half* __restrict__ scales) {
  constexpr float kQ = (QB == 8) ? 127.f : (QB == 4 ? 7.f : 6.f);
  const int lane = threadIdx.x & 31;
  const long warps = (long)gridDim.x * (blockDim.x >> 5);
  const int kb = k / 32;
  for (long b = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < nblocks; b += warps) {
    const long row = b / kb, blk = b - row * kb;
    const float v = w[row * k + blk * 32 + lane];
    float m = fabsf(v);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const __half s16 = __float2half_rn(__fdiv_rn(m, kQ));
    const float sf = __half2float(s16);
    int q = 0;
    if (sf != 0.f) {
      if (QB == 2) {
        const float r = __fdiv_rn(v, sf), a = fabsf(r);
        // magnitude index = thresholds passed; a tie rounds to the even mantissa
        const int idx = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) +
                        (a > 5.f);
        q = idx | ((r < 0.f && idx > 0) ? 8 : 0);
      } else {
        const float r = rintf(__fdiv_rn(v, sf));
        q = (int)fminf(fmaxf(r, -kQ), kQ);
      }
    }
    if (QB == 8) {
      codes[row * k + blk * 32 + lane] = (uint8_t)(int8_t)q;
    } else {
      const int hi = __shfl_down_sync(0xffffffffu, q, 1);
      if ((lane & 1) == 0)
        codes[row * (k / 2) + blk * 16 + lane / 2] = (uint8_t)((q & 0xF) | ((hi & 0xF) << 4));
    }
    if (lane == 0) scales[row * kb + blk] = s16;
  }
}

// Greedy longest-prefix accept ("Stream C -- Speculative decoding: feasibility
// verdict + implementation plan", section "The delta"): accept d_i while
// d_i == argmax[i] for i < n_valid; the next a0 is argmax[accepted].
__global__ void greedy_accept_kernel(const int32_t* __restrict__ argmax, const int32_t* __restrict__ drafts,
                                     int n_valid, int32_t* accepted, int32_t* next_a0) {
  if (threadIdx.x != 0) return;
  int j = 0;
  while (j < n_valid && drafts[j] == argmax[j]) ++j;
  *accepted = j;
  *next_a0 = argmax[j];
}

// Tree accept over S <= 32 nodes, one warp: lane i walks up from node i and
// finds whether every edge (p -> c) on the way has tokens[c] == argmax[p]; the
// deepest accepted node (lowest index among equals) wins; lane 0 writes its
// path from the root's child down and argmax of that node.  A parent index
// outside [0, i) marks an absent (pad) node.
__global__ void tree_accept_kernel(const int32_t* __restrict__ argmax, int S, const int32_t* __restrict__ tokens,
                                   const int32_t* __restrict__ parent, int32_t* path, int32_t* accepted,
                                   int32_t* next_a0) {
  __shared__ int s_am[32], s_tok[32], s_par[32];
  const int lane = threadIdx.x;
  if (lane < S) {
    s_am[lane] = argmax[lane];
    s_tok[lane] = lane > 0 ? tokens[lane] : 0;
    s_par[lane] = lane > 0 ? parent[lane] : -1;
  }
  __syncwarp();
  int depth = -1;  // -1: not accepted
  if (lane == 0) {
    depth = 0;
  } else if (lane < S) {
    int j = lane, d = 0;
    bool ok = true;
    while (j != 0) {  // at most 31 steps: every step moves to a smaller index
      const int p = s_par[j];
      if (p < 0 || p >= j || s_tok[j] != s_am[p]) {
        ok = false;
        break;
      }
      j = p;
      ++d;
    }
    if (ok) depth = d;
  }
  // deepest, then lowest index
  int best_d = depth, best_i = lane;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const int od = __shfl_xor_sync(0xffffffffu, best_d, off);
    const int oi = __shfl_xor_sync(0xffffffffu, best_i, off);
    if (od > best_d || (od == best_d && oi < best_i)) {
      best_d = od;
      best_i = oi;
    }
  }
  if (lane == 0) {
    for (int j = best_i, k = best_d - 1; j != 0; j = s_par[j], --k) path[k] = j;
    *accepted = best_d;
    *next_a0 = s_am[best_i];
  }
}

// Tail of the verify head when the window's rows fit the tensor-core plan only
// with the reduction split (e.g. k = 2560 at S >= 17): the split GEMM has written
// fp32 partial logits part[split][s][v]; here logits[s][v] = their sum in split
// order (written when `logits` is not null), each CTA reduces its slab of the
// vocabulary to per-row (max, lowest index) partials, and the last CTA to finish
// (acquire-release ticket) merges them, writes argmax[S] and runs the greedy accept
// ("Stream C -- Speculative decoding: feasibility verdict + implementation plan",
// section "The delta").
constexpr int kSplitSumThreads = 256;

__global__ void __launch_bounds__(kSplitSumThreads) head_splitsum_kernel(
    const float* __restrict__ part, int splits, int S, int n, float* __restrict__ logits, float* part_v, int* part_i,
    const int32_t* __restrict__ drafts, int n_valid, int32_t* argmax, int32_t* accepted, int32_t* next_a0,
    unsigned* ticket) {
  griddep_wait();
  __shared__ float s_v[kSplitSumThreads / 32][32];
  __shared__ int s_i[kSplitSumThreads / 32][32];
  __shared__ int s_am[32], s_dr[32], s_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = (int)((long)blockIdx.x * n / gridDim.x), c1 = (int)((long)(blockIdx.x + 1) * n / gridDim.x);
  const long plane = (long)S * n;  // one split's partials
  float bv[32];
  int bi[32];
#pragma unroll
  for (int s = 0; s < 32; ++s) {
    bv[s] = -FLT_MAX;
    bi[s] = INT_MAX;
  }
  for (int v = c0 + threadIdx.x; v < c1; v += kSplitSumThreads) {
#pragma unroll
    for (int s = 0; s < 32; ++s) {
      if (s < S) {
        const float* pp = part + (long)s * n + v;
        float val = __ldcg(pp);
        for (int sp = 1; sp < splits; ++sp) val += __ldcg(pp + sp * plane);
        if (logits != nullptr) logits[(long)s * n + v] = val;
        argmax_merge(bv[s], bi[s], val, v);
      }
    }
  }
  // per row: the warp's best, then the block's (one warp per row group of 32)
#pragma unroll
  for (int s = 0; s < 32; ++s) {
    if (s < S) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv[s], off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi[s], off);
        argmax_merge(bv[s], bi[s], ov, oi);
      }
      if (lane == 0) {
        s_v[warp][s] = bv[s];
        s_i[warp][s] = bi[s];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < S) {
    const int s = threadIdx.x;
    float v = s_v[0][s];
    int i = s_i[0][s];
    for (int w = 1; w < kSplitSumThreads / 32; ++w) argmax_merge(v, i, s_v[w][s], s_i[w][s]);
    __stcg(part_v + (long)blockIdx.x * S + s, v);
    __stcg(part_i + (long)blockIdx.x * S + s, i);
  }
  // The next kernel in the stream may launch once every block is past its
  // share of the sum: triggered earlier, its CTAs (which wait for this grid to
  // complete) would take SMs that blocks of this grid have yet to run on.
  griddep_launch_dependents();
  __syncthreads();
  if (threadIdx.x == 0) {
    // publishes this CTA's partials (cumulative over the block's stores before the
    // barrier) and, for the last CTA, acquires everyone else's
    unsigned tk;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(tk) : "l"(ticket) : "memory");
    s_flag = (tk == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (s_flag == 0) return;
  for (int s = warp; s < S; s += kSplitSumThreads / 32) {
    float v = -FLT_MAX;
    int i = INT_MAX;
    for (int j = lane; j < (int)gridDim.x; j += 32)
      argmax_merge(v, i, __ldcg(part_v + (long)j * S + s), __ldcg(part_i + (long)j * S + s));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, off);
      const int oi = __shfl_xor_sync(0xffffffffu, i, off);
      argmax_merge(v, i, ov, oi);
    }
    if (lane == 0) {
      s_am[s] = i;
      argmax[s] = i;
    }
  }
  if (threadIdx.x < n_valid) s_dr[threadIdx.x] = drafts[threadIdx.x];
  __syncthreads();
  if (warp == 0) {  // accepted = the first window position whose draft misses (n_valid <= 31)
    const bool hit = lane < n_valid && s_dr[lane] == s_am[lane];
    const unsigned miss = ~__ballot_sync(0xffffffffu, hit);
    const int j = __ffs(miss) - 1;
    if (lane == 0) {
      *accepted = j;
      *next_a0 = s_am[j];
      *ticket = 0u;
    }
  }
}

}  // namespace

int head_splitsum_grid(int n, int sms) {
  int g = (n + kSplitSumThreads - 1) / kSplitSumThreads;
  const int cap = 2 * (sms > 0 ? sms : 1);
  return g < cap ? g : cap;
}

cudaError_t launch_head_splitsum(const float* part, int splits, int S, int n, float* logits, float* part_v,
                                 int* part_i, const int32_t* drafts, int n_valid, int32_t* argmax, int32_t* accepted,
                                 int32_t* next_a0, unsigned* ticket, int grid, cudaStream_t st) {
  if (S < 1 || S > 32 || n_valid < 0 || n_valid > S - 1 || grid < 1) return cudaErrorInvalidValue;
  return launch_pdl(head_splitsum_kernel, dim3((unsigned)grid), dim3(kSplitSumThreads), 0, st, part, splits, S, n,
                    logits, part_v, part_i, drafts, n_valid, argmax, accepted, next_a0, ticket);
}

cudaError_t launch_tree_accept(const int32_t* argmax, int S, const int32_t* tokens, const int32_t* parent,
                               int32_t* path, int32_t* accepted, int32_t* next_a0, cudaStream_t st) {
  tree_accept_kernel<<<1, 32, 0, st>>>(argmax, S, tokens, parent, path, accepted, next_a0);
  return counted(cudaGetLastError());
}

cudaError_t launch_quantize(const float* w, int n, int k, int qbits, void* codes, uint16_t* scales,
                            cudaStream_t st) {
  const long nblocks = (long)n * (k / 32);
  const int threads = 256;
  long grid = (nblocks + 7) / 8;
  if (grid > 65535L * 16) grid = 65535L * 16;
  if (qbits == 8)
    quantize_block32_kernel<8><<<(unsigned)grid, threads, 0, st>>>(
        w, nblocks, k, static_cast<uint8_t*>(codes), reinterpret_cast<__half*>(scales));
  else if (qbits == 2)
    quantize_block32_kernel<2><<<(unsigned)grid, threads, 0, st>>>(
        w, nblocks, k, static_cast<uint8_t*>(codes), reinterpret_cast<__half*>(scales));
  else
    quantize_block32_kernel<4><<<(unsigned)grid, threads, 0, st>>>(
        w, nblocks, k, static_cast<uint8_t*>(codes), reinterpret_cast<__half*>(scales));
  return counted(cudaGetLastError());
}

cudaError_t launch_greedy_accept(const int32_t* argmax, int S, const int32_t* drafts, int n_valid,
                                 int32_t* accepted, int32_t* next_a0, cudaStream_t st) {
  (void)S;
  greedy_accept_kernel<<<1, 32, 0, st>>>(argmax, drafts, n_valid, accepted, next_a0);
  return counted(cudaGetLastError());
}

}  // namespace sdv
