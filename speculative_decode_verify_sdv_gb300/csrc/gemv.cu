// Dequantised GEMV on the CUDA cores for windows of one or two rows (S <= 2),
// sm_103a: the alternative to the tensor-core path that the small windows are
// measured against ("Stream C -- Speculative decoding: feasibility verdict +
// implementation plan", section "TL;DR": a decode step and a short verify window
// both stream every weight byte once; "Riding Apple's pipelined GPU engine",
// section "Quantization on the GPU delegate": per-block-32 int8 / int4 weights).
//
// y[s][r] = sum_h x[s][h] q[r][h] s[r][h/32]: every product x * q is exact in
// fp32 (11 + 8 significant bits), sums are fp32, the block scale multiplies each
// 16- or 32-weight chunk's fp32 sum.
//
// Layout of the work: one CTA of 16 warps per SM.  A row is handled by a group
// of G warps (G = the warps whose lanes cover the row's 16-byte code chunks, up to
// CPL chunks per lane), 16 / G groups per CTA; lane L of a group owns chunks
// L, L + 32 G, ... of every row it handles, so its window values are fixed for
// the whole launch and live in fp32 registers.  A row's chunks are read as one
// contiguous coalesced stretch, and two rows per group are loaded before either
// is used.  Codes become fp32 exactly by the exponent trick: a byte b (the code
// plus a bias) permuted into the low byte of 2^23 reads as 2^23 + b, and one packed
// subtract of (2^23 + bias) leaves the code; products accumulate with packed fp32
// FMAs (fma.rn.f32x2).  A row's value is the shuffle sum over a warp, then over
// the group's warps in warp order (deterministic).  Head mode keeps each group's
// per-row (max, lowest index), merges the groups in order, and ends with the
// acquire-release ticket: the last CTA merges all CTAs' partials and runs the
// greedy accept.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cstdint>

#include "sdv_device.cuh"
#include "sdv_kernels.h"

namespace sdv {

namespace {

constexpr int kGemvRows = 2;    // rows loaded ahead of their use, per group
constexpr int kGemvWarps = 16;  // warps per CTA (one CTA per SM)

// Chunks per lane: keep the window values of a lane within 64 fp32 registers.
template <int QT, int S>
struct GemvShape {
  static constexpr int W = (QT == 8) ? 16 : 32;  // weights per 16-byte chunk
  static constexpr int CPL = 64 / (W * S);       // int8: 4 / 2, 4-bit: 2 / 1
};

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ unsigned long long pack2(uint32_t lo, uint32_t hi) {
  return ((unsigned long long)hi << 32) | lo;
}
__device__ __forceinline__ void fadd2(unsigned long long& a, unsigned long long b) {
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(a) : "l"(b));
}
__device__ __forceinline__ void ffma2(unsigned long long& acc, unsigned long long a, unsigned long long b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ float lo_f(unsigned long long v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f(unsigned long long v) { return __uint_as_float((uint32_t)(v >> 32)); }

// 2^23 + b for a byte b: the byte placed below the exponent field of 2^23.
__device__ __forceinline__ uint32_t magic_byte(uint32_t word, int j) {
  return __byte_perm(word, 0x4B000000u, 0x7540u | (uint32_t)j);
}

// The fp32 values of one chunk's codes as pairs (w[2i], w[2i+1]) in k order.
// QT 8: 16 int8 codes; 4: 32 int4 codes (two's-complement nibbles, even element
// low); 2: 32 E2M1 codes (the hardware E2M1 -> f16x2 conversion, then to fp32).
template <int QT>
__device__ __forceinline__ void chunk_pairs(const uint4 c, unsigned long long (&out)[GemvShape<QT, 1>::W / 2]) {
  const uint32_t wv[4] = {c.x, c.y, c.z, c.w};
  if (QT == 8) {
    const unsigned long long bias = pack2(0x4B000080u, 0x4B000080u);  // -(2^23 + 128) below
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t u = wv[i] ^ 0x80808080u;  // code + 128 in every byte
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        unsigned long long v = pack2(magic_byte(u, 2 * j), magic_byte(u, 2 * j + 1));
        unsigned long long nb = bias ^ 0x8000000080000000ull;
        fadd2(v, nb);
        out[2 * i + j] = v;
      }
    }
  } else if (QT == 4) {
    const unsigned long long nb = pack2(0xCB000008u, 0xCB000008u);  // -(2^23 + 8)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t u = wv[i] ^ 0x88888888u;  // code + 8 in every nibble
      const uint32_t lo = u & 0x0F0F0F0Fu, hi = (u >> 4) & 0x0F0F0F0Fu;  // even, odd elements
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        unsigned long long v = pack2(magic_byte(lo, j), magic_byte(hi, j));
        fadd2(v, nb);
        out[4 * i + j] = v;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t h[4];
      e2m1x8_to_h2x4(wv[i], h[0], h[1], h[2], h[3]);  // (k0, k1), (k2, k3), ...
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(u32_as_h2(h[j]));
        out[4 * i + j] = pack2(__float_as_uint(f.x), __float_as_uint(f.y));
      }
    }
  }
}

template <int QT, int S, int MODE>
__global__ void __launch_bounds__(kGemvWarps * 32, 1) gemv_kernel(const uint8_t* __restrict__ codes,
                                                                  const __half* __restrict__ scales,
                                                                  const GemmArgs p, int G) {
  using Sh = GemvShape<QT, S>;
  constexpr int W = Sh::W, CPL = Sh::CPL, NP = W / 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int groups = kGemvWarps / G, g = warp / G, sub = warp % G;
  const int gl = sub * 32 + lane;  // lane index within the group
  const int row_bytes = (QT == 8) ? p.K : p.K / 2;
  const int nc = row_bytes / 16;   // chunks of a row
  const int nb = p.K / 32;         // scale blocks of a row
  const int rstep = gridDim.x * groups;
  __shared__ float s_red[kGemvWarps][kGemvRows][2];
  __shared__ float s_bv[kGemvWarps][2];
  __shared__ int s_bi[kGemvWarps][2], s_am[32], s_dr[32], s_flag;

  griddep_wait();
  griddep_launch_dependents();
  // this lane's window values, fp32, as pairs in k order
  unsigned long long xr[CPL][S][NP];
#pragma unroll
  for (int m = 0; m < CPL; ++m) {
    const int c = gl + m * 32 * G;
#pragma unroll
    for (int s = 0; s < S; ++s)
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        float2 f = make_float2(0.f, 0.f);
        if (c < nc) f = __half22float2(*reinterpret_cast<const __half2*>(p.x + (size_t)s * p.K + (size_t)c * W + 2 * i));
        xr[m][s][i] = pack2(__float_as_uint(f.x), __float_as_uint(f.y));
      }
  }
  float best_v[S];  // lane 0 of the group's first warp: row s's running (max, lowest index)
  int best_i[S];
#pragma unroll
  for (int s = 0; s < S; ++s) {
    best_v[s] = -FLT_MAX;
    best_i[s] = INT_MAX;
  }
  // every group runs the same number of iterations (rows past the end are skipped
  // inside), so the block-wide barriers below are reached by all
  const int iters = (p.N + kGemvRows * rstep - 1) / (kGemvRows * rstep);
  for (int it = 0; it < iters; ++it) {
    const int base = blockIdx.x * groups + g + it * kGemvRows * rstep;
    uint4 cw[kGemvRows][CPL];
    float sc[kGemvRows][CPL];
#pragma unroll
    for (int rr = 0; rr < kGemvRows; ++rr) {
      const int r = base + rr * rstep;
#pragma unroll
      for (int m = 0; m < CPL; ++m) {
        const int c = gl + m * 32 * G;
        cw[rr][m] = make_uint4(0u, 0u, 0u, 0u);
        sc[rr][m] = 0.f;
        if (r < p.N && c < nc) {
          cw[rr][m] = ldg_stream(codes + (size_t)r * row_bytes + (size_t)c * 16);
          sc[rr][m] = __half2float(scales[(size_t)r * nb + (QT == 8 ? c / 2 : c)]);
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < kGemvRows; ++rr) {
      float part[S];
#pragma unroll
      for (int s = 0; s < S; ++s) part[s] = 0.f;
#pragma unroll
      for (int m = 0; m < CPL; ++m) {
        unsigned long long q[NP];
        chunk_pairs<QT>(cw[rr][m], q);
#pragma unroll
        for (int s = 0; s < S; ++s) {
          unsigned long long acc = 0ull;
#pragma unroll
          for (int i = 0; i < NP; ++i) ffma2(acc, q[i], xr[m][s][i]);
          part[s] = fmaf(lo_f(acc) + hi_f(acc), sc[rr][m], part[s]);
        }
      }
#pragma unroll
      for (int s = 0; s < S; ++s) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part[s] += __shfl_xor_sync(0xffffffffu, part[s], off);
        if (lane == 0) s_red[warp][rr][s] = part[s];
      }
    }
    __syncthreads();
    if (sub == 0 && lane == 0) {
#pragma unroll
      for (int rr = 0; rr < kGemvRows; ++rr) {
        const int r = base + rr * rstep;
        if (r < p.N) {
#pragma unroll
          for (int s = 0; s < S; ++s) {
            float v = s_red[warp][rr][s];
            for (int w = 1; w < G; ++w) v += s_red[warp + w][rr][s];
            if (p.y != nullptr) p.y[(size_t)s * p.N + r] = v;
            if (MODE == kModeHead) argmax_merge(best_v[s], best_i[s], v, r);
          }
        }
      }
    }
    __syncthreads();
  }
  if (MODE != kModeHead) return;
  if (sub == 0 && lane == 0)
#pragma unroll
    for (int s = 0; s < S; ++s) {
      s_bv[g][s] = best_v[s];
      s_bi[g][s] = best_i[s];
    }
  __syncthreads();
  if (threadIdx.x < S) {
    const int s = threadIdx.x;
    float v = s_bv[0][s];
    int i = s_bi[0][s];
    for (int gg = 1; gg < groups; ++gg) argmax_merge(v, i, s_bv[gg][s], s_bi[gg][s]);
    __stcg(p.part_v + (size_t)blockIdx.x * S + s, v);
    __stcg(p.part_i + (size_t)blockIdx.x * S + s, i);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // publishes this CTA's partials (cumulative over the block's stores before the
    // barrier) and, for the last CTA, acquires everyone else's
    unsigned tk;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(tk) : "l"(p.ticket) : "memory");
    s_flag = (tk == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (s_flag == 0) return;
  for (int s = warp; s < S; s += kGemvWarps) {
    float v = -FLT_MAX;
    int i = INT_MAX;
    for (int j = lane; j < (int)gridDim.x; j += 32)
      argmax_merge(v, i, __ldcg(p.part_v + (size_t)j * S + s), __ldcg(p.part_i + (size_t)j * S + s));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, off);
      const int oi = __shfl_xor_sync(0xffffffffu, i, off);
      argmax_merge(v, i, ov, oi);
    }
    if (lane == 0) {
      s_am[s] = i;
      p.argmax[s] = i;
    }
  }
  if (threadIdx.x < p.n_valid) s_dr[threadIdx.x] = p.drafts[threadIdx.x];
  __syncthreads();
  if (warp == 0) {  // accepted = the first window position whose draft misses
    const bool hit = lane < p.n_valid && s_dr[lane] == s_am[lane];
    const unsigned miss = ~__ballot_sync(0xffffffffu, hit);
    const int j = __ffs(miss) - 1;
    if (lane == 0) {
      *p.accepted = j;
      *p.next_a0 = s_am[j];
      *p.ticket = 0u;
    }
  }
}

template <int QT, int S>
cudaError_t gemv_launch_s(int mode, const GemmArgs& a, int G, int grid, cudaStream_t st) {
  const uint8_t* codes = static_cast<const uint8_t*>(a.codes);
  const __half* scales = reinterpret_cast<const __half*>(a.scales);
  if (mode == kModeHead)
    return launch_pdl(gemv_kernel<QT, S, kModeHead>, dim3((unsigned)grid), dim3(kGemvWarps * 32), 0, st, codes,
                      scales, a, G);
  return launch_pdl(gemv_kernel<QT, S, kModeY>, dim3((unsigned)grid), dim3(kGemvWarps * 32), 0, st, codes, scales,
                    a, G);
}

}  // namespace

// Warps per row (a power of two dividing 16; 0: the shape is not covered) for
// S <= 2; the grid is one CTA per SM.
int gemv_plan(int qbits, int k, int S) {
  if (S < 1 || S > 2 || k < 32 || k % 32 != 0) return 0;
  const int w = (qbits == 8) ? 16 : 32;
  const int cpl = 64 / (w * S);
  const int nc = (qbits == 8 ? k : k / 2) / 16;
  int g = 1;
  while (g < kGemvWarps && g * 32 * cpl < nc) g *= 2;
  return g * 32 * cpl >= nc ? g : 0;
}

cudaError_t launch_gemv(int qbits, int mode, const GemmArgs& a, int G, int grid, cudaStream_t st) {
  if (a.S == 1) {
    if (qbits == 8) return gemv_launch_s<8, 1>(mode, a, G, grid, st);
    if (qbits == 4) return gemv_launch_s<4, 1>(mode, a, G, grid, st);
    return gemv_launch_s<2, 1>(mode, a, G, grid, st);
  }
  if (qbits == 8) return gemv_launch_s<8, 2>(mode, a, G, grid, st);
  if (qbits == 4) return gemv_launch_s<4, 2>(mode, a, G, grid, st);
  return gemv_launch_s<2, 2>(mode, a, G, grid, st);
}

}  // namespace sdv
