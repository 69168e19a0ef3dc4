// Weight-streaming dequantised skinny GEMM over a verify window of S rows.
//
// The verify forward is bound by reading every weight byte once for all S
// window rows ("Stream C -- Speculative decoding: feasibility verdict +
// implementation plan", section "TL;DR": a K-token verify forward costs about
// one decode step; "Flagship dramatic-speedup plan", section "Baseline byte
// model": the lm_head is the single biggest matvec).  Weights are per-block-32
// absmax int8 / int4 ("Riding Apple's pipelined GPU engine", section
// "Quantization on the GPU delegate").
//
// Design (sm_103a):
//  * persistent grid, one CTA of 4 warps per SM; each warp owns a contiguous
//    range of 16-row tiles of W and streams them through its own ring of TMA
//    stages (cp.async.bulk.tensor, 128-byte swizzle, completion on mbarriers,
//    bounded waits), so every warp keeps several stages of HBM reads in flight;
//  * a stage is MT tiles x 256 reduction elements (8 scale blocks) of codes plus
//    their fp16 scales;
//  * codes are converted to exact fp16 integers in registers and fed to the
//    m16n8k16 tensor-core MMA as the A operand (16 weight rows); the window rows
//    are the B operand (n8 tiles), staged once per CTA in shared memory with the
//    reduction index permuted to match the register layout of the codes;
//  * each 32-block is accumulated separately and folded into the fp32
//    accumulator with its fp32 scale, so the result is sum_b s_b * (x . q_b)
//    with exact products and fp32 accumulation;
//  * epilogues: fp32 Y (sdv_qlinear) or, for the verify head, a per-row
//    (max, lowest index) reduction whose CTA partials are reduced by the last
//    CTA to finish (atomic ticket) together with the greedy accept.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cstdint>

#include "sdv_device.cuh"
#include "sdv_kernels.h"

namespace sdv {

namespace {

constexpr int kWarps = 4;
constexpr int kStageK = 256;  // reduction elements per stage (8 scale blocks)


__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

template <int QB>
struct Layout {
  static constexpr int kBoxes = (QB == 8) ? 2 : 1;  // 128-byte code boxes per stage row
};

// Dynamic shared memory layout (offsets from a 1024-aligned base).
struct SmemPlan {
  int depth;
  int code_slot, sc_slot;
  int codes_off, sc_off, x_off, bar_off, best_off, am_off, flag_off, total;
  int xpitch;
};

__host__ __device__ inline int round_up(int a, int b) { return (a + b - 1) / b * b; }

__host__ __device__ inline SmemPlan make_plan(int qb, int mt, int S, int k_len, int depth) {
  SmemPlan p;
  p.depth = depth;
  const int boxes = (qb == 8) ? 2 : 1;
  p.code_slot = mt * 16 * 128 * boxes;
  p.sc_slot = mt * 16 * 16;
  p.codes_off = 0;
  p.sc_off = p.codes_off + kWarps * depth * p.code_slot;
  p.x_off = round_up(p.sc_off + kWarps * depth * p.sc_slot, 128);
  p.xpitch = round_up(k_len, 64) * 2 + 64;  // == 64 (mod 128): conflict-free 16-byte B loads
  p.bar_off = round_up(p.x_off + S * p.xpitch, 16);
  p.best_off = p.bar_off + kWarps * depth * 8;
  p.am_off = p.best_off + kWarps * 32 * 8;
  p.flag_off = p.am_off + 32 * 4;
  p.total = p.flag_off + 16;
  return p;
}

template <int QB, int NT, int MT, int MODE>
__global__ void __launch_bounds__(kWarps * 32, 1)
    dq_gemm_kernel(const __grid_constant__ CUtensorMap tm_codes,
                   const __grid_constant__ CUtensorMap tm_scales, const GemmArgs p) {
  using L = Layout<QB>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  // reduction range of this CTA (split-K over gridDim.y)
  const int k_begin = blockIdx.y * p.k_chunk;
  const int k_len = min(p.k_chunk, p.K - k_begin);
  const SmemPlan sp = make_plan(QB, MT, p.S, p.k_chunk, p.depth);
  const int depth = sp.depth;

  const uint32_t codes_ring = base + sp.codes_off + warp * depth * sp.code_slot;
  const uint32_t sc_ring = base + sp.sc_off + warp * depth * sp.sc_slot;
  const uint32_t xs = base + sp.x_off;
  const uint8_t* const xsp = sbase + sp.x_off;
  const uint32_t bars = base + sp.bar_off + warp * depth * 8;
  float* const best_v = reinterpret_cast<float*>(sbase + sp.best_off);
  int* const best_i = reinterpret_cast<int*>(sbase + sp.best_off + kWarps * 32 * 4);
  int* const s_am = reinterpret_cast<int*>(sbase + sp.am_off);
  int* const s_flag = reinterpret_cast<int*>(sbase + sp.flag_off);

  // ---- this warp's tiles -------------------------------------------------------
  const long total_warps = (long)gridDim.x * kWarps;
  const long gw = (long)blockIdx.x * kWarps + warp;
  const int tile_lo = (int)(gw * p.m16_tiles / total_warps);
  const int tile_hi = (int)((gw + 1) * p.m16_tiles / total_warps);
  const int ntiles = tile_hi - tile_lo;
  const int nunits = (ntiles + MT - 1) / MT;
  const int kst = (k_len + kStageK - 1) / kStageK;
  const int nstages = nunits * kst;
  const int kbyte0 = (QB == 8) ? k_begin : k_begin / 2;
  const int kbyte_end = (QB == 8) ? k_begin + k_len : (k_begin + k_len) / 2;

  if (lane == 0) {
    for (int d = 0; d < depth; ++d) mbar_init(bars + 8 * d, 1);
    fence_barrier_init();
    if (warp == 0) {
      tma_prefetch_desc(&tm_codes);
      if (p.scales_tma) tma_prefetch_desc(&tm_scales);
    }
  }
  __syncwarp();

  const uint64_t policy = l2_policy_evict_first();

  auto issue = [&](int i) {
    const int u = i / kst, ks = i - (i / kst) * kst;
    const int slot = i % depth;
    const int mt_cnt = min(MT, ntiles - u * MT);
    const int row0 = (tile_lo + u * MT) * 16;
    const uint32_t bar = bars + 8 * slot;
    const uint32_t cdst = codes_ring + slot * sp.code_slot;
    const int xb = kbyte0 + ks * 128 * L::kBoxes;
    uint32_t bytes = 0;
    for (int mt = 0; mt < mt_cnt; ++mt)
      for (int bx = 0; bx < L::kBoxes; ++bx)
        if (xb + 128 * bx < kbyte_end) bytes += 16 * 128;
    if (p.scales_tma) bytes += MT * 16 * 16;
    mbar_arrive_expect_tx(bar, bytes);
    for (int mt = 0; mt < mt_cnt; ++mt)
      for (int bx = 0; bx < L::kBoxes; ++bx)
        if (xb + 128 * bx < kbyte_end)
          tma_load_2d(cdst + (mt * L::kBoxes + bx) * 2048, &tm_codes, xb + 128 * bx, row0 + mt * 16,
                      bar, policy);
    if (p.scales_tma)
      tma_load_2d(sc_ring + slot * sp.sc_slot, &tm_scales, k_begin / 32 + ks * 8, row0, bar,
                  policy);
  };

  // Start streaming before staging the window rows.
  if (lane == 0) {
    const int pro = min(depth, nstages);
    for (int i = 0; i < pro; ++i) issue(i);
  }

  // ---- stage X (window rows) with the reduction index permuted ---------------
  {
    const int v8 = k_len / 8;
    for (int v = threadIdx.x; v < p.S * v8; v += blockDim.x) {
      const int s = v / v8, k8 = (v - s * v8) * 8;
      const uint4 in = *reinterpret_cast<const uint4*>(p.x + (size_t)s * p.K + k_begin + k8);
      uint4 o;
      if (QB == 8) {  // per 4 elements: (k0, k2, k1, k3)
        o.x = __byte_perm(in.x, in.y, 0x5410);
        o.y = __byte_perm(in.x, in.y, 0x7632);
        o.z = __byte_perm(in.z, in.w, 0x5410);
        o.w = __byte_perm(in.z, in.w, 0x7632);
      } else {  // per 8 elements: (k0, k4, k1, k5, k2, k6, k3, k7)
        o.x = __byte_perm(in.x, in.z, 0x5410);
        o.y = __byte_perm(in.x, in.z, 0x7632);
        o.z = __byte_perm(in.y, in.w, 0x5410);
        o.w = __byte_perm(in.y, in.w, 0x7632);
      }
      sts128(xs + s * sp.xpitch + k8 * 2, o);
    }
  }
  __syncthreads();

  const int nblk_total = k_len / 32;
  const int ks_per_row = p.K / 32;  // scale entries per weight row
  bool dead = false;

  // running per-column argmax (head mode); lanes with equal c hold equal values
  float rb_v[NT][2];
  int rb_i[NT][2];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      rb_v[t][cc] = -FLT_MAX;
      rb_i[t][cc] = INT_MAX;
    }

  int i_stage = 0;
  for (int u = 0; u < nunits && !dead; ++u) {
    const int mt_cnt = min(MT, ntiles - u * MT);
    const int row0 = (tile_lo + u * MT) * 16;
    float acc[MT][NT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[mt][t][r] = 0.f;

    for (int ks = 0; ks < kst; ++ks, ++i_stage) {
      const int slot = i_stage % depth;
      if (!mbar_wait_bounded(bars + 8 * slot, (i_stage / depth) & 1)) {
        dead = true;
        break;
      }
      const uint8_t* const cbase = sbase + (codes_ring - base) + slot * sp.code_slot;
      const uint8_t* const scbase = sbase + (sc_ring - base) + slot * sp.sc_slot;
      const int nblk = min(8, nblk_total - ks * 8);

      // operands of one 32-block, loaded one block ahead of their use
      constexpr int AW = (QB == 8) ? 2 : 1;  // 32-bit code words per row per block
      struct Ops {
        uint32_t a[MT][2][AW];
        float s[MT][2];
        uint4 b[NT];
      };
      auto load_ops = [&](int blk, Ops& o) {
        const int kb = ks * 8 + blk;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int n = 8 * t + g;
          o.b[t] = (n < p.S) ? *reinterpret_cast<const uint4*>(xsp + n * sp.xpitch + (kb * 32 + 8 * c) * 2)
                             : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int r = g + 8 * hr;
            if (QB == 8) {
              const int bx = blk >> 2, bb = blk & 3;
              const int chunk = (2 * bb + (c >> 1)) ^ g;
              const uint2 w = *reinterpret_cast<const uint2*>(cbase + (mt * 2 + bx) * 2048 + r * 128 +
                                                              chunk * 16 + 8 * (c & 1));
              o.a[mt][hr][0] = w.x;
              o.a[mt][hr][AW - 1] = w.y;
            } else {
              o.a[mt][hr][0] = *reinterpret_cast<const uint32_t*>(cbase + mt * 2048 + r * 128 +
                                                                  ((blk ^ g) << 4) + 4 * c);
            }
            if (p.scales_tma) {
              o.s[mt][hr] = __half2float(*reinterpret_cast<const __half*>(scbase + (mt * 16 + r) * 16 + blk * 2));
            } else {
              const int row = row0 + mt * 16 + r;
              o.s[mt][hr] = row < p.N ? __half2float(__ushort_as_half(__ldg(
                                            p.scales + (size_t)row * ks_per_row + k_begin / 32 + kb)))
                                      : 0.f;
            }
          }
        }
      };
      auto compute = [&](const Ops& o) {
        uint32_t a0[MT][4], a1[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          if (QB == 8) {
            i8x4_to_h2x2(o.a[mt][0][0], a0[mt][0], a0[mt][2]);
            i8x4_to_h2x2(o.a[mt][1][0], a0[mt][1], a0[mt][3]);
            i8x4_to_h2x2(o.a[mt][0][AW - 1], a1[mt][0], a1[mt][2]);
            i8x4_to_h2x2(o.a[mt][1][AW - 1], a1[mt][1], a1[mt][3]);
          } else {
            i4x8_to_h2x4(o.a[mt][0][0], a0[mt][0], a0[mt][2], a1[mt][0], a1[mt][2]);
            i4x8_to_h2x4(o.a[mt][1][0], a0[mt][1], a0[mt][3], a1[mt][1], a1[mt][3]);
          }
        }
        float tmp[MT][NT][4];
        const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int t = 0; t < NT; ++t)
            mma_16816(tmp[mt][t], a0[mt][0], a0[mt][1], a0[mt][2], a0[mt][3], o.b[t].x, o.b[t].y, zero4);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int t = 0; t < NT; ++t)
            mma_16816(tmp[mt][t], a1[mt][0], a1[mt][1], a1[mt][2], a1[mt][3], o.b[t].z, o.b[t].w, tmp[mt][t]);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            acc[mt][t][0] = fmaf(o.s[mt][0], tmp[mt][t][0], acc[mt][t][0]);
            acc[mt][t][1] = fmaf(o.s[mt][0], tmp[mt][t][1], acc[mt][t][1]);
            acc[mt][t][2] = fmaf(o.s[mt][1], tmp[mt][t][2], acc[mt][t][2]);
            acc[mt][t][3] = fmaf(o.s[mt][1], tmp[mt][t][3], acc[mt][t][3]);
          }
      };

      Ops cur, nxt;
      load_ops(0, cur);
#pragma unroll
      for (int blk = 0; blk < 8; ++blk) {
        if (blk >= nblk) break;
        if (blk + 1 < nblk) load_ops(blk + 1, nxt);
        compute(cur);
        cur = nxt;
      }
      __syncwarp();
      if (lane == 0 && i_stage + depth < nstages) issue(i_stage + depth);
    }
    if (dead) break;

    // ---- epilogue of this unit -------------------------------------------------
    float* const yout = p.y == nullptr ? nullptr : p.y + (size_t)blockIdx.y * p.S * p.N;
    if (yout != nullptr) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        if (mt >= mt_cnt) break;
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int row = row0 + mt * 16 + g + 8 * (r >> 1);
            const int col = 8 * t + 2 * c + (r & 1);
            if (row < p.N && col < p.S) yout[(size_t)col * p.N + row] = acc[mt][t][r];
          }
      }
    }
    if (MODE == kModeHead) {
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float bv = -FLT_MAX;
          int bi = INT_MAX;
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            if (mt >= mt_cnt) break;
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
              const int row = row0 + mt * 16 + g + 8 * hr;
              if (row < p.N) argmax_merge(bv, bi, acc[mt][t][2 * hr + cc], row);
            }
          }
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            argmax_merge(bv, bi, ov, oi);
          }
          argmax_merge(rb_v[t][cc], rb_i[t][cc], bv, bi);
        }
    }
  }

  if (dead) {
    if (lane == 0) atomicOr(p.status, kDevErrTimeout);
    // let copies still in flight land (bounded) before the CTA exits
    for (int j = i_stage + 1; j < min(nstages, i_stage + depth); ++j)
      mbar_wait_bounded(bars + 8 * (j % depth), (j / depth) & 1, 100000000ull);
  }

  if (MODE != kModeHead) return;

  // ---- CTA partials, then the last CTA reduces and accepts -----------------------
  if (g == 0) {
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int col = 8 * t + 2 * c + cc;
        if (col < p.S) {
          best_v[warp * 32 + col] = rb_v[t][cc];
          best_i[warp * 32 + col] = rb_i[t][cc];
        }
      }
  }
  __syncthreads();
  if (threadIdx.x < p.S) {
    const int col = threadIdx.x;
    float bv = best_v[col];
    int bi = best_i[col];
    for (int w = 1; w < kWarps; ++w) argmax_merge(bv, bi, best_v[w * 32 + col], best_i[w * 32 + col]);
    __stcg(p.part_v + (size_t)blockIdx.x * p.S + col, bv);
    __stcg(p.part_i + (size_t)blockIdx.x * p.S + col, bi);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned tk = atomicAdd(p.ticket, 1u);
    *s_flag = (tk == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (*s_flag == 0) return;
  __threadfence();
  for (int col = warp; col < p.S; col += kWarps) {
    float bv = -FLT_MAX;
    int bi = INT_MAX;
    for (int j = lane; j < (int)gridDim.x; j += 32)
      argmax_merge(bv, bi, __ldcg(p.part_v + (size_t)j * p.S + col), __ldcg(p.part_i + (size_t)j * p.S + col));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      argmax_merge(bv, bi, ov, oi);
    }
    if (lane == 0) {
      s_am[col] = bi;
      p.argmax[col] = bi;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int j = 0;
    while (j < p.n_valid && p.drafts[j] == s_am[j]) ++j;
    *p.accepted = j;
    *p.next_a0 = s_am[j];
    *p.ticket = 0u;  // every CTA has taken its ticket: leave the counter at zero
  }
}

template <int QB, int NT, int MT, int MODE>
cudaError_t launch_t(const CUtensorMap& tc, const CUtensorMap& tsc, const GemmArgs& a, int grid,
                     int smem, cudaStream_t st) {
  auto k = dq_gemm_kernel<QB, NT, MT, MODE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<dim3(grid, a.splits), kWarps * 32, smem, st>>>(tc, tsc, a);
  return counted(cudaGetLastError());
}

template <int QB, int MT, int MODE>
cudaError_t launch_nt(int nt, const CUtensorMap& tc, const CUtensorMap& tsc, const GemmArgs& a,
                      int grid, int smem, cudaStream_t st) {
  switch (nt) {
    case 1: return launch_t<QB, 1, MT, MODE>(tc, tsc, a, grid, smem, st);
    case 2: return launch_t<QB, 2, MT, MODE>(tc, tsc, a, grid, smem, st);
    case 3: return launch_t<QB, 3, MT, MODE>(tc, tsc, a, grid, smem, st);
    case 4: return launch_t<QB, 4, MT, MODE>(tc, tsc, a, grid, smem, st);
  }
  return cudaErrorInvalidValue;
}

// y[s][n] = sum over splits of part[split][s][n], in split order (deterministic).
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int splits, long count,
                                     float* __restrict__ y) {
  griddep_wait();
  griddep_launch_dependents();
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += (long)gridDim.x * blockDim.x) {
    // loads in batches of 16 (independent, one L2 round trip per batch), sums
    // in split order
    float v = 0.f;
    for (int sp0 = 0; sp0 < splits; sp0 += 16) {
      float b[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) b[j] = sp0 + j < splits ? __ldcg(part + (long)(sp0 + j) * count + i) : 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (sp0 + j >= splits) break;
        v = (sp0 + j == 0) ? b[j] : v + b[j];
      }
    }
    y[i] = v;
  }
}

}  // namespace

cudaError_t launch_splitk_reduce(const float* part, int splits, long count, float* y, cudaStream_t st) {
  long grid = (count + 255) / 256;
  if (grid > 4096) grid = 4096;
  return launch_pdl(splitk_reduce_kernel, dim3((unsigned)grid), dim3(256), 0, st, part, splits, count, y);
}

int gemm_tile_mt(int qbits) { return qbits == 8 ? 2 : 4; }

int gemm_smem_bytes(int qbits, int S, int k_len, int depth) {
  return make_plan(qbits, gemm_tile_mt(qbits), S, k_len, depth).total + 1024;
}

int gemm_warps_per_cta() { return kWarps; }

cudaError_t launch_dq_gemm(int qbits, int mode, const CUtensorMap& tm_codes,
                           const CUtensorMap& tm_scales, const GemmArgs& a, int grid, int smem,
                           cudaStream_t st) {
  const int nt = (a.S + 7) / 8;
  if (qbits == 8) {
    return mode == kModeHead ? launch_nt<8, 2, kModeHead>(nt, tm_codes, tm_scales, a, grid, smem, st)
                             : launch_nt<8, 2, kModeY>(nt, tm_codes, tm_scales, a, grid, smem, st);
  }
  return mode == kModeHead ? launch_nt<4, 4, kModeHead>(nt, tm_codes, tm_scales, a, grid, smem, st)
                           : launch_nt<4, 4, kModeY>(nt, tm_codes, tm_scales, a, grid, smem, st);
}

}  // namespace sdv
