// Weight-streaming dequantised skinny GEMM on the 5th-generation tensor cores
// (tcgen05, tensor memory), sm_103a.
//
// Same operation and epilogues as dq_gemm.cu (the verify forward reads every
// weight byte once for all S window rows: "Stream C -- Speculative decoding:
// feasibility verdict + implementation plan", section "TL;DR"; per-block-32
// int8/int4 weights: "Riding Apple's pipelined GPU engine", section
// "Quantization on the GPU delegate").
//
// One CTA per SM, warp roles:
//   warp 0        TMA producer: 128-row x 256-element stages of codes (128-byte
//                 swizzled boxes) and their fp16 scales into a shared-memory ring;
//   warp 1        allocates tensor memory and issues every tcgen05.mma (one
//                 elected thread per stage), committing completion to mbarriers;
//   warps 2-5     tile epilogue, one per tensor-memory lane quarter;
//   warps 6..     4*G converter warps: group g (warps 6+4g .. 9+4g) converts the
//                 whole stages g, g+G, g+2G, ...; warp w serves tensor-memory lane
//                 quarter w % 4 (rows 32q..32q+31 of the tile) and each thread owns
//                 one weight row.  Codes become fp16 n*s, rounded once (one-FMA or
//                 two-step form, the same bits; int4 codes at bits 0-3 of a half
//                 as n*s/16), stored into tensor memory as the A operand (M = 128
//                 rows, K = 16 per MMA).  The window rows are the B operand (N = 16
//                 or 32), staged once in shared memory in the K-major core-matrix
//                 layout, the reduction index permuted like the converted codes.
//   The MMAs of a 128-row tile accumulate in fp32 tensor memory (double-buffered
//   across tiles); the epilogue warps load the result (tcgen05.ld) while the next
//   tile streams and write Y, or reduce the verify head's per-row
//   (max, lowest index) through shared memory.  The MMA warp runs a
//   warp-uniform loop and one elected lane issues each stage's MMAs.
// Tensor memory: columns 0-383 hold A (3 stage buffers x 8 blocks x 16 columns),
// columns 384.. two tile buffers of kAcc accumulators (N columns each): a tile's
// MMAs rotate over them so that consecutive MMAs do not depend on each other,
// and the epilogue adds them (int4: the even ones 16-fold).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cstdint>
#include <type_traits>

#include "moe_route.cuh"
#include "sdv_device.cuh"
#include "sdv_kernels.h"

namespace sdv {

namespace {

constexpr int kTileRows = 128;
constexpr uint32_t kTmemCols = 512;
constexpr int kABufs = 3;        // A operand stage buffers in tensor memory
constexpr int kMinDepth = 4;     // ring stages (see tc_plan_valid)
constexpr int kACols = kABufs * 128;
constexpr uint64_t kDrainLimitNs = 100000000ull;  // 0.1 s: in-flight work at teardown

// Converter groups: group g takes the stages i with i % G == g.  An int4 stage
// carries twice the weights per byte of an int8 stage, so it gets a third group.
template <int QB>
struct TcRoles {
  static constexpr int G = (QB == 4) ? 3 : 2;
  static constexpr int kConvWarps = 4 * G;   // one warp per tensor-memory lane quarter per group
  static constexpr int kConv0 = 6;           // first converter warp (0 TMA, 1 MMA, 2-5 epilogue)
  static constexpr int kWarps = kConv0 + kConvWarps;
  static constexpr int kThreads = 32 * kWarps;
  // A group converting stage i first waits (by parity) for the release of A
  // buffer i % kABufs by the MMAs of stage i - kABufs; the wait is unambiguous
  // only if the buffer's previous release (stage i - 2 kABufs) has completed.
  // The group's own previous stage, i - G, waited for stage i - G - kABufs, and
  // the MMAs complete in stage order, so that holds while G <= kABufs (with
  // more groups a group can pass a stale phase and overwrite operands in use).
  static_assert(G <= kABufs, "converter groups must not outnumber the A buffers");
};

struct TcPlan {
  int depth, nmma, xrows, kpad, code_stage, sc_stage;
  int x_off, ring_off, sc_off, red_off, bar_off, best_off, misc_off, route_off, total;
};

// The in-prologue MoE routing's region: hit count (16 bytes), hit list
// [kRouteMaxE], picks [kRouteMaxS][kRouteMaxTopK] and their weights.
constexpr int kRouteBytes = 16 + 4 * kRouteMaxE + 2 * 4 * kRouteMaxS * kRouteMaxTopK;

__host__ __device__ inline int rup(int a, int b) { return (a + b - 1) / b * b; }

__host__ __device__ inline TcPlan tc_plan(int qb, int S, int kc, int depth, bool route = false) {
  TcPlan p;
  p.depth = depth;
  p.nmma = S <= 16 ? 16 : 32;
  p.xrows = rup(S, 8);
  // window rows are staged zero-padded to whole 256-element stages, so every
  // stage runs all 16 MMAs (missing code blocks get a zero scale)
  p.kpad = rup(kc, 256);
  p.code_stage = kTileRows * 128 * (qb == 8 ? 2 : 1);
  p.sc_stage = kTileRows * 16;
  // The window rows come first: when N exceeds the staged rows, the MMA's reads
  // of the missing 8-row groups land in the ring and only feed discarded columns.
  p.x_off = 0;
  p.ring_off = rup(p.xrows * p.kpad * 2, 1024);
  p.sc_off = p.ring_off + depth * p.code_stage;
  p.red_off = p.sc_off + depth * p.sc_stage;           // epilogue: [4 warps][S][33] floats
  p.bar_off = rup(p.red_off + 4 * S * 33 * 4, 16);
  // ring full/empty, A buffers afull/afree, tiles tfull/tfree, row slices xready, drain
  p.best_off = p.bar_off + (2 * depth + 2 * kABufs + 4 + p.kpad / 256 + 1) * 8;
  p.misc_off = p.best_off + 4 * 32 * 8;
  p.route_off = rup(p.misc_off + 16 + 32 * 4 + 32 * 4, 16);  // after flags, argmax [32], drafts [32]
  p.total = p.route_off + (route ? kRouteBytes : 0);
  return p;
}

// Tail of the sampling verify, run by every thread of the CTA after the
// teardown barrier.  `stb` holds the four epilogue warps' column states
// ([field][quarter][S] floats: top-1 z and entry over the entries other than
// the row's draft, the draft's z, softmax max and sum, the draft's L/T).  Each
// CTA publishes its merged partial per window row; the last CTA (acquire-release
// ticket, as for the verify head) merges all of them and runs the accept: draft
// d_i is kept iff u_i < p_i(d_i) = exp(L_i(d_i)/T - M_i) / sum_v exp(L_i(v)/T - M_i);
// at the first rejection the token is the largest L/T + g of row i other than d_i
// (the residual draw), and if every draft is kept it is row n_valid's draw.  A
// row's draw from its full distribution is d_i where d_i's z wins the argmax
// order against the residual draw, else the residual draw.
__device__ __noinline__ void sample_tail(const GemmArgs& p, uint8_t* stb, const int* s_drafts, int* s_flag,
                                         int warp, int lane, int nwarps) {
  float* const st = reinterpret_cast<float*>(stb);
  const int S = p.S, f = 4 * S;
  auto take_number = [](float& into, float v) {  // the one CTA / quarter holding the draft reports it
    if (v == v) into = v;
  };
  if ((int)threadIdx.x < S) {
    const int c = threadIdx.x;
    float zx = st[c], zd = st[2 * f + c], m = st[3 * f + c], s = st[4 * f + c], ld = st[5 * f + c];
    int vx = __float_as_int(st[f + c]);
    for (int q = 1; q < 4; ++q) {
      const int o = q * S + c;
      top1_add(zx, vx, st[o], __float_as_int(st[f + o]));
      take_number(zd, st[2 * f + o]);
      softmax_merge(m, s, st[3 * f + o], st[4 * f + o]);
      take_number(ld, st[5 * f + o]);
    }
    float* const out = p.part_s + ((size_t)blockIdx.x * S + c) * 8;
    __stcg(out + 0, zx);
    __stcg(out + 1, __int_as_float(vx));
    __stcg(out + 2, zd);
    __stcg(out + 3, m);
    __stcg(out + 4, s);
    __stcg(out + 5, ld);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned tk;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(tk) : "l"(p.ticket) : "memory");
    *s_flag = (tk == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (*s_flag == 0) return;
  // merged rows: [S][8] = residual draw, full draw, m, s, ld
  for (int col = warp; col < S; col += nwarps) {
    float zx = -INFINITY, zd = __int_as_float(0x7fc00000), m = -INFINITY, s = 0.f, ld = __int_as_float(0x7fc00000);
    int vx = INT_MAX;
    for (int j = lane; j < (int)gridDim.x; j += 32) {
      const float* const in = p.part_s + ((size_t)j * S + col) * 8;
      top1_add(zx, vx, __ldcg(in + 0), __float_as_int(__ldcg(in + 1)));
      take_number(zd, __ldcg(in + 2));
      softmax_merge(m, s, __ldcg(in + 3), __ldcg(in + 4));
      take_number(ld, __ldcg(in + 5));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float oz = __shfl_xor_sync(0xffffffffu, zx, off), ozd = __shfl_xor_sync(0xffffffffu, zd, off);
      const int ov = __shfl_xor_sync(0xffffffffu, vx, off);
      const float om = __shfl_xor_sync(0xffffffffu, m, off), os = __shfl_xor_sync(0xffffffffu, s, off);
      const float old = __shfl_xor_sync(0xffffffffu, ld, off);
      top1_add(zx, vx, oz, ov);
      take_number(zd, ozd);
      softmax_merge(m, s, om, os);
      take_number(ld, old);
    }
    if (lane == 0) {
      // zd is a number only where the row has a draft inside the vocabulary
      const int d = (col < p.n_valid) ? s_drafts[col] : -1;
      const int full = (zd == zd && (zd > zx || (zd == zx && d < vx))) ? d : vx;
      float* const r = st + col * 8;
      r[0] = __int_as_float(vx);
      r[1] = __int_as_float(full);
      r[2] = m;
      r[3] = s;
      r[4] = ld;
      p.argmax[col] = full;  // the row's draw from its full distribution
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int j = p.n_valid;
    int token = __float_as_int(st[p.n_valid * 8 + 1]);
    for (int i = 0; i < p.n_valid; ++i) {
      const float* const r = st + i * 8;
      const float pr = expf(r[4] - r[2]) / r[3];
      const float u = counter_uniform(p.rng_key, 32ull * (unsigned)p.N + (unsigned)i);
      if (!(u < pr)) {
        j = i;
        token = __float_as_int(r[0]);  // the residual draw: the best entry other than d_i
        break;
      }
    }
    *p.accepted = j;
    *p.next_a0 = token;
    *p.ticket = 0u;
  }
}

// The MoE window's routing in the prologue of its gate/up launch (GemmArgs
// route_*): the rows over the CTA's warps (route_row), then a flag per hit
// expert and one warp's prefix count over the flags give the hit list, experts
// ascending -- the grouping of moe_route_kernel without its per-expert row
// lists, which no GEMM reads.  `rt` is the plan's routing region, `scratch`
// kRouteMaxE ints that are free until the weight stream starts.  CTA 0
// publishes the picks and the hit list for the down projection.
__device__ __forceinline__ void route_prologue(const GemmArgs& p, int* rt, int* scratch, int warp, int lane,
                                               int nwarps) {
  int* const s_hit = rt + 4;
  int* const s_ids = s_hit + kRouteMaxE;
  float* const s_w = reinterpret_cast<float*>(s_ids + kRouteMaxS * kRouteMaxTopK);
  const int E = p.route_E, K = p.route_top_k;
  for (int e = threadIdx.x; e < kRouteMaxE; e += blockDim.x) scratch[e] = 0;
  for (int s = warp; s < p.S; s += nwarps)
    route_row<kRouteMaxE / 32>(p.route_logits + (size_t)s * E, E, K, lane, s_ids + s * kRouteMaxTopK,
                               s_w + s * kRouteMaxTopK);
  __syncthreads();
  for (int v = threadIdx.x; v < p.S * K; v += blockDim.x) scratch[s_ids[(v / K) * kRouteMaxTopK + v % K]] = 1;
  __syncthreads();
  if (warp == 0) {
    constexpr int kPer = kRouteMaxE / 32;  // experts lane * kPer .. of each lane
    int f[kPer], c = 0;
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      f[m] = scratch[lane * kPer + m];
      c += f[m];
    }
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    int pos = incl - c;
#pragma unroll
    for (int m = 0; m < kPer; ++m)
      if (f[m]) s_hit[pos++] = lane * kPer + m;
    if (lane == 31) rt[0] = incl;
  }
  __syncthreads();
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    for (int v = threadIdx.x; v < p.S * K; v += blockDim.x) {
      const int o = (v / K) * kRouteMaxTopK + v % K;
      p.route_ids[v] = s_ids[o];
      p.route_w[v] = s_w[o];
    }
    for (int j = threadIdx.x; j < rt[0]; j += blockDim.x) p.route_hit[j] = s_hit[j];
    if (threadIdx.x == 0) *p.route_n_hit = rt[0];
  }
}

// QT: the weight type -- 8 int8, 4 int4, 2 FP4 (E2M1); QB below is its code
// width in bits (8 or 4), which sets the byte layout of a stage.
template <int QT, int MODE, int NM>
__global__ void __launch_bounds__(TcRoles<(QT == 8 ? 8 : 4)>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tm_codes,
                   const __grid_constant__ CUtensorMap tm_scales,
                   const __grid_constant__ CUtensorMap tm_codes2,
                   const __grid_constant__ CUtensorMap tm_scales2, const GemmArgs p) {
  constexpr int QB = (QT == 8) ? 8 : 4;
  using R = TcRoles<QB>;
  // independent fp32 accumulators per tile (MMA m of a stage -> m % kAcc), two
  // tile buffers, in the tensor-memory columns behind the A buffers
  constexpr int kAcc = (512 - kACols) / (2 * NM);
  static_assert(kAcc >= 2 && (kAcc & (kAcc - 1)) == 0, "accumulator count");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* const sb = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Launched as a programmatic dependent of the previous kernel in the stream:
  // nothing in global memory is read or written before that grid has completed.
  // Only the MoE mappings need global data (the hit count) up front; other
  // launches set up barriers and tensor memory first, overlapping its tail.
  const bool routed = (MODE == kModeY) && (p.route_logits != nullptr);  // Y mode only
  const bool listed = routed || (p.n_hit != nullptr);  // hit-list mappings (MoE)
  const bool dep_early = listed;
  if (dep_early) griddep_wait();
  const TcPlan pl = tc_plan(QB, p.S, p.k_chunk, p.depth, routed);
  int* const s_route = reinterpret_cast<int*>(sb + pl.route_off);  // hit count, hit list, picks, weights
  if (routed) route_prologue(p, s_route, reinterpret_cast<int*>(sb + pl.ring_off), threadIdx.x >> 5,
                             threadIdx.x & 31, blockDim.x >> 5);
  const int* const s_hit = s_route + 4;
  const int* const s_rids = s_hit + kRouteMaxE;  // [kRouteMaxS][kRouteMaxTopK]
  const float* const s_rw = reinterpret_cast<const float*>(s_rids + kRouteMaxS * kRouteMaxTopK);
  auto hit_of = [&](int j) -> int { return routed ? s_hit[j] : __ldg(p.hit + j); };
  // Row and reduction mappings (all uniform over the CTA):
  //  * plain: tile t covers weight rows 128t.., the reduction [k_begin, k_begin + k_len);
  //  * dual: tiles [0, T) read the first matrix, [T, 2T) the second (T tiles each);
  //  * hit-list tiles (n_hit, no seg_k): the T tiles of a matrix run over the hit
  //    experts' row blocks, rows_per_expert rows each;
  //  * expert segments (n_hit and seg_k): the reduction runs over the hit experts'
  //    seg_k columns, segment j reading expert hit[j]'s rows.
  const bool segs = listed && p.seg_k > 0;
  const bool hit_tiles = listed && p.seg_k == 0;
  const int n_hit = routed ? s_route[0] : (p.n_hit != nullptr) ? *p.n_hit : 0;
  int k_begin, k_len;
  if (segs) {
    const int s_lo = (int)((long)blockIdx.y * n_hit / gridDim.y);
    const int s_hi = (int)((long)(blockIdx.y + 1) * n_hit / gridDim.y);
    k_begin = s_lo * p.seg_k;
    k_len = (s_hi - s_lo) * p.seg_k;
  } else {
    k_begin = blockIdx.y * p.k_chunk;
    k_len = min(p.k_chunk, p.K - k_begin);
  }
  const int n_one = hit_tiles ? n_hit * p.rows_per_expert : p.N;  // rows of one matrix
  const int ldx = p.ldx > 0 ? p.ldx : p.K;
  const int t_one = (n_one + kTileRows - 1) / kTileRows;          // tiles of one matrix
  const int ldy = p.ldy > 0 ? p.ldy : p.N;
  // tile t -> (matrix, tile within the matrix, first weight row)
  auto tile_split = [&](int t, int& mat, int& lt) {
    if (p.dual == 2) {  // interleaved (first, second) pairs
      mat = t & 1;
      lt = t >> 1;
    } else {
      mat = (p.dual && t >= t_one) ? 1 : 0;
      lt = t - mat * t_one;
    }
  };
  auto tile_map = [&](int t, int& mat, int& lt) -> int {
    tile_split(t, mat, lt);
    if (hit_tiles) {
      const int tpe = p.rows_per_expert / kTileRows;
      const int j = lt / tpe;
      return hit_of(j) * p.rows_per_expert + (lt - j * tpe) * kTileRows;
    }
    return lt * kTileRows;
  };

  // tiles of this CTA (whole pairs for the SwiGLU epilogue)
  const int tiles = p.dual ? 2 * t_one : t_one;
  const int unit = (p.dual == 2) ? 2 : 1;
  const int tile_lo = unit * (int)((long)blockIdx.x * (tiles / unit) / gridDim.x);
  const int tile_hi = unit * (int)((long)(blockIdx.x + 1) * (tiles / unit) / gridDim.x);
  const int ntile = tile_hi - tile_lo;
  if (MODE == kModeY && k_len <= 0) {
    // an empty reduction range still owns its split's partial outputs: zeros
    float* const yo = p.y + (size_t)blockIdx.y * p.S * ldy;
    for (int v = threadIdx.x; v < ntile * kTileRows * p.S; v += blockDim.x) {
      const int n = v / (ntile * kTileRows), tr = v - n * (ntile * kTileRows);
      int mat, lt;
      tile_split(tile_lo + tr / kTileRows, mat, lt);
      const int row = lt * kTileRows + (tr % kTileRows);
      if (row < n_one) yo[(size_t)n * ldy + mat * p.N + row] = 0.f;
    }
    return;
  }
  const int depth = pl.depth;

  const uint32_t x_base = base + pl.x_off;
  const uint32_t ring = base + pl.ring_off;
  const uint32_t sc_ring = base + pl.sc_off;
  const uint32_t bars = base + pl.bar_off;
  const uint32_t bar_full = bars, bar_empty = bars + 8 * depth;
  const uint32_t bar_afull = bars + 16 * depth;        // [A buffer]
  const uint32_t bar_afree = bar_afull + 8 * kABufs;  // [A buffer]
  const uint32_t bar_tfull = bar_afree + 8 * kABufs;  // [tile buf]
  const uint32_t bar_tfree = bar_tfull + 2 * 8;  // [tile buf]
  const uint32_t bar_xready = bar_tfree + 2 * 8;  // [row slice]: staged (epilogue warps)
  const uint32_t bar_drain = bar_xready + 8 * (pl.kpad / 256);  // MMA warp: all its tcgen05 work done
  float* const best_v = reinterpret_cast<float*>(sb + pl.best_off);
  int* const best_i = reinterpret_cast<int*>(sb + pl.best_off + 4 * 32 * 4);
  uint32_t* const s_tmem = reinterpret_cast<uint32_t*>(sb + pl.misc_off);
  volatile int* const s_dead = reinterpret_cast<volatile int*>(sb + pl.misc_off + 4);
  int* const s_flag = reinterpret_cast<int*>(sb + pl.misc_off + 8);
  int* const s_am = reinterpret_cast<int*>(sb + pl.misc_off + 16);
  int* const s_drafts = reinterpret_cast<int*>(sb + pl.misc_off + 16 + 32 * 4);

  // the stage sequence
  const int kst = (k_len + 255) / 256;
  const int nblk_total = k_len / 32;
  const int nstages = ntile * kst;
  const int kbyte0 = (QB == 8) ? k_begin : k_begin / 2;
  const int kbyte_end = (QB == 8) ? k_begin + k_len : (k_begin + k_len) / 2;

  auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
    if (*s_dead) return false;
    if (mbar_try_wait(bar, parity)) return true;
    // the limit is read only on the slow path (a test may shorten it)
    if (mbar_wait_bounded(bar, parity, p.wait_ns != 0 ? p.wait_ns : kWaitLimitNs)) return true;
    *s_dead = 1;
    atomicOr(p.status, kDevErrTimeout);
    return false;
  };
  // all 32 lanes wait (each acquires the phase), then agree, so that the
  // warp-wide tcgen05.ld / tcgen05.st that follow run converged
  auto wait_warp = [&](uint32_t bar, uint32_t parity) -> bool {
    const bool ok = wait(bar, parity);
    return __all_sync(0xffffffffu, ok) != 0;
  };
  // Stage cursor: position i in the stage sequence and its derived indices,
  // advanced incrementally (no per-stage integer division).
  // ks is the stage's position within its tile, kx the 256-column slice of the
  // reduction it covers: each CTA walks a tile's slices starting at its own
  // rotation, so the CTAs do not all fetch the same window-row slice at once.
  struct Cursor {
    int i, slot, phase, ks, kx, t, ab, abphase;
  };
  const int rot = (kst > 0) ? (int)(blockIdx.x % (unsigned)kst) : 0;
  auto cursor_at = [&](int i) -> Cursor {
    const int ks = i % kst;
    return Cursor{i, i % depth, (i / depth) & 1, ks, (ks + rot) % kst, i / kst, i % kABufs, (i / kABufs) & 1};
  };
  auto advance = [&](Cursor& c) {
    ++c.i;
    if (++c.slot == depth) { c.slot = 0; c.phase ^= 1; }
    if (++c.ks == kst) {
      c.ks = 0;
      c.kx = rot;
      ++c.t;
    } else if (++c.kx == kst) {
      c.kx = 0;
    }
    if (++c.ab == kABufs) { c.ab = 0; c.abphase ^= 1; }
  };
  // advance by the G stages between a converter group's stages: the same state
  // as G calls of advance() (G < depth and G <= kABufs, so slot and A buffer wrap
  // at most once), in fewer instructions
  auto advance_g = [&](Cursor& c, int G) {
    c.i += G;
    c.slot += G;
    if (c.slot >= depth) {
      c.slot -= depth;
      c.phase ^= 1;
    }
    c.ks += G;
    c.kx += G;
    while (c.ks >= kst) {  // a new tile starts at slice rot
      c.ks -= kst;
      ++c.t;
    }
    while (c.kx >= kst) c.kx -= kst;  // kx = (ks + rot) mod kst throughout
    c.ab += G;
    if (c.ab >= kABufs) {
      c.ab -= kABufs;
      c.abphase ^= 1;
    }
  };
  uint64_t policy = 0;
  auto issue = [&](const Cursor& c) {  // TMA of stage c.i into ring slot c.slot
    // the timeout-path test withholds one stage: its slot never fills, and the
    // slot's previous copy has been consumed, so nothing is in flight there
    if (p.debug_withhold == c.i + 1) return;
    const int slot = c.slot, ks = c.kx;
    int mat, lt;
    int row0 = tile_map(tile_lo + c.t, mat, lt);
    const int boxes = (QB == 8) ? 2 : 1;
    int xb, sc_col;
    bool all_boxes = false;
    if (segs) {  // expert segment of this stage (seg_k is a multiple of 256)
      const int kk = k_begin + ks * 256;
      const int j = kk / p.seg_k, col = kk - j * p.seg_k;
      row0 = hit_of(j) * p.rows_per_expert + lt * kTileRows;
      xb = (QB == 8) ? col : col / 2;
      sc_col = col / 32;
      all_boxes = true;
    } else {
      xb = kbyte0 + ks * 128 * boxes;
      sc_col = k_begin / 32 + ks * 8;
    }
    const CUtensorMap* const mc = mat ? &tm_codes2 : &tm_codes;
    const CUtensorMap* const ms = mat ? &tm_scales2 : &tm_scales;
    uint32_t bytes = p.scales_tma ? kTileRows * 16 : 0;
    for (int bx = 0; bx < boxes; ++bx)
      if (all_boxes || xb + 128 * bx < kbyte_end) bytes += kTileRows * 128;
    const uint32_t fb = bar_full + 8 * slot;
    mbar_arrive_expect_tx(fb, bytes);
    for (int bx = 0; bx < boxes; ++bx)
      if (all_boxes || xb + 128 * bx < kbyte_end)
        tma_load_2d(ring + slot * pl.code_stage + bx * kTileRows * 128, mc, xb + 128 * bx, row0, fb, policy);
    if (p.scales_tma) tma_load_2d(sc_ring + slot * pl.sc_stage, ms, sc_col, row0, fb, policy);
  };

  if (threadIdx.x == 0) {
    for (int d = 0; d < depth; ++d) {
      mbar_init(bar_full + 8 * d, 1);
      mbar_init(bar_empty + 8 * d, 4);  // the four warps of the stage's group
    }
    for (int j = 0; j < kABufs; ++j) {
      mbar_init(bar_afull + 8 * j, 4);
      mbar_init(bar_afree + 8 * j, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tfree + 8 * b, 4);
    }
    for (int j = 0; j < pl.kpad / 256; ++j) mbar_init(bar_xready + 8 * j, 4 * 32);
    mbar_init(bar_drain, 1);
    *s_dead = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(s_tmem), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x < 4 * 32) {
    best_v[threadIdx.x] = -FLT_MAX;
    best_i[threadIdx.x] = INT_MAX;
  }
  if (!dep_early) griddep_wait();
  // the drafts, for the accept at the end (whichever CTA runs it)
  if (MODE != kModeY && warp == 2 && lane < p.n_valid) s_drafts[lane] = p.drafts[lane];

  tc_fence_before();
  __syncthreads();  // barriers initialised, tensor memory allocated
  tc_fence_after();
  // An allocation of all 512 columns always starts at lane 0, column 0.  Every
  // tensor-memory address below is built on that constant, so the MMA operands
  // are warp-uniform expressions of the loop counters (a base loaded from shared
  // memory is not provably uniform and each MMA would pay to make it so).
  constexpr uint32_t tmem = 0u;
  if (threadIdx.x == 0 && *s_tmem != tmem) atomicOr(p.status, kDevErrTmemBase);

  // ---- start the weight stream (the TMA unit carries only weights: each TMA
  // issue costs ~0.15 us at start-up) ----
  if (threadIdx.x == 0) {
    policy = l2_policy_evict_first();
    tma_prefetch_desc(&tm_codes);
    if (p.scales_tma) tma_prefetch_desc(&tm_scales);
    if (p.dual) {
      tma_prefetch_desc(&tm_codes2);
      if (p.scales_tma) tma_prefetch_desc(&tm_scales2);
    }
    Cursor c = cursor_at(0);
    for (; c.i < depth && c.i < nstages; advance(c)) issue(c);
  }
  // ---- window rows, slice by slice in this CTA's rotated order: the epilogue
  // warps (idle until the first tile) load each 16-byte chunk, permute it like
  // the converted codes and store it as K-major core matrices (zeros past S and
  // past the reduction length); the MMA warp waits for the slice it multiplies ----
  if (warp >= 2 && warp < R::kConv0) {
    const int st = threadIdx.x - 64;
    constexpr int kStagers = 4 * 32;
    constexpr int kBatch = 4;
    const int sbo = pl.kpad * 16;     // bytes between 8-row groups
    const int chunks = pl.xrows * 32;  // 16-byte chunks of one slice
    for (int j = 0; j < kst; ++j) {
      const int ks = (rot + j) % kst;
      const int gv = min(32, max(0, k_len / 8 - 32 * ks));  // groups holding window data
      for (int base = st; base < chunks; base += kBatch * kStagers) {
        uint4 in[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int v = base + u * kStagers;
          const int n = v >> 5, g = v & 31;
          in[u] = make_uint4(0u, 0u, 0u, 0u);
          if (v < chunks && n < p.S && g < gv)
            in[u] = *reinterpret_cast<const uint4*>(p.x + (size_t)n * ldx + k_begin + 8 * (32 * ks + g));
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int v = base + u * kStagers;
          if (v >= chunks) break;
          const int n = v >> 5, g8 = 32 * ks + (v & 31);
          const uint4 x4 = in[u];
          uint4 o;
          if (QT == 2) {  // FP4: the converters' pairs are (k0, k1), (k2, k3), ...: as stored
            o = x4;
          } else if (QB == 8) {  // per 4 elements: (k0, k2, k1, k3)
            o.x = __byte_perm(x4.x, x4.y, 0x5410);
            o.y = __byte_perm(x4.x, x4.y, 0x7632);
            o.z = __byte_perm(x4.z, x4.w, 0x5410);
            o.w = __byte_perm(x4.z, x4.w, 0x7632);
          } else {  // int4, per 8 elements (word j of a 32-block): pairs (k0, k4), (k1, k5), (k2, k6), (k3, k7)
            o.x = __byte_perm(x4.x, x4.z, 0x5410);
            o.y = __byte_perm(x4.x, x4.z, 0x7632);
            o.z = __byte_perm(x4.y, x4.w, 0x5410);
            o.w = __byte_perm(x4.y, x4.w, 0x7632);
            // the converters put a block's (k0, k4) and (k2, k6) pairs in its first
            // eight columns (the first MMA of the block) and (k1, k5), (k3, k7) in
            // the last eight: word j's pairs go to columns 2j, 2j + 1 and 8 + 2j,
            // 9 + 2j, 4 columns (16 bytes) per core-matrix row
            const int j = g8 & 3, blk0 = g8 - j;
            uint8_t* const row = sb + pl.x_off + (n >> 3) * sbo + (n & 7) * 16 + (j & 1) * 8;
            *reinterpret_cast<uint2*>(row + (blk0 + (j >> 1)) * 128) = make_uint2(o.x, o.z);
            *reinterpret_cast<uint2*>(row + (blk0 + 2 + (j >> 1)) * 128) = make_uint2(o.y, o.w);
            continue;
          }
          *reinterpret_cast<uint4*>(sb + pl.x_off + (n >> 3) * sbo + g8 * 128 + (n & 7) * 16) = o;
        }
      }
      fence_proxy_async_smem();  // generic-proxy writes, read by the tensor cores
      mbar_arrive(bar_xready + 8 * ks);
    }
  }

  if (warp == 0) {
    // ---------------- TMA producer -------------------------------------------------
    if (lane == 0) {
      int issued = min(depth, nstages);
      for (Cursor c = cursor_at(depth); c.i < nstages; advance(c)) {
        if (!wait(bar_empty + 8 * c.slot, c.phase ^ 1)) break;
        // a slot released by a converter that gave up (it did not wait for the
        // slot's copy) is not refilled: every slot keeps at most one copy in flight
        if (*s_dead) break;
        issue(c);
        issued = c.i + 1;
      }
      // No copy may outlive the CTA.  The latest copy into each slot is the only
      // one that can still be pending: an earlier one was waited for by the
      // converter that released the slot, or the slot was not refilled.  Wait for
      // them (bounded) whatever happens to the rest of the CTA: in a normal run
      // they land and are consumed anyway; after a timeout a converter may have
      // stopped waiting for them.
      for (int j = max(0, issued - depth); j < issued; ++j)
        if (p.debug_withhold != j + 1)  // a withheld stage has no copy to wait for
          mbar_wait_bounded(bar_full + 8 * (j % depth), (j / depth) & 1, kDrainLimitNs);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (warp-uniform loop, one elected lane issues) ------
    // Per stage: uniform bases, then 16 MMAs at compile-time offsets.
    const uint32_t idesc = idesc_f16_f32(kTileRows, NM);
    const uint64_t bdesc0 = smem_desc_kmajor(x_base, 128u, (uint32_t)pl.kpad * 16u);
    Cursor c = cursor_at(0);
    for (; c.i < nstages; advance(c)) {
      const int t = c.t, ks = c.ks, tb = t & 1;
      const int ab = c.ab;
      if (ks == 0 && t >= 2 && !wait_warp(bar_tfree + 8 * tb, ((t >> 1) - 1) & 1)) break;
      // first tile: the slice of window rows this stage multiplies must be in place
      if (t == 0 && !wait_warp(bar_xready + 8 * c.kx, 0)) break;
      const uint32_t a_stage = tmem + (uint32_t)(ab * 128);
      const uint32_t d_tile = tmem + (uint32_t)(kACols + tb * kAcc * NM);
      // descriptor start address advances by k (16-byte units) per reduction element k
      const uint64_t b_stage = bdesc0 + (uint64_t)(c.kx * 256);
      const bool later = ks > 0;
      if (!wait_warp(bar_afull + 8 * ab, c.abphase)) break;
      tc_fence_after();
      // the stage's 16 MMAs (k = 16m .. 16m+15) in one straight-line block under a
      // single elect: a branch or a fresh elect per MMA costs issue slots that
      // the converters on this scheduler need
      tc_mma_stage16<kAcc>(d_tile, a_stage, b_stage, idesc, (uint32_t)NM, later ? 1u : 0u);
      tc_commit_elect(bar_afree + 8 * ab);
      if (ks == kst - 1) tc_commit_elect(bar_tfull + 8 * tb);
    }
    // No asynchronous arrive may outlive the CTA (a late one would land in the
    // shared memory of the next CTA on this SM), and no MMA may run into freed
    // tensor memory: one more commit tracks every MMA and commit this thread
    // issued, and the warp waits for it -- bounded, and also after a timeout,
    // when the loop above stopped early (c.i stages issued).
    for (int d = max(0, c.i - kABufs); d < c.i; ++d) {  // the last A-buffer releases
      const Cursor cd = cursor_at(d);
      mbar_wait_bounded(bar_afree + 8 * cd.ab, cd.abphase, kDrainLimitNs);
    }
    tc_commit_elect(bar_drain);
    mbar_wait_bounded(bar_drain, 0, kDrainLimitNs);
    __syncwarp();
  } else if (warp < R::kConv0) {
    // ---------------- tile epilogue (one warp per tensor-memory lane quarter) --------
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    float* const red = reinterpret_cast<float*>(sb + pl.red_off) + q * p.S * 33;  // [S][33]
    float run_v = -INFINITY;  // running best of column n = lane (no row yet: -inf, INT_MAX)
    int run_i = INT_MAX;
    // sampling verify, per column: the top 1 of z = L/T + g over the entries other
    // than the row's draft (with its entry), the draft's own z and L/T (NaN: not
    // in this CTA's rows), the softmax max and sum of L/T
    float zx = -INFINITY, z_d = __int_as_float(0x7fc00000), sm_m = -INFINITY, sm_s = 0.f,
          l_d = __int_as_float(0x7fc00000);
    int vx = INT_MAX;
    // sampling scans: L lanes per column (32 over the next power of two >= S), so a
    // small window spreads each column's 32 rows over many lanes; lane cc * L owns
    // column cc's running state
    const int s_pow2 = p.S <= 1 ? 1 : p.S <= 2 ? 2 : p.S <= 4 ? 4 : p.S <= 8 ? 8 : p.S <= 16 ? 16 : 32;
    const int s_lanes = 32 / s_pow2;
    const int s_col = lane / s_lanes, s_sub = lane % s_lanes;
    const bool s_act = s_col < p.S, s_own = s_act && s_sub == 0;
    const int s_dv = (MODE == kModeSample && s_col < p.n_valid) ? s_drafts[s_col] : -1;  // the column's draft
    const int tpe = p.rows_per_expert > 0 ? p.rows_per_expert / kTileRows : 1;
    for (int t = 0; t < ntile; ++t) {
      const int tb = t & 1;
      if (!wait_warp(bar_tfull + 8 * tb, (t >> 1) & 1)) break;
      tc_fence_after();
      float acc[32];
#pragma unroll
      for (int n = 0; n < 32; ++n) acc[n] = 0.f;
      // int4: the even MMAs of a block (into the even accumulators) carry the
      // pairs the converters scaled by 2^-4, so those accumulators count 16-fold
      // (an exact power of two)
#pragma unroll
      for (int j = 0; j < kAcc; ++j) {
        const uint32_t col = (uint32_t)(kACols + (tb * kAcc + j) * NM);
        const float wj = (QT == 4 && (j & 1) == 0) ? 16.f : 1.f;
        uint32_t v[16];
        tmem_ld16(tmem + lane_base + col, v);
        tmem_wait_ld();
#pragma unroll
        for (int n = 0; n < 16; ++n) acc[n] = fmaf(wj, __uint_as_float(v[n]), acc[n]);
        if (NM == 32) {
          tmem_ld16(tmem + lane_base + col + 16, v);
          tmem_wait_ld();
#pragma unroll
          for (int n = 0; n < 16; ++n) acc[16 + n] = fmaf(wj, __uint_as_float(v[n]), acc[16 + n]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tfree + 8 * tb);
      int mat, lt;
      tile_split(tile_lo + t, mat, lt);
      const int lrow = lt * kTileRows + r;  // row within its matrix
      const bool valid = lrow < n_one;
      if (MODE == kModeY && p.dual == 2) {
        // the pair's first tile waits in this warp's shared-memory rows (lane = row)
        if (mat == 0) {
#pragma unroll
          for (int n = 0; n < 32; ++n)
            if (n < p.S) red[n * 33 + lane] = acc[n];
        } else {
          // the routing weights of this tile's expert slot, all in registers before
          // the first store of h (which the compiler could not otherwise move them
          // past): written by the router before this grid started, or, routed in
          // this launch, lane n's weight of row n for the slot's expert (zero where
          // row n did not pick it), passed round the warp
          const bool weighted = routed || p.row_w != nullptr;
          float wv[32];
          if (routed) {
            const int e = s_hit[lt / tpe];
            float mine = 0.f;
            if (lane < p.S)
              for (int i = 0; i < p.route_top_k; ++i)
                if (s_rids[lane * kRouteMaxTopK + i] == e) mine = s_rw[lane * kRouteMaxTopK + i];
#pragma unroll
            for (int n = 0; n < 32; ++n) wv[n] = __shfl_sync(0xffffffffu, mine, n);
          } else {
            const float* const rw = (p.row_w != nullptr) ? p.row_w + lt / tpe : nullptr;
#pragma unroll
            for (int n = 0; n < 32; ++n) wv[n] = (rw != nullptr && n < p.S) ? __ldg(rw + (size_t)n * p.ldw) : 1.f;
          }
          if (valid) {
#pragma unroll
            for (int n = 0; n < 32; ++n) {
              if (n < p.S) {
                // SiLU(g) = g / (1 + exp(-g)) with the hardware exponential and
                // division (relative error ~1e-6, far below the fp16 rounding of h;
                // large negative g: the quotient goes to -0)
                const float g = red[n * 33 + lane];
                float v = __fdividef(g, 1.f + __expf(-g)) * acc[n];
                if (weighted) v *= wv[n];
                p.h[(size_t)n * p.ldh + lrow] = __float2half_rn(v);
              }
            }
          }
        }
      } else if (p.y != nullptr && valid) {
        float* const yo = p.y + (size_t)blockIdx.y * p.S * ldy + mat * p.N + lrow;
#pragma unroll
        for (int n = 0; n < 32; ++n)
          if (n < p.S) yo[(size_t)n * ldy] = acc[n];
      }
      if (MODE == kModeHead) {
        // columns through shared memory: lane n then scans the warp's 32 rows
        // (rows past the vocabulary as -inf, which never wins the scan below)
#pragma unroll
        for (int n = 0; n < 32; ++n)
          if (n < p.S) red[n * 33 + lane] = valid ? acc[n] : -INFINITY;
        __syncwarp();
        if (lane < p.S) {
          // rows reach a lane in increasing index order (tiles, then rows), so a
          // later row wins only with a strictly larger value: the argmax order
          // (larger value, then lower index) without its tie test
          const int row0 = (tile_lo + t) * kTileRows + 32 * q;
          for (int j = 0; j < 32; ++j) {
            const float v = red[lane * 33 + j];
            if (v > run_v) {
              run_v = v;
              run_i = row0 + j;
            }
          }
        }
        __syncwarp();
      }
      if (MODE == kModeSample) {
        // Rolled loops over small bodies throughout (the fully unrolled form of
        // this code measured 25-35 % slower); the epilogue warps share their
        // schedulers with busy converters, so every instruction here counts.
        // (1) l = L/T of this thread's row, column n at red[n][lane]
#pragma unroll
        for (int n = 0; n < 32; ++n)
          if (n < p.S) red[n * 33 + lane] = acc[n] * p.inv_temp;
        __syncwarp();
        const int row0 = (tile_lo + t) * kTileRows + 32 * q;
        const int nrow = max(0, min(32, p.N - row0));  // rows of this warp's slab inside the vocabulary
        // (2) column s_col over its lanes: the slab's max, its sum of exp(l - max)
        // (butterflies within the lane group), and the draft's l
        {
          const float* const col = red + s_col * 33;
          float m = -INFINITY;
          if (s_act)
            for (int j = s_sub; j < nrow; j += s_lanes) m = fmaxf(m, col[j]);
          for (int o = s_lanes >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          float e = 0.f;
          if (s_act)
            for (int j = s_sub; j < nrow; j += s_lanes) e += expf(col[j] - m);
          for (int o = s_lanes >> 1; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
          if (s_own) {
            softmax_merge(sm_m, sm_s, m, e);
            if (s_dv >= row0 && s_dv < row0 + nrow) l_d = col[s_dv - row0];
          }
        }
        __syncwarp();
        // (3) z = l + g for this thread's row: entry lrow, column n is element
        // 32 lrow + n, so one counter output serves columns 2c and 2c + 1
        if (valid) {
          const unsigned long long c0 = (unsigned long long)(unsigned)lrow * 16ull;
#pragma unroll 2
          for (int c = 0; c < (p.S + 1) / 2; ++c) {
            const unsigned long long w = counter_pair(p.rng_key, c0 + (unsigned)c);
            red[(2 * c) * 33 + lane] += gumbel_of(half_uniform((unsigned)w));
            if (2 * c + 1 < p.S) red[(2 * c + 1) * 33 + lane] += gumbel_of(half_uniform((unsigned)(w >> 32)));
          }
        }
        __syncwarp();
        // (4) column s_col over its lanes: the draft's entry leaves the slab (its z
        // kept aside), then the top 1 of z over the rest, merged across the lane
        // group by a butterfly.  The draw from p without the draft is that top 1;
        // the draw from p is the draft where its z beats it, else the same entry.
        {
          float* const col = red + s_col * 33;
          if (s_own && s_dv >= row0 && s_dv < row0 + nrow) {
            z_d = col[s_dv - row0];
            col[s_dv - row0] = -INFINITY;
          }
          __syncwarp();
          // a lane's rows come in increasing index order, so a later row wins
          // only with a strictly larger z (the argmax order without its tie test)
          float a = -INFINITY;
          int b = INT_MAX;
          if (s_act)
            for (int j = s_sub; j < nrow; j += s_lanes) {
              const float z = col[j];
              if (z > a) {
                a = z;
                b = row0 + j;
              }
            }
          for (int o = s_lanes >> 1; o > 0; o >>= 1)
            top1_add(a, b, __shfl_xor_sync(0xffffffffu, a, o), __shfl_xor_sync(0xffffffffu, b, o));
          // earlier tiles hold lower rows: again a strictly larger z wins
          if (s_own && a > zx) {
            zx = a;
            vx = b;
          }
        }
        __syncwarp();
      }
    }
    if (MODE == kModeHead && lane < p.S) {
      best_v[q * 32 + lane] = run_v;
      best_i[q * 32 + lane] = run_i;
    }
    if (MODE == kModeSample) {
      // the four warps' column states into shared memory, [field][quarter][S],
      // once every epilogue warp is done with its rows of the reduction buffer
      named_bar_sync(1, 4 * 32);
      float* const st = reinterpret_cast<float*>(sb + pl.red_off);
      if (s_own) {
        const int o = q * p.S + s_col, f = 4 * p.S;
        st[o] = zx;
        st[f + o] = __int_as_float(vx);
        st[2 * f + o] = z_d;
        st[3 * f + o] = sm_m;
        st[4 * f + o] = sm_s;
        st[5 * f + o] = l_d;
      }
    }
  } else {
    // ---------------- converters ------------------------------------------------------
    // Group g converts whole stages g, g+G, g+2G, ...: while one group waits for
    // its next stage the others convert, and each stage is one hand-off to the
    // MMA warp.
    const int cw = warp - R::kConv0;
    const int q = warp & 3;
    const int g = cw >> 2;
    const int r = 32 * q + lane;  // row within the tile (= TMEM lane)
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const int ks_per_row = p.K / 32;
    // A row's codes of a stage are loaded in parts of kHalfBlocks blocks: int8
    // two halves (a 128-byte row of each half of the stage); int4 two halves of
    // its 128-byte row (fewer registers held by the codes); FP4 the whole row at
    // once (measured faster for its shorter conversion).
    constexpr int kHalves = (QT == 2) ? 1 : 2;
    constexpr int kHalfBlocks = 8 / kHalves;               // 32-blocks per part
    constexpr int kLoads = (QB == 8) ? 8 : kHalfBlocks;    // 16-byte loads per part
    const int sw = r & 7;
    Cursor c = cursor_at(0);
    for (int j = 0; j < g; ++j) advance(c);
    for (; c.i < nstages;) {
      const int slot = c.slot;
      const int ab = c.ab;
      // the A buffer first, then the ring slot (the order tc_plan_valid relies on)
      bool ok = true;
      if (c.i >= kABufs) ok = wait_warp(bar_afree + 8 * ab, c.abphase ^ 1);
      if (ok) ok = wait_warp(bar_full + 8 * slot, c.phase);
      const uint8_t* const cb = sb + pl.ring_off + slot * pl.code_stage;
      // the 8 block scales of row r, two per word (block 2j in the low half);
      // blocks past the reduction length get zero, so their A columns are zero
      // (the padded window rows are zero too)
      uint32_t sc_w[4] = {0u, 0u, 0u, 0u};
      if (ok) {
        if (p.scales_tma) {
          const uint4 sv = *reinterpret_cast<const uint4*>(sb + pl.sc_off + slot * pl.sc_stage + r * 16);
          sc_w[0] = sv.x;
          sc_w[1] = sv.y;
          sc_w[2] = sv.z;
          sc_w[3] = sv.w;
        } else {
          const int row = (tile_lo + c.t) * kTileRows + r;
          const int ks = c.kx;
          const int nb = max(0, min(8, nblk_total - ks * 8));  // blocks within the reduction length
#pragma unroll
          for (int blk = 0; blk < 8; ++blk)
            if (blk < nb && row < p.N)
              sc_w[blk >> 1] |= (uint32_t)__ldg(p.scales + (size_t)row * ks_per_row + k_begin / 32 + ks * 8 + blk)
                                << (16 * (blk & 1));
        }
      }
      // The stage's conversion, in one of two forms chosen once per stage (a
      // branch per block inside the unrolled loop costs more than it saves):
      // integer codes with scale and bias in one HFMA2 per pair where every
      // row's eight block scales are in range -- int4: s * 2^20 <= 65504 (fp16
      // bits <= 0x2BFF) and s / 2 exact, int8: s * 2^24 <= 65504 (bits <=
      // 0x1BFF), the common case -- else the two-step form; the same bits.
      auto convert = [&](auto fma_tag) {
        constexpr bool kFma = decltype(fma_tag)::value;
#pragma unroll
      for (int h = 0; h < kHalves; ++h) {
        uint4 wreg[kLoads];
        if (ok) {
          const uint8_t* const row_p = cb + (QB == 8 ? h * kTileRows * 128 : 0) + r * 128;
#pragma unroll
          for (int w = 0; w < kLoads; ++w) {
            const int chunk = (QB == 8) ? w : kLoads * h + w;
            wreg[w] = *reinterpret_cast<const uint4*>(row_p + ((chunk ^ sw) << 4));
          }
        }
        if (h == kHalves - 1) {  // the ring slot goes back to the producer
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
        }
        if (h == 0 && ok) tc_fence_after();
        if (ok) {
#pragma unroll
          for (int blk = 0; blk < kHalfBlocks; ++blk) {
            const int sblk = h * kHalfBlocks + blk;  // block within the stage
            // the block's scale in both halves of a pair: one byte permute
            const __half2 s2 = u32_as_h2(__byte_perm(sc_w[sblk >> 1], 0u, (sblk & 1) ? 0x3232u : 0x1010u));
            uint32_t cols[16];
            if (QB == 8) {
              const uint32_t wv[8] = {wreg[2 * blk].x, wreg[2 * blk].y, wreg[2 * blk].z, wreg[2 * blk].w,
                                      wreg[2 * blk + 1].x, wreg[2 * blk + 1].y, wreg[2 * blk + 1].z,
                                      wreg[2 * blk + 1].w};
              if constexpr (kFma) {
                const __half2 k12 = __float2half2_rn(4096.f);
                const __half2 m2 = __hmul2(__hmul2(s2, k12), k12);
                const __half2 c2 = __hmul2(s2, __float2half2_rn(-128.f));
#pragma unroll
                for (int j = 0; j < 8; ++j) i8x4_to_h2x2_scaled(wv[j], m2, c2, cols[2 * j], cols[2 * j + 1]);
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) i8x4_to_h2x2(wv[j], cols[2 * j], cols[2 * j + 1]);
              }
            } else if (QT == 4) {
              // word j's (n0, n4), (n2, n6) pairs (scaled by 2^-4) to columns 2j,
              // 2j + 1 (the block's first MMA, accumulated into the accumulators
              // the epilogue scales by 16), (n1, n5), (n3, n7) to 8 + 2j, 9 + 2j
              const uint32_t wv[4] = {wreg[blk].x, wreg[blk].y, wreg[blk].z, wreg[blk].w};
              if constexpr (kFma) {
                const __half2 m2 = __hmul2(__hmul2(s2, __float2half2_rn(1024.f)), __float2half2_rn(1024.f));
                const __half2 c2 = __hmul2(s2, __float2half2_rn(-8.f));
                const __half2 clo2 = __hmul2(s2, __float2half2_rn(-0.5f));
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  i4x8_to_h2x4_split(wv[j], m2, c2, clo2, cols[2 * j], cols[8 + 2 * j], cols[2 * j + 1],
                                     cols[9 + 2 * j]);
              } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  i4x8_to_h2x4_split_exact(wv[j], cols[2 * j], cols[8 + 2 * j], cols[2 * j + 1], cols[9 + 2 * j]);
              }
            } else {  // FP4: the hardware E2M1 -> f16x2 conversion, one byte (two codes) at a time
              const uint32_t wv[4] = {wreg[blk].x, wreg[blk].y, wreg[blk].z, wreg[blk].w};
#pragma unroll
              for (int j = 0; j < 4; ++j)
                e2m1x8_to_h2x4(wv[j], cols[4 * j], cols[4 * j + 1], cols[4 * j + 2], cols[4 * j + 3]);
            }
            // the two-step form (and FP4) multiply by the scale after the conversion
            if (!(kFma && QT != 2)) {
#pragma unroll
              for (int j = 0; j < 16; ++j) cols[j] = h2_as_u32(__hmul2(u32_as_h2(cols[j]), s2));
            }
            tmem_st16(tmem + lane_base + (uint32_t)(ab * 128 + sblk * 16), cols);
          }
        }
      }
      };
      bool fma_form = false;
      if ((QT == 4 || QT == 8) && ok) {
        constexpr uint32_t kMaxBits = (QT == 4) ? 0x2BFFu : 0x1BFFu;  // the largest scale in range
        // int4 also needs s / 2 exact: s = 0 or s >= 2^-13 (fp16 bits 0x0800)
        auto in_range = [](uint32_t b) {
          return b <= kMaxBits && (QT != 4 || b == 0u || b >= 0x0800u);
        };
        bool small = true;
#pragma unroll
        for (int w = 0; w < 4; ++w) small = small && in_range(sc_w[w] & 0xFFFFu) && in_range(sc_w[w] >> 16);
        fma_form = __all_sync(0xffffffffu, small);
      }
      if (fma_form)
        convert(std::true_type{});
      else
        convert(std::false_type{});
      if (ok) {
        tmem_wait_st();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_afull + 8 * ab);
      advance_g(c, R::G);
    }
  }

  // ---- teardown ------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();  // the next grid may take this SM once the CTA exits
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }

  if (MODE == kModeY) return;
  if (MODE == kModeSample) {
    sample_tail(p, sb + pl.red_off, s_drafts, s_flag, warp, lane, R::kWarps);
    return;
  }
  if (threadIdx.x < p.S) {
    const int col = threadIdx.x;
    float bv = best_v[col];
    int bi = best_i[col];
    for (int q = 1; q < 4; ++q) argmax_merge(bv, bi, best_v[q * 32 + col], best_i[q * 32 + col]);
    __stcg(p.part_v + (size_t)blockIdx.x * p.S + col, bv);
    __stcg(p.part_i + (size_t)blockIdx.x * p.S + col, bi);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // one acquire-release ticket: publishes this CTA's partials (the release is
    // cumulative over the block's stores before the barrier) and, for the last
    // CTA, acquires every other CTA's; the barrier below passes that on
    unsigned tk;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(tk) : "l"(p.ticket) : "memory");
    *s_flag = (tk == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (*s_flag == 0) return;
  for (int col = warp; col < p.S; col += R::kWarps) {
    float bv = -FLT_MAX;
    int bi = INT_MAX;
    // all of a lane's partials are loaded before they are merged (one round of latency)
    constexpr int kPf = 8;
    float pv[kPf];
    int pi[kPf];
#pragma unroll
    for (int u = 0; u < kPf; ++u) {
      const int j = lane + 32 * u;
      pv[u] = -FLT_MAX;
      pi[u] = INT_MAX;
      if (j < (int)gridDim.x) {
        pv[u] = __ldcg(p.part_v + (size_t)j * p.S + col);
        pi[u] = __ldcg(p.part_i + (size_t)j * p.S + col);
      }
    }
#pragma unroll
    for (int u = 0; u < kPf; ++u) argmax_merge(bv, bi, pv[u], pi[u]);
    for (int j = lane + 32 * kPf; j < (int)gridDim.x; j += 32)
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
  if (warp == 0) {  // accepted = the first window position whose draft misses (n_valid <= 31)
    const bool hit = lane < p.n_valid && s_drafts[lane] == s_am[lane];
    const unsigned miss = ~__ballot_sync(0xffffffffu, hit);
    const int j = __ffs(miss) - 1;
    if (lane == 0) {
      *p.accepted = j;
      *p.next_a0 = s_am[j];
      *p.ticket = 0u;
    }
  }
}

struct TcMaps {
  const CUtensorMap &c, &s, &c2, &s2;
};

template <int QT, int MODE, int NM>
cudaError_t tc_launch_t(const TcMaps& m, const GemmArgs& a, int grid, int smem, cudaStream_t st) {
  auto k = tc_gemm_kernel<QT, MODE, NM>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // the CTAs may be scheduled while the previous kernel drains; they wait for it
  // in griddep_wait()
  constexpr int kThreads = TcRoles<(QT == 8 ? 8 : 4)>::kThreads;
  return launch_pdl(k, dim3(grid, a.splits), dim3(kThreads), (size_t)smem, st, m.c, m.s, m.c2, m.s2, a);
}

template <int QT, int MODE>
cudaError_t tc_launch_nm(const TcMaps& m, const GemmArgs& a, int grid, int smem, cudaStream_t st) {
  return a.S <= 16 ? tc_launch_t<QT, MODE, 16>(m, a, grid, smem, st)
                   : tc_launch_t<QT, MODE, 32>(m, a, grid, smem, st);
}

}  // namespace

int tc_smem_bytes(int qbits, int S, int k_chunk, int depth, bool route) {
  return tc_plan(qbits, S, k_chunk, depth, route).total + 1024;
}

// The aliased 8-row groups of N read up to one group stride past the staged
// rows; the ring behind them must be at least that long.
//
// Before a converter group waits on slot (i % depth) for stage i, the slot's
// previous phase (stage i - depth) must be complete, else the parity wait would
// match the phase before that and return early.  The group first waits for the
// release of its A buffer by the MMAs of stage i - kABufs; the MMAs run in stage
// order, so every stage up to i - kABufs has been converted, hence has landed,
// and any depth >= kABufs is safe.  The ring takes at least kMinDepth stages so
// that the weight stream has some stages in flight.
bool tc_plan_valid(int qbits, int S, int k_chunk, int depth) {
  if (depth < kMinDepth) return false;
  const TcPlan p = tc_plan(qbits, S, k_chunk, depth);
  const int ring_bytes = depth * p.code_stage;
  const int over = (p.nmma - p.xrows) * p.kpad * 2;  // bytes of missing groups
  return over <= ring_bytes;
}

cudaError_t launch_tc_gemm(int qbits, int mode, const CUtensorMap& tm_codes, const CUtensorMap& tm_scales,
                           const CUtensorMap& tm_codes2, const CUtensorMap& tm_scales2, const GemmArgs& a,
                           int grid, int smem, cudaStream_t st) {
  const TcMaps m{tm_codes, tm_scales, tm_codes2, tm_scales2};
  // qbits: 8 int8, 4 int4, 2 FP4 (E2M1)
  if (mode == kModeSample) {
    if (qbits == 8) return tc_launch_nm<8, kModeSample>(m, a, grid, smem, st);
    if (qbits == 4) return tc_launch_nm<4, kModeSample>(m, a, grid, smem, st);
    return tc_launch_nm<2, kModeSample>(m, a, grid, smem, st);
  }
  const bool head = mode == kModeHead;
  if (qbits == 8)
    return head ? tc_launch_nm<8, kModeHead>(m, a, grid, smem, st) : tc_launch_nm<8, kModeY>(m, a, grid, smem, st);
  if (qbits == 4)
    return head ? tc_launch_nm<4, kModeHead>(m, a, grid, smem, st) : tc_launch_nm<4, kModeY>(m, a, grid, smem, st);
  return head ? tc_launch_nm<2, kModeHead>(m, a, grid, smem, st) : tc_launch_nm<2, kModeY>(m, a, grid, smem, st);
}

}  // namespace sdv
