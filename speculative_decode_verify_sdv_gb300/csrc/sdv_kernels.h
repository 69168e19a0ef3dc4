// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace sdv {

// Counts one kernel launch of this library (process-wide; read through
// sdv_launch_count).  Every launch site calls it once its launch succeeded.
void count_launch();
inline cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) count_launch();
  return e;
}

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the previous kernel in the stream drains, and must call
// griddepcontrol.wait before reading anything that kernel wrote.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return counted(cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...));
}

// Device status word bits (first word of every workspace).
constexpr int kDevErrTimeout = 1;
constexpr int kDevErrTmemBase = 2;  // tensor-memory allocation not at column 0

constexpr int kModeY = 0;     // write fp32 Y [S][N]
constexpr int kModeHead = 1;  // verify head: argmax partials + last-CTA reduce + accept
constexpr int kModeSample = 2;  // sampling verify: Gumbel-max draws + softmax partials + last-CTA accept

struct GemmArgs {
  const void* codes;        // weight codes (read directly by the CUDA-core GEMV)
  const __half* x;          // fp16 [S][K]
  const uint16_t* scales;   // fp16 [N][K/32] (read directly when scales_tma == 0)
  int S, N, K;              // window rows, weight rows, reduction length
  int k_chunk;              // reduction length per split (multiple of 256 unless splits == 1)
  int splits;               // gridDim.y; split s covers [s * k_chunk, min(K, (s+1) * k_chunk))
  int m16_tiles;            // ceil(N / 16)
  int depth;                // TMA ring stages per warp
  int scales_tma;           // 1: scales staged by TMA (needs K % 256 == 0)
  float* y;                 // fp32 [splits][S][N]: Y or its split-K partials (kModeY),
                            // or the optional logits (kModeHead, splits == 1)
  // verify head
  const int32_t* drafts;
  int n_valid;
  int32_t* argmax;
  int32_t* accepted;
  int32_t* next_a0;
  float* part_v;            // [grid][S]
  int* part_i;              // [grid][S]
  unsigned* ticket;
  int* status;
  // sampling verify (kModeSample): p_i = softmax(L_i * inv_temp); draws from the
  // counter stream rng_key; per-CTA partials [grid][S][8] (top 1 of L/T + g over
  // the entries other than the row's draft, with its entry; the draft's z;
  // softmax max and sum of L/T; the draft's L/T)
  float inv_temp;
  unsigned long long rng_key;
  float* part_s;
  // ---- row / reduction mappings of the tcgen05 path (kModeY; zero = plain) ----
  int ldx;                  // row stride of x in elements (0: K)
  int ldy;                  // row stride of y in elements (0: N)
  int dual;                 // 1: two weight matrices of N rows each (second tensor maps);
                            //    output column mat * N + row, mat = 0 for the first;
                            // 2: the same two matrices as interleaved (first, second) tile
                            //    pairs with the SwiGLU epilogue: h = SiLU(first) * second
  const int* n_hit;         // device [1]: number of hit experts (MoE), or null
  const int* hit;           // device [n_hit]: expert ids, ascending
  int rows_per_expert;      // rows of one expert in a stacked weight
  int seg_k;                // > 0: the reduction is n_hit segments of seg_k columns, segment j
                            //    reading expert hit[j]'s rows; split y covers segments
                            //    [y * n_hit / splits, (y + 1) * n_hit / splits)
  // SwiGLU epilogue (dual == 2, one split): h[s * ldh + row] = fp16(SiLU(g) * u
  // [* row_w[s * ldw + row / rows_per_expert]])
  __half* h;
  int ldh;
  const float* row_w;
  int ldw;
  // MoE gate/up that routes the window in its own prologue (dual == 2, hit-list
  // tiles; n_hit and hit null): every CTA selects the top route_top_k of each
  // row's route_E router logits ([S][route_E] fp32) and takes the hit list and
  // the routing weights from its own selection; CTA 0 publishes the picks
  // (route_ids, route_w: [S][route_top_k]) and the hit list (route_n_hit,
  // route_hit, experts ascending) for the down projection.  Null: off.
  const float* route_logits;
  int route_E, route_top_k;
  int32_t* route_ids;
  float* route_w;
  int32_t* route_n_hit;
  int32_t* route_hit;
  // ---- timeout-path test hooks of the tcgen05 path (zero = off) ----
  unsigned long long wait_ns;  // limit of every bounded wait (0: kWaitLimitNs)
  int debug_withhold;          // 1 + the stage index whose weight copy the producer never
                               //    issues (its ring slot then never fills), 0 = none
};

int gemm_tile_mt(int qbits);
int gemm_smem_bytes(int qbits, int S, int k_len, int depth);
int gemm_warps_per_cta();
cudaError_t launch_dq_gemm(int qbits, int mode, const CUtensorMap& tm_codes,
                           const CUtensorMap& tm_scales, const GemmArgs& a, int grid, int smem,
                           cudaStream_t st);

int tc_smem_bytes(int qbits, int S, int k_chunk, int depth, bool route = false);
bool tc_plan_valid(int qbits, int S, int k_chunk, int depth);
// The in-prologue MoE routing of the tcgen05 GEMM: its limits
constexpr int kRouteMaxE = 256, kRouteMaxTopK = 8, kRouteMaxS = 32;
cudaError_t launch_tc_gemm(int qbits, int mode, const CUtensorMap& tm_codes,
                           const CUtensorMap& tm_scales, const CUtensorMap& tm_codes2,
                           const CUtensorMap& tm_scales2, const GemmArgs& a, int grid, int smem,
                           cudaStream_t st);

// CUDA-core GEMV for S <= 2: warps per row (0 = not covered), one CTA per SM.
int gemv_plan(int qbits, int k, int S);
cudaError_t launch_gemv(int qbits, int mode, const GemmArgs& a, int warps_per_row, int grid, cudaStream_t st);

cudaError_t launch_splitk_reduce(const float* part, int splits, long count, float* y, cudaStream_t st);

// h[s][c] = fp16(SiLU(g) * u [* row_w[s][c / seg]]) for c < n (or c < *n_dev * seg
// when n_dev is given), with g = sum over splits of part[sp * pstride + s * ldp + c]
// and u the same at + u_off.
cudaError_t launch_swiglu_reduce(const float* part, int splits, long pstride, int ldp, long u_off, int S,
                                 int n, __half* h, int ldh, const float* row_w, int ldw, int seg,
                                 const int* n_dev, cudaStream_t st);

// MoE routing (top_k of E per row, ties to the lower id, softmax over the
// selection) and grouping (per-expert row lists by counting sort, the ascending
// list of hit experts, a dense [S][n_cap] routing-weight table by hit slot).
cudaError_t launch_moe_route(const float* logits, int S, int E, int top_k, int32_t* ids, float* w,
                             int32_t* offsets, int32_t* pair_rows, int32_t* n_hit, int32_t* hit,
                             float* row_w, int n_cap, cudaStream_t st);

cudaError_t launch_quantize(const float* w, int n, int k, int qbits, void* codes, uint16_t* scales,
                            cudaStream_t st);
cudaError_t launch_tree_accept(const int32_t* argmax, int S, const int32_t* tokens, const int32_t* parent,
                               int32_t* path, int32_t* accepted, int32_t* next_a0, cudaStream_t st);
// The split-reduction head's tail: logits = sum over splits of part[split][s][v]
// (written when logits is not null), argmax per row, accept; grid CTAs of per-row
// partials part_v/part_i [grid][S]; the last CTA resets *ticket.
int head_splitsum_grid(int n, int sms);
cudaError_t launch_head_splitsum(const float* part, int splits, int S, int n, float* logits, float* part_v,
                                 int* part_i, const int32_t* drafts, int n_valid, int32_t* argmax, int32_t* accepted,
                                 int32_t* next_a0, unsigned* ticket, int grid, cudaStream_t st);
cudaError_t launch_greedy_accept(const int32_t* argmax, int S, const int32_t* drafts, int n_valid,
                                 int32_t* accepted, int32_t* next_a0, cudaStream_t st);

}  // namespace sdv
