// C ABI of libsdv (declared in include/sdv.h): argument validation, TMA
// descriptor encoding, launch configuration and workspace layout.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include "sdv.h"
#include "sdv_device.cuh"
#include "sdv_kernels.h"

namespace {

using sdv::GemmArgs;

constexpr size_t kWsHeader = 256;  // status word, ticket counter, reserved
constexpr int kMaxExperts = 1024;  // MoE routing: one block of 1024 threads
constexpr int kMaxTopK = 32;
constexpr int kMaxS = 32;
constexpr int kMaxDepth = 8;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

sdv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SDV_OK : SDV_ERR_CUDA; }

// cuTensorMapEncodeTiled, fetched from the driver once (no link-time libcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

int device_smem_optin() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
  return v;
}

// Shape of a [n, k] weight the launch plans accept: k a positive multiple of 32
// and both small enough that tile-count roundings stay inside int32.
constexpr int32_t kMaxDim = INT32_MAX - 1024;
bool valid_shape(int32_t n, int32_t k) { return n >= 1 && n <= kMaxDim && k >= 32 && k <= kMaxDim && k % 32 == 0; }

bool valid_weight(const sdv_qweight* w) {
  if (w == nullptr || w->codes == nullptr || w->scales == nullptr) return false;
  if (w->qtype != SDV_Q8 && w->qtype != SDV_Q4 && w->qtype != SDV_F4) return false;
  if (!valid_shape(w->n, w->k)) return false;
  if (!aligned16(w->codes) || !aligned16(w->scales)) return false;
  return true;
}

// Codes: uint8 [n][row_bytes], box 128 bytes x code_rows rows, 128-byte swizzle.
// Scales: fp16 [n][k/32], box 8 x sc_rows rows (only when k % 256 == 0).
sdv_status encode_maps(const sdv_qweight* w, int code_rows, int sc_rows, CUtensorMap* tc, CUtensorMap* tsc,
                       int* scales_tma) {
  auto enc = encode_fn();
  if (enc == nullptr) return SDV_ERR_CUDA;
  const uint64_t row_bytes = (w->qtype == SDV_Q8) ? (uint64_t)w->k : (uint64_t)w->k / 2;
  {
    cuuint64_t dims[2] = {row_bytes, (cuuint64_t)w->n};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {128, (cuuint32_t)code_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(tc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(w->codes), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return SDV_ERR_CUDA;
  }
  *scales_tma = (w->k % 256) == 0 ? 1 : 0;
  std::memset(tsc, 0, sizeof(*tsc));
  if (*scales_tma) {
    cuuint64_t dims[2] = {(cuuint64_t)(w->k / 32), (cuuint64_t)w->n};
    cuuint64_t strides[1] = {(cuuint64_t)(w->k / 32) * 2};
    cuuint32_t box[2] = {8, (cuuint32_t)sc_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(tsc, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t*>(w->scales), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return SDV_ERR_CUDA;
  }
  return SDV_OK;
}

// Largest ring depth whose shared-memory plan fits; 0 if none >= 2 does.
int pick_depth(int qbits, int S, int k_len, int* smem) {
  const int limit = device_smem_optin();
  for (int d = kMaxDepth; d >= 2; --d) {
    const int b = sdv::gemm_smem_bytes(qbits, S, k_len, d);
    if (b <= limit) {
      *smem = b;
      return d;
    }
  }
  return 0;
}

struct GemmPlan {
  int splits = 0, k_chunk = 0, depth = 0, smem = 0, grid = 0;
  bool tc = false;  // tcgen05 path
};

// Launch plan of the weight-streaming GEMM.  Without split-K (the verify head,
// whose argmax needs complete logits) one CTA per SM covers the full reduction.
// With split-K the reduction is cut into 256-multiples until every warp has a
// few 16-row tiles and the window rows of one split fit in shared memory.
GemmPlan plan_gemm(int qbits, int n, int k, int S, bool allow_split) {
  GemmPlan pl;
  const int sms = device_sms();
  if (sms <= 0) return pl;
  const int tiles = (n + 15) / 16;
  const int warps_total = sms * sdv::gemm_warps_per_cta();
  const int kst = (k + 255) / 256;
  int want = 1;  // requested splits; rounding the chunk to 256 may give fewer
  if (allow_split) {
    want = (4 * warps_total + tiles - 1) / tiles;
    if (want > kst) want = kst;
    if (want < 1) want = 1;
  }
  for (;; ++want) {
    int k_chunk = k, splits = 1;
    if (want > 1) {
      k_chunk = ((k + want - 1) / want + 255) / 256 * 256;
      splits = (k + k_chunk - 1) / k_chunk;
    }
    int smem = 0;
    const int depth = pick_depth(qbits, S, k_chunk, &smem);
    if (depth >= 3 || (depth == 2 && (!allow_split || splits >= kst))) {
      pl.splits = splits;
      pl.k_chunk = k_chunk;
      pl.depth = depth;
      pl.smem = smem;
      int grid = (tiles + sdv::gemm_warps_per_cta() - 1) / sdv::gemm_warps_per_cta();
      const int per_split = (sms + splits - 1) / splits;
      if (grid > per_split) grid = per_split;
      pl.grid = grid < 1 ? 1 : grid;
      return pl;
    }
    if (!allow_split || want >= kst) return GemmPlan{};
  }
}

// GEMM implementation: 0 = choose (tcgen05 when its plan fits), 1 = the
// mma.sync path, 2 = the tcgen05 path only, 3 = the CUDA-core GEMV for windows
// of one or two rows (else as 0).
std::atomic<int> g_gemm_path{0};

// Timeout-path test hooks (sdv_debug_fault): applied to every tcgen05 launch.
std::atomic<unsigned long long> g_debug_wait_ns{0};
std::atomic<int> g_debug_withhold{0};
std::atomic<uint64_t> g_launches{0};  // kernels launched by this library (sdv_launch_count)

void apply_debug(GemmArgs& a) {
  a.wait_ns = g_debug_wait_ns.load();
  a.debug_withhold = g_debug_withhold.load();
}

// tcgen05 path plan: 128-row tiles, at most one CTA per SM.  Without split-K
// (the verify head, the MoE gate/up) one split covers the full reduction.
// With split-K every split count whose window rows fit next to a ring of at
// least four stages is costed in bytes at the HBM rate: the busiest CTA's weight
// stages (a stage is one 128 x 256 code tile; every SM streams at the same rate)
// plus the split partials' write and read-back; the cheapest wins, ties to fewer
// splits.  `unit` tiles move together (2: the gate/up pairs of the fused SwiGLU).
GemmPlan plan_tc(int qbits, int n, int k, int S, bool allow_split, int unit = 1, bool route = false) {
  GemmPlan best;
  const int sms = device_sms();
  const int limit = device_smem_optin();
  if (sms <= 0 || limit <= 0) return best;
  const int tiles = (n + 127) / 128;
  const int units = tiles / unit > 0 ? tiles / unit : 1;
  const int kst = (k + 255) / 256;
  const long long stage_bytes = 128LL * 128 * (qbits == 8 ? 2 : 1);
  long long best_cost = 0;
  for (int want = 1; want <= (allow_split ? kst : 1); ++want) {
    const int stages = (kst + want - 1) / want;  // per split
    const int k_chunk = want > 1 ? stages * 256 : k;
    const int splits = (k + k_chunk - 1) / k_chunk;
    if (splits != want) continue;  // the same chunk as a smaller split count
    int depth = 0, bytes = 0;
    for (int d = kMaxDepth; d >= 4 && depth == 0; --d) {  // tc_plan_valid rejects shallower rings
      const int b = sdv::tc_smem_bytes(qbits, S, k_chunk, d, route);
      if (b <= limit && sdv::tc_plan_valid(qbits, S, k_chunk, d)) {
        depth = d;
        bytes = b;
      }
    }
    if (depth == 0) continue;
    int grid = sms / splits;  // one wave: at most one CTA per SM over all splits
    if (grid > units) grid = units;
    if (grid < 1) continue;
    const long long busiest = (long long)((units + grid - 1) / grid) * unit * stages;
    const long long cost = busiest * stage_bytes * sms + (splits > 1 ? 2LL * splits * S * n * 4 : 0);
    if (best.splits != 0 && cost >= best_cost) continue;
    best_cost = cost;
    best.splits = splits;
    best.k_chunk = k_chunk;
    best.depth = depth;
    // at least half the SM's shared memory: one CTA (one 512-column tensor
    // memory allocation) per SM
    best.smem = bytes > limit / 2 + 1024 ? bytes : limit / 2 + 1024;
    best.grid = grid;
    best.tc = true;
  }
  return best;
}

GemmPlan choose_plan(int qbits, int n, int k, int S, bool allow_split) {
  const int path = g_gemm_path.load();
  if (qbits == SDV_F4)  // FP4 weights exist on the tcgen05 path only
    return path == 1 ? GemmPlan{} : plan_tc(qbits, n, k, S, allow_split);
  if (path != 1) {
    const GemmPlan t = plan_tc(qbits, n, k, S, allow_split);
    if (t.splits != 0 || path == 2) return t;
  }
  return plan_gemm(qbits, n, k, S, allow_split);
}

size_t head_ws_bytes(int S) {
  const int sms = device_sms();
  return kWsHeader + (size_t)(sms > 0 ? sms : 1024) * (size_t)S * 8;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// Verify head whose window rows fit the tcgen05 plan only with the reduction
// split (e.g. k = 2560 at S >= 17): plan of the split pass (splits >= 2), or
// splits == 0 where the whole-window plan fits or no split plan does.
GemmPlan plan_head_split(int qbits, int n, int k, int S) {
  if (S < 2 || g_gemm_path.load() == 1) return GemmPlan{};
  if (plan_tc(qbits, n, k, S, false).splits != 0) return GemmPlan{};
  const GemmPlan pl = plan_tc(qbits, n, k, S, true);
  return pl.splits >= 2 ? pl : GemmPlan{};
}

// Its workspace: header, fp32 partial logits [splits][S][n], then the tail's
// per-CTA (max, index) partials [grid][S] of each kind.
size_t head_split_ws_bytes(const GemmPlan& pl, int n, int S) {
  const int grid = sdv::head_splitsum_grid(n, device_sms());
  return kWsHeader + align256((size_t)pl.splits * S * n * sizeof(float)) + align256((size_t)grid * S * 4) * 2;
}

// [grid][S][8] floats of per-CTA sampling partials behind the header
size_t sample_ws_bytes(int S) {
  const int sms = device_sms();
  return kWsHeader + (size_t)(sms > 0 ? sms : 1024) * (size_t)S * 32;
}

size_t qlinear_ws_bytes(int qbits, int n, int k, int S) {
  size_t need = kWsHeader;
  for (const GemmPlan& pl : {plan_gemm(qbits, n, k, S, true), plan_tc(qbits, n, k, S, true)}) {
    if (pl.splits > 1) {
      const size_t b = kWsHeader + (size_t)pl.splits * S * n * sizeof(float);
      if (b > need) need = b;
    }
  }
  return need;
}

// Common part of the weight-streaming GEMM launches.  For kModeY the output
// `y_final` receives Y (through split-K partials in ws when the plan splits).
// Split-K partials go to part_area when given (part_bytes long), else behind
// the workspace header.
sdv_status run_gemm(const sdv_qweight* w, const uint16_t* x, int S, int mode, GemmArgs& a, void* ws,
                    size_t ws_bytes, float* y_final, cudaStream_t st, char* part_area = nullptr,
                    size_t part_bytes = 0) {
  if (g_gemm_path.load() == 3 && (mode == sdv::kModeY || mode == sdv::kModeHead)) {
    const int g = sdv::gemv_plan(w->qtype, w->k, S);
    const int sms = device_sms();
    if (g > 0 && sms > 0) {
      // the CUDA-core GEMV: one pass, no split; head partials as for the GEMM
      a.codes = w->codes;
      a.x = reinterpret_cast<const __half*>(x);
      a.scales = w->scales;
      a.S = S;
      a.N = w->n;
      a.K = w->k;
      a.status = static_cast<int*>(ws);
      a.ticket = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + 4);
      if (mode == sdv::kModeY) a.y = y_final;
      a.part_v = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader);
      a.part_i = reinterpret_cast<int*>(static_cast<char*>(ws) + kWsHeader + (size_t)sms * S * 4);
      return cuda_status(sdv::launch_gemv(w->qtype, mode, a, g, sms, st));
    }
  }
  const GemmPlan pl = choose_plan(w->qtype, w->n, w->k, S, mode == sdv::kModeY);
  if (pl.splits == 0) return SDV_ERR_UNSUPPORTED;
  if (mode == sdv::kModeHead) {
    a.part_v = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader);
    a.part_i = reinterpret_cast<int*>(static_cast<char*>(ws) + kWsHeader + (size_t)pl.grid * S * 4);
  }
  if (mode == sdv::kModeSample) {
    if (!pl.tc) return SDV_ERR_UNSUPPORTED;  // the sampling epilogue exists on the tcgen05 path only
    a.part_s = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader);
  }
  CUtensorMap tc, tsc;
  int scales_tma = 0;
  // box heights: the tcgen05 path moves whole 128-row tiles, the mma.sync path
  // 16-row tiles (scales for its MT tiles at once)
  const int code_rows = pl.tc ? 128 : 16;
  const int sc_rows = pl.tc ? 128 : 16 * sdv::gemm_tile_mt(w->qtype);
  sdv_status s = encode_maps(w, code_rows, sc_rows, &tc, &tsc, &scales_tma);
  if (s != SDV_OK) return s;
  a.x = reinterpret_cast<const __half*>(x);
  a.scales = w->scales;
  a.S = S;
  a.N = w->n;
  a.K = w->k;
  a.k_chunk = pl.k_chunk;
  a.splits = pl.splits;
  a.m16_tiles = (w->n + 15) / 16;
  a.depth = pl.depth;
  a.scales_tma = scales_tma;
  a.status = static_cast<int*>(ws);
  a.ticket = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + 4);
  float* part = nullptr;
  if (mode == sdv::kModeY) {
    if (pl.splits > 1) {
      const size_t pbytes = (size_t)pl.splits * S * w->n * sizeof(float);
      if (part_area != nullptr) {
        if (part_bytes < pbytes) return SDV_ERR_WORKSPACE;
        part = reinterpret_cast<float*>(part_area);
      } else {
        if (ws_bytes < kWsHeader + pbytes) return SDV_ERR_WORKSPACE;
        part = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader);
      }
      a.y = part;
    } else {
      a.y = y_final;
    }
  }
  if (pl.tc) apply_debug(a);
  cudaError_t e = pl.tc ? sdv::launch_tc_gemm(w->qtype, mode, tc, tsc, tc, tsc, a, pl.grid, pl.smem, st)
                        : sdv::launch_dq_gemm(w->qtype, mode, tc, tsc, a, pl.grid, pl.smem, st);
  if (e == cudaSuccess && part != nullptr)
    e = sdv::launch_splitk_reduce(part, pl.splits, (long)S * w->n, y_final, st);
  return cuda_status(e);
}

sdv_status run_gemm_ws(const sdv_qweight* w, const uint16_t* x, int S, GemmArgs& a, void* ws, char* part_area,
                       size_t part_bytes, float* y, cudaStream_t st) {
  return run_gemm(w, x, S, sdv::kModeY, a, ws, kWsHeader, y, st, part_area, part_bytes);
}

// One tcgen05 GEMM in Y mode over w (and w2 when dual): fills the launch fields of
// `a` from the plan and the weights; the mapping fields are the caller's.
sdv_status launch_tc_y(const sdv_qweight* w, const sdv_qweight* w2, const GemmPlan& pl, GemmArgs& a,
                       void* ws, cudaStream_t st) {
  CUtensorMap tc, tsc, tc2, tsc2;
  int sc_tma = 0, sc_tma2 = 0;
  sdv_status s = encode_maps(w, 128, 128, &tc, &tsc, &sc_tma);
  if (s != SDV_OK) return s;
  if (w2 != nullptr) {
    s = encode_maps(w2, 128, 128, &tc2, &tsc2, &sc_tma2);
    if (s != SDV_OK) return s;
    if (sc_tma2 != sc_tma) return SDV_ERR_UNSUPPORTED;
  } else {
    tc2 = tc;
    tsc2 = tsc;
  }
  a.scales = w->scales;
  a.scales_tma = sc_tma;
  a.k_chunk = pl.k_chunk;
  a.splits = pl.splits;
  a.m16_tiles = 0;
  a.depth = pl.depth;
  a.status = static_cast<int*>(ws);
  a.ticket = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + 4);
  apply_debug(a);
  return cuda_status(sdv::launch_tc_gemm(w->qtype, sdv::kModeY, tc, tsc, tc2, tsc2, a, pl.grid, pl.smem, st));
}

// Fused SwiGLU gate/up: one tcgen05 launch over both matrices (dual tiles,
// split-K when the window rows of the full reduction do not fit), fp32 partials
// [splits][S][2n] in the workspace, then the reduce that applies SwiGLU.
GemmPlan plan_swiglu(int qbits, int n, int k, int S) {
  if (k % 256 != 0) return GemmPlan{};
  return plan_tc(qbits, 2 * n, k, S, true, 2);
}

size_t swiglu_ws_bytes(int qbits, int n, int k, int S) {
  const GemmPlan t = plan_swiglu(qbits, n, k, S);
  size_t b = kWsHeader + (size_t)2 * S * n * sizeof(float);  // the two-GEMM form: g, u
  if (t.splits > 0) {
    const size_t bt = kWsHeader + (size_t)t.splits * S * 2 * n * sizeof(float);
    if (bt > b) b = bt;
  }
  // the two-GEMM form also holds each GEMM's split-K partials behind g and u
  const size_t q = qlinear_ws_bytes(qbits, n, k, S);
  return b + q;
}

// Gathered-expert MoE workspace layout (all offsets 256-aligned).
struct MoeLayout {
  int n_cap = 0;       // most experts a window can hit: min(E, S * top_k)
  bool route = false;  // the gate/up launch routes the window itself (no routing launch)
  int gx = 0, ys = 0;  // down projection: CTAs per split, splits (expert-segment slots)
  GemmPlan gu, dn;     // gate/up and down launch plans
  size_t ids, w, offsets, pair_rows, n_hit, hit, row_w, hbuf, dn_part, total;
};

MoeLayout plan_moe(int qbits, int E, int I, int H, int top_k, int S) {
  MoeLayout L;
  const int sms = device_sms();
  const int limit = device_smem_optin();
  if (sms <= 0 || limit <= 0) return L;
  L.n_cap = E < S * top_k ? E : S * top_k;
  // gate/up: both matrices of the hit experts, full reduction H, no split; it
  // routes the window in its prologue where the routing fits its limits and
  // shared memory, else a routing launch runs first
  if (E <= sdv::kRouteMaxE && top_k <= sdv::kRouteMaxTopK && S <= sdv::kRouteMaxS) {
    L.gu = plan_tc(qbits, 2 * L.n_cap * I, H, S, false, 1, true);
    L.route = L.gu.splits == 1;
  }
  if (!L.route) L.gu = plan_tc(qbits, 2 * L.n_cap * I, H, S, false);
  if (L.gu.splits != 1) return MoeLayout{};
  L.gu.grid = sms;
  // down: the reduction is the hit experts' I-column segments; gx CTAs share one
  // split (expert-segment slot) and cover the H rows between them
  const int tiles = (H + 127) / 128;
  for (int gx : {4, 2, 1}) {
    if (gx > tiles) continue;
    const int ys = sms / gx;
    if (ys < 1) continue;
    const int segs = (L.n_cap + ys - 1) / ys;
    const int k_chunk = segs * I;
    for (int d = kMaxDepth; d >= 4; --d) {  // tc_plan_valid rejects shallower rings
      const int b = sdv::tc_smem_bytes(qbits, S, k_chunk, d);
      if (b <= limit && sdv::tc_plan_valid(qbits, S, k_chunk, d)) {
        L.dn.splits = ys;
        L.dn.k_chunk = k_chunk;
        L.dn.depth = d;
        L.dn.smem = b > limit / 2 + 1024 ? b : limit / 2 + 1024;
        L.dn.grid = gx;
        L.dn.tc = true;
        L.gx = gx;
        L.ys = ys;
        break;
      }
    }
    if (L.ys > 0) break;
  }
  if (L.ys == 0) return MoeLayout{};
  size_t o = kWsHeader;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L.ids = take((size_t)S * top_k * 4);
  L.w = take((size_t)S * top_k * 4);
  L.offsets = take((size_t)(E + 1) * 4);
  L.pair_rows = take((size_t)S * top_k * 4);
  L.n_hit = take(4);
  L.hit = take((size_t)E * 4);
  L.row_w = take((size_t)S * L.n_cap * 4);
  L.hbuf = take((size_t)S * L.n_cap * I * 2);
  L.dn_part = take((size_t)L.ys * S * H * 4);
  L.total = o;
  return L;
}

bool moe_args_ok(const sdv_qweight* gate, const sdv_qweight* up, const sdv_qweight* down, int E, int I, int H,
                 int top_k) {
  if (!valid_weight(gate) || !valid_weight(up) || !valid_weight(down)) return false;
  if (E < 1 || I < 32 || H < 32 || top_k < 1 || top_k > E) return false;
  if (gate->qtype != up->qtype || gate->qtype != down->qtype) return false;
  const long long ei = (long long)E * I, eh = (long long)E * H;
  if (gate->n != ei || up->n != ei || gate->k != H || up->k != H) return false;
  if (down->n != eh || down->k != I) return false;
  return true;
}

}  // namespace

namespace sdv {
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace sdv

extern "C" {

int32_t sdv_version(void) { return 100; }

sdv_status sdv_debug_fault(int32_t withhold_stage, uint64_t wait_limit_ns) {
  if (withhold_stage < -1 || (wait_limit_ns != 0 && wait_limit_ns < 100000ull)) return SDV_ERR_INVALID_ARG;
  g_debug_withhold.store(withhold_stage < 0 ? 0 : withhold_stage + 1);
  g_debug_wait_ns.store(wait_limit_ns);
  return SDV_OK;
}

uint64_t sdv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int32_t sdv_set_gemm_path(int32_t path) {
  if (path < 0 || path > 3) return -1;
  return g_gemm_path.exchange(path);
}

const char* sdv_status_string(sdv_status s) {
  switch (s) {
    case SDV_OK: return "SDV_OK";
    case SDV_ERR_INVALID_ARG: return "SDV_ERR_INVALID_ARG";
    case SDV_ERR_UNSUPPORTED: return "SDV_ERR_UNSUPPORTED";
    case SDV_ERR_CUDA: return "SDV_ERR_CUDA";
    case SDV_ERR_TIMEOUT: return "SDV_ERR_TIMEOUT";
    case SDV_ERR_WORKSPACE: return "SDV_ERR_WORKSPACE";
  }
  return "SDV_ERR_UNKNOWN";
}

size_t sdv_workspace_bytes(int32_t op, int32_t n, int32_t k, int32_t S, int32_t E, int32_t top_k) {
  if (S < 1 || S > kMaxS) return 0;
  // n, k: the weight's [n, k] (for the MoE op, I and H of one expert)
  if (!valid_shape(n, k)) return 0;
  switch (op) {
    case SDV_OP_QLINEAR: {  // the larger of the two weight types' plans
      const size_t a = qlinear_ws_bytes(8, n, k, S), b = qlinear_ws_bytes(4, n, k, S);
      return a > b ? a : b;
    }
    case SDV_OP_QLINEAR_SWIGLU: {
      const size_t a = swiglu_ws_bytes(8, n, k, S), b = swiglu_ws_bytes(4, n, k, S);
      return a > b ? a : b;
    }
    case SDV_OP_VERIFY_HEAD: {  // the larger of the weight types' split plans, if any
      size_t b = head_ws_bytes(S);
      for (int q : {8, 4}) {
        const GemmPlan pl = plan_head_split(q, n, k, S);
        if (pl.splits >= 2) {
          const size_t bs = head_split_ws_bytes(pl, n, S);
          if (bs > b) b = bs;
        }
      }
      return b;
    }
    case SDV_OP_VERIFY_SAMPLE: return sample_ws_bytes(S);
    case SDV_OP_MOE: {  // n = I, k = H
      if (E < 1 || top_k < 1 || top_k > E) return 0;
      const MoeLayout a = plan_moe(8, E, n, k, top_k, S), b = plan_moe(4, E, n, k, top_k, S);
      return a.total > b.total ? a.total : b.total;
    }
  }
  return 0;
}

sdv_status sdv_workspace_init(void* ws, size_t ws_bytes, sdv_stream_t stream) {
  if (ws == nullptr || ws_bytes < kWsHeader) return SDV_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

sdv_status sdv_last_device_status(void* ws, sdv_stream_t stream) {
  if (ws == nullptr) return SDV_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return SDV_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SDV_ERR_CUDA;
  if (word == 0) return SDV_OK;
  const int zero = 0;
  if (cudaMemcpy(ws, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return SDV_ERR_CUDA;
  return (word & sdv::kDevErrTimeout) ? SDV_ERR_TIMEOUT : SDV_ERR_CUDA;
}

sdv_status sdv_device_status(void* ws, sdv_stream_t stream) { return sdv_last_device_status(ws, stream); }

sdv_status sdv_quantize_block32(const float* w, int32_t n, int32_t k, int32_t qtype, void* codes,
                                uint16_t* scales, sdv_stream_t stream) {
  if (w == nullptr || codes == nullptr || scales == nullptr) return SDV_ERR_INVALID_ARG;
  if (n < 1 || k < 32 || (k % 32) != 0) return SDV_ERR_INVALID_ARG;
  if (qtype != SDV_Q8 && qtype != SDV_Q4 && qtype != SDV_F4) return SDV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w) & 3u) || (reinterpret_cast<uintptr_t>(scales) & 1u))
    return SDV_ERR_INVALID_ARG;
  return cuda_status(sdv::launch_quantize(w, n, k, qtype, codes, scales,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

sdv_status sdv_qlinear(const sdv_qweight* w, const uint16_t* x, int32_t S, float* y, void* ws,
                       size_t ws_bytes, sdv_stream_t stream) {
  if (!valid_weight(w) || x == nullptr || y == nullptr || !aligned16(x)) return SDV_ERR_INVALID_ARG;
  if (S < 1) return SDV_ERR_INVALID_ARG;
  if (S > kMaxS) return SDV_ERR_UNSUPPORTED;
  if (ws == nullptr || !aligned16(ws) || ws_bytes < kWsHeader) return SDV_ERR_WORKSPACE;
  GemmArgs a{};
  return run_gemm(w, x, S, sdv::kModeY, a, ws, ws_bytes, y, reinterpret_cast<cudaStream_t>(stream));
}

sdv_status sdv_verify_sample(const sdv_qweight* head, const uint16_t* x, int32_t S, const int32_t* drafts,
                             int32_t n_valid, float temperature, uint64_t seed, uint64_t counter,
                             float* logits_or_null, int32_t* samples, int32_t* accepted, int32_t* next_token,
                             void* ws, size_t ws_bytes, sdv_stream_t stream) {
  if (!valid_weight(head) || x == nullptr || !aligned16(x)) return SDV_ERR_INVALID_ARG;
  if (samples == nullptr || accepted == nullptr || next_token == nullptr) return SDV_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !(temperature < INFINITY)) return SDV_ERR_INVALID_ARG;
  if (S < 1) return SDV_ERR_INVALID_ARG;
  if (S > kMaxS) return SDV_ERR_UNSUPPORTED;
  if (n_valid < 0 || n_valid > S - 1) return SDV_ERR_INVALID_ARG;
  if (n_valid > 0 && drafts == nullptr) return SDV_ERR_INVALID_ARG;
  const size_t need = sdv_workspace_bytes(SDV_OP_VERIFY_SAMPLE, head->n, head->k, S, 0, 0);
  if (ws == nullptr || !aligned16(ws) || ws_bytes < need) return SDV_ERR_WORKSPACE;
  const int path = g_gemm_path.load();
  if (path == 1) return SDV_ERR_UNSUPPORTED;
  GemmArgs a{};
  a.y = logits_or_null;
  a.drafts = drafts;
  a.n_valid = n_valid;
  a.argmax = samples;
  a.accepted = accepted;
  a.next_a0 = next_token;
  a.inv_temp = 1.f / temperature;
  a.rng_key = sdv::splitmix_mix(seed + (counter + 1ull) * sdv::kSplitMixG);
  return run_gemm(head, x, S, sdv::kModeSample, a, ws, ws_bytes, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

sdv_status sdv_verify_head(const sdv_qweight* head, const uint16_t* x, int32_t S, const int32_t* drafts,
                           int32_t n_valid, float* logits_or_null, int32_t* argmax, int32_t* accepted,
                           int32_t* next_a0, void* ws, size_t ws_bytes, sdv_stream_t stream) {
  if (!valid_weight(head) || x == nullptr || !aligned16(x)) return SDV_ERR_INVALID_ARG;
  if (argmax == nullptr || accepted == nullptr || next_a0 == nullptr) return SDV_ERR_INVALID_ARG;
  if (S < 1) return SDV_ERR_INVALID_ARG;
  if (S > kMaxS) return SDV_ERR_UNSUPPORTED;
  if (n_valid < 0 || n_valid > S - 1) return SDV_ERR_INVALID_ARG;
  if (n_valid > 0 && drafts == nullptr) return SDV_ERR_INVALID_ARG;
  // the least a head call needs (the row-chunked form below); the split form
  // needs more and runs when the workspace is large enough for it
  if (ws == nullptr || !aligned16(ws) || ws_bytes < head_ws_bytes(S)) return SDV_ERR_WORKSPACE;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  {
    // The window rows of a long reduction may not fit one tcgen05 launch next
    // to its ring.  Then each CTA takes half (or a smaller share) of the
    // reduction, whose rows fit: one pass over the head writes fp32 partial
    // logits (a few % of the weight bytes), and the split-sum tail adds them in
    // order, takes the argmax and runs the accept.
    const GemmPlan sp = plan_head_split(head->qtype, head->n, head->k, S);
    if (sp.splits >= 2 && ws_bytes >= head_split_ws_bytes(sp, head->n, S)) {
      char* const w8 = static_cast<char*>(ws);
      float* const part = reinterpret_cast<float*>(w8 + kWsHeader);
      const int grid = sdv::head_splitsum_grid(head->n, device_sms());
      const size_t pbytes = align256((size_t)sp.splits * S * head->n * sizeof(float));
      float* const pv = reinterpret_cast<float*>(w8 + kWsHeader + pbytes);
      int* const pi = reinterpret_cast<int*>(w8 + kWsHeader + pbytes + align256((size_t)grid * S * 4));
      GemmArgs a{};
      a.x = reinterpret_cast<const __half*>(x);
      a.S = S;
      a.N = head->n;
      a.K = head->k;
      a.y = part;
      sdv_status s = launch_tc_y(head, nullptr, sp, a, ws, st);
      if (s != SDV_OK) return s;
      return cuda_status(sdv::launch_head_splitsum(part, sp.splits, S, head->n, logits_or_null, pv, pi, drafts,
                                                   n_valid, argmax, accepted, next_a0,
                                                   reinterpret_cast<unsigned*>(w8 + 4), grid, st));
    }
  }
  GemmArgs a{};
  a.y = logits_or_null;
  a.drafts = drafts;
  a.n_valid = n_valid;
  a.argmax = argmax;
  a.accepted = accepted;
  a.next_a0 = next_a0;
  // The window rows of a long reduction may not fit one tcgen05 launch's shared
  // memory next to its ring.  Two row chunks on the tcgen05 path (each streams
  // the head once) then beat one launch of the mma.sync path, which streams at
  // well under half the rate (q4b head, S = 17: 145 us against 209 us).
  const int path = g_gemm_path.load();
  int chunk = 0;
  if (path != 1 && S > 1 && plan_tc(head->qtype, head->n, head->k, S, false).splits == 0 &&
      plan_tc(head->qtype, head->n, head->k, (S + 1) / 2, false).splits != 0)
    chunk = (S + 1) / 2;
  if (chunk == 0) {
    const sdv_status s = run_gemm(head, x, S, sdv::kModeHead, a, ws, ws_bytes, nullptr, st);
    if (s != SDV_ERR_UNSUPPORTED || S == 1) return s;
    // neither path fits the whole window: the largest halving that does
    chunk = S / 2;
    while (chunk > 1 && choose_plan(head->qtype, head->n, head->k, chunk, false).splits == 0) chunk /= 2;
    if (choose_plan(head->qtype, head->n, head->k, chunk, false).splits == 0) return SDV_ERR_UNSUPPORTED;
  }
  // verify the rows in chunks, then run the accept over the whole argmax
  for (int r0 = 0; r0 < S; r0 += chunk) {
    const int rows = S - r0 < chunk ? S - r0 : chunk;
    GemmArgs b{};
    b.y = logits_or_null != nullptr ? logits_or_null + (size_t)r0 * head->n : nullptr;
    b.drafts = nullptr;
    b.n_valid = 0;
    b.argmax = argmax + r0;
    b.accepted = accepted;  // overwritten by the accept below
    b.next_a0 = next_a0;
    const sdv_status c = run_gemm(head, x + (size_t)r0 * head->k, rows, sdv::kModeHead, b, ws, ws_bytes, nullptr, st);
    if (c != SDV_OK) return c;
  }
  return cuda_status(sdv::launch_greedy_accept(argmax, S, drafts, n_valid, accepted, next_a0, st));
}

sdv_status sdv_tree_accept(const int32_t* argmax, int32_t S, const int32_t* tokens, const int32_t* parent,
                           int32_t* path, int32_t* accepted, int32_t* next_a0, sdv_stream_t stream) {
  if (argmax == nullptr || accepted == nullptr || next_a0 == nullptr) return SDV_ERR_INVALID_ARG;
  if (S < 1) return SDV_ERR_INVALID_ARG;
  if (S > kMaxS) return SDV_ERR_UNSUPPORTED;
  if (S > 1 && (tokens == nullptr || parent == nullptr || path == nullptr)) return SDV_ERR_INVALID_ARG;
  return cuda_status(sdv::launch_tree_accept(argmax, S, tokens, parent, path, accepted, next_a0,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

sdv_status sdv_greedy_accept(const int32_t* argmax, int32_t S, const int32_t* drafts, int32_t n_valid,
                             int32_t* accepted, int32_t* next_a0, sdv_stream_t stream) {
  if (argmax == nullptr || accepted == nullptr || next_a0 == nullptr) return SDV_ERR_INVALID_ARG;
  if (S < 1 || n_valid < 0 || n_valid > S - 1) return SDV_ERR_INVALID_ARG;
  if (n_valid > 0 && drafts == nullptr) return SDV_ERR_INVALID_ARG;
  return cuda_status(sdv::launch_greedy_accept(argmax, S, drafts, n_valid, accepted, next_a0,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

sdv_status sdv_qlinear_swiglu(const sdv_qweight* gate, const sdv_qweight* up, const uint16_t* x,
                              int32_t S, uint16_t* h, void* ws, size_t ws_bytes, sdv_stream_t stream) {
  if (!valid_weight(gate) || !valid_weight(up) || x == nullptr || h == nullptr || !aligned16(x))
    return SDV_ERR_INVALID_ARG;
  if (gate->qtype != up->qtype || gate->n != up->n || gate->k != up->k) return SDV_ERR_INVALID_ARG;
  if (S < 1) return SDV_ERR_INVALID_ARG;
  if (S > kMaxS) return SDV_ERR_UNSUPPORTED;
  const int n = gate->n, k = gate->k;
  const size_t need = swiglu_ws_bytes(gate->qtype, n, k, S);
  if (ws == nullptr || !aligned16(ws) || ws_bytes < need) return SDV_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  __half* const hh = reinterpret_cast<__half*>(h);
  float* const part = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader);
  const GemmPlan pl = g_gemm_path.load() == 1 ? GemmPlan{} : plan_swiglu(gate->qtype, n, k, S);
  if (pl.splits > 0) {
    GemmArgs a{};
    a.x = reinterpret_cast<const __half*>(x);
    a.S = S;
    a.N = n;
    a.K = k;
    if (pl.splits == 1) {  // SwiGLU in the GEMM epilogue
      a.dual = 2;
      a.h = hh;
      a.ldh = n;
      return launch_tc_y(gate, up, pl, a, ws, st);
    }
    a.ldy = 2 * n;
    a.dual = 1;
    a.y = part;
    sdv_status s = launch_tc_y(gate, up, pl, a, ws, st);
    if (s != SDV_OK) return s;
    return cuda_status(sdv::launch_swiglu_reduce(part, pl.splits, (long)S * 2 * n, 2 * n, n, S, n, hh, n,
                                                 nullptr, 0, 1, nullptr, st));
  }
  // two GEMMs (g then u, each [S][n] fp32 behind the header), then the SwiGLU reduce;
  // each GEMM's split-K partials live behind g and u
  float* const g = part;
  float* const u = part + (size_t)S * n;
  char* const ws2 = reinterpret_cast<char*>(u + (size_t)S * n);
  const size_t ws2_bytes = ws_bytes - (size_t)(ws2 - static_cast<char*>(ws));
  for (int m = 0; m < 2; ++m) {
    GemmArgs a{};
    sdv_status s = run_gemm_ws(m == 0 ? gate : up, x, S, a, ws, ws2, ws2_bytes, m == 0 ? g : u, st);
    if (s != SDV_OK) return s;
  }
  return cuda_status(sdv::launch_swiglu_reduce(part, 1, 0, n, (long)S * n, S, n, hh, n, nullptr, 0, 1, nullptr, st));
}

sdv_status sdv_moe_route(const float* router_logits, int32_t S, int32_t E, int32_t top_k, int32_t* ids,
                         float* weights, int32_t* offsets, int32_t* pair_rows, int32_t* n_hit, int32_t* hit,
                         sdv_stream_t stream) {
  if (router_logits == nullptr || ids == nullptr || weights == nullptr || offsets == nullptr ||
      pair_rows == nullptr || n_hit == nullptr || hit == nullptr)
    return SDV_ERR_INVALID_ARG;
  if (S < 1 || E < 1 || top_k < 1 || top_k > E) return SDV_ERR_INVALID_ARG;
  if (S > kMaxS || E > kMaxExperts || top_k > kMaxTopK) return SDV_ERR_UNSUPPORTED;
  const int n_cap = E < S * top_k ? E : S * top_k;
  return cuda_status(sdv::launch_moe_route(router_logits, S, E, top_k, ids, weights, offsets, pair_rows, n_hit,
                                           hit, nullptr, n_cap, reinterpret_cast<cudaStream_t>(stream)));
}

sdv_status sdv_moe_gather_qmm(const sdv_qweight* gate, const sdv_qweight* up, const sdv_qweight* down,
                              int32_t E, int32_t I, int32_t H, int32_t top_k, const uint16_t* x,
                              const float* router_logits, int32_t S, float* out,
                              int32_t* topk_ids_or_null, float* topk_w_or_null, void* ws,
                              size_t ws_bytes, sdv_stream_t stream) {
  if (!moe_args_ok(gate, up, down, E, I, H, top_k)) return SDV_ERR_INVALID_ARG;
  if (x == nullptr || router_logits == nullptr || out == nullptr || !aligned16(x)) return SDV_ERR_INVALID_ARG;
  if (S < 1) return SDV_ERR_INVALID_ARG;
  if (S > kMaxS || E > kMaxExperts || top_k > kMaxTopK) return SDV_ERR_UNSUPPORTED;
  // the tcgen05 path streams whole 128-row tiles of each expert and 256-column
  // stages of each segment
  if (I % 256 != 0 || H % 256 != 0 || g_gemm_path.load() == 1) return SDV_ERR_UNSUPPORTED;
  const MoeLayout L = plan_moe(gate->qtype, E, I, H, top_k, S);
  if (L.total == 0) return SDV_ERR_UNSUPPORTED;
  if (ws == nullptr || !aligned16(ws) || ws_bytes < L.total) return SDV_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* const w8 = static_cast<char*>(ws);
  int32_t* const ids = reinterpret_cast<int32_t*>(w8 + L.ids);
  float* const rw8 = reinterpret_cast<float*>(w8 + L.w);
  int32_t* const n_hit = reinterpret_cast<int32_t*>(w8 + L.n_hit);
  int32_t* const hit = reinterpret_cast<int32_t*>(w8 + L.hit);
  float* const row_w = reinterpret_cast<float*>(w8 + L.row_w);
  __half* const hb = reinterpret_cast<__half*>(w8 + L.hbuf);
  float* const dn = reinterpret_cast<float*>(w8 + L.dn_part);
  const int ncap_i = L.n_cap * I;
  // a7 + a8: route and group -- in the gate/up launch's prologue where it fits
  // (each CTA routes the window itself, CTA 0 publishes the picks and the hit
  // list), else a routing launch first
  cudaError_t e = cudaSuccess;
  if (!L.route) {
    e = sdv::launch_moe_route(router_logits, S, E, top_k, ids, rw8, reinterpret_cast<int32_t*>(w8 + L.offsets),
                              reinterpret_cast<int32_t*>(w8 + L.pair_rows), n_hit, hit, row_w, L.n_cap, st);
    if (e != cudaSuccess) return cuda_status(e);
  }
  // a9, gate and up: every window row through each hit expert's rows (gate/up
  // tile pairs over the hit list) with the SwiGLU epilogue writing
  // h'[s][j * I + c] = fp16(w(s, hit j) * SiLU(g) * u), zero where row s did not pick hit j
  {
    GemmArgs a{};
    a.x = reinterpret_cast<const __half*>(x);
    a.S = S;
    a.N = ncap_i;
    a.K = H;
    a.dual = 2;
    a.rows_per_expert = I;
    a.h = hb;
    a.ldh = ncap_i;
    if (L.route) {
      a.route_logits = router_logits;
      a.route_E = E;
      a.route_top_k = top_k;
      a.route_ids = ids;
      a.route_w = rw8;
      a.route_n_hit = n_hit;
      a.route_hit = hit;
    } else {
      a.n_hit = n_hit;
      a.hit = hit;
      a.row_w = row_w;
      a.ldw = L.n_cap;
    }
    sdv_status s = launch_tc_y(gate, up, L.gu, a, ws, st);
    if (s != SDV_OK) return s;
  }
  // a9, down and combine: out = h' (hit experts' segments along the reduction) x
  // the hit experts' down rows, split by expert-segment slots, reduced in order
  {
    GemmArgs a{};
    a.x = hb;
    a.S = S;
    a.N = H;
    a.K = ncap_i;
    a.ldx = ncap_i;
    a.n_hit = n_hit;
    a.hit = hit;
    a.rows_per_expert = H;
    a.seg_k = I;
    a.y = dn;
    sdv_status s = launch_tc_y(down, nullptr, L.dn, a, ws, st);
    if (s != SDV_OK) return s;
  }
  e = sdv::launch_splitk_reduce(dn, L.ys, (long)S * H, out, st);
  if (e != cudaSuccess) return cuda_status(e);
  if (topk_ids_or_null != nullptr)
    e = cudaMemcpyAsync(topk_ids_or_null, ids, (size_t)S * top_k * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && topk_w_or_null != nullptr)
    e = cudaMemcpyAsync(topk_w_or_null, rw8, (size_t)S * top_k * 4, cudaMemcpyDeviceToDevice, st);
  return cuda_status(e);
}

}  // extern "C"
