// sdv_verify_head_noalloc: the verify head for callers that cannot allocate
// device memory.
//
// Some callers of this library hold only a stream and the tensors a host
// framework hands them: the framework owns every byte of device memory (a
// fixed pool carved out at start-up) and forbids side allocations, or the call
// sits in a latency-critical loop where cudaMalloc, which may synchronise the
// device, is not allowed.  Such callers cannot provide the workspace that
// sdv_verify_head needs.  This entry point runs the same kernel with its
// scratch (status word, last-CTA ticket, per-CTA argmax partials) in a
// file-scope device array instead.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "sdv.h"
#include "sdv_kernels.h"

namespace {

// 256-byte header (word 0: status, word 1: last-CTA ticket) + per-CTA
// (max, index) partials: room for grid * S <= 8192, i.e. S <= 32 on devices
// with up to 256 SMs.
constexpr size_t kScratchBytes = 256 + 64 * 1024;
constexpr size_t kTicketOffset = 4;

// One copy per device that loads the library; it stays resident until the
// process exits.  Zero-initialised when the module is loaded.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// In host code the name g_scratch is only a host-side stand-in, so its device
// address is looked up (cudaGetSymbolAddress) with the device current, once
// per CUDA context: a context made after cudaDeviceReset loads the module
// again, and the array may then sit elsewhere.
constexpr int kMaxDevices = 128;
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
ScratchEntry g_scratch_at[kMaxDevices] = {};
std::mutex g_scratch_mu;

struct DriverCalls {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const DriverCalls& driver_calls() {
  static DriverCalls d;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      d.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      d.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return d;
}

// Unique id of the calling thread's current context (0 when none is current).
bool current_context_id(unsigned long long* id) {
  const DriverCalls& d = driver_calls();
  if (d.get_current == nullptr || d.get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (d.get_current(&ctx) != CUDA_SUCCESS) return false;
  *id = 0;
  if (ctx == nullptr) return true;
  return d.get_id(ctx, id) == CUDA_SUCCESS;
}

sdv_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SDV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SDV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long ctx = 0;
  if (!current_context_id(&ctx)) return SDV_ERR_CUDA;
  ScratchEntry& e = g_scratch_at[dev];
  if (ctx == 0 || e.addr == nullptr || e.ctx_id != ctx) {
    // the lookup makes the device's primary context current if none was, and
    // loads this file's module if lazy loading had not loaded it yet
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return SDV_ERR_CUDA;
    if (!current_context_id(&ctx) || ctx == 0) return SDV_ERR_CUDA;
    e.addr = p;
    e.ctx_id = ctx;
  }
  *out = e.addr;
  return SDV_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The argument checks of sdv_verify_head, done here before anything touches the
// device, so that an invalid call launches nothing and leaves the scratch as it was.
sdv_status check_args(const sdv_qweight* head, const uint16_t* x, int32_t S, const int32_t* drafts,
                      int32_t n_valid, const int32_t* argmax, const int32_t* accepted, const int32_t* next_a0) {
  if (head == nullptr || head->codes == nullptr || head->scales == nullptr) return SDV_ERR_INVALID_ARG;
  if (head->qtype != SDV_Q8 && head->qtype != SDV_Q4 && head->qtype != SDV_F4) return SDV_ERR_INVALID_ARG;
  if (head->n < 1 || head->k < 32 || head->k % 32 != 0) return SDV_ERR_INVALID_ARG;
  if (!aligned16(head->codes) || !aligned16(head->scales)) return SDV_ERR_INVALID_ARG;
  if (x == nullptr || !aligned16(x)) return SDV_ERR_INVALID_ARG;
  if (argmax == nullptr || accepted == nullptr || next_a0 == nullptr) return SDV_ERR_INVALID_ARG;
  if (S < 1) return SDV_ERR_INVALID_ARG;
  if (S > 32) return SDV_ERR_UNSUPPORTED;
  if (n_valid < 0 || n_valid > S - 1) return SDV_ERR_INVALID_ARG;
  if (n_valid > 0 && drafts == nullptr) return SDV_ERR_INVALID_ARG;
  return SDV_OK;
}

}  // namespace

extern "C" SDV_API sdv_status sdv_verify_head_noalloc(const sdv_qweight* head, const uint16_t* x,
                                                      int32_t S, const int32_t* drafts,
                                                      int32_t n_valid, float* logits_or_null,
                                                      int32_t* argmax, int32_t* accepted,
                                                      int32_t* next_a0, sdv_stream_t stream) {
  const sdv_status bad = check_args(head, x, S, drafts, n_valid, argmax, accepted, next_a0);
  if (bad != SDV_OK) return bad;
  // the weight is valid here, so 0 can only mean a shape the plans reject
  if (sdv_workspace_bytes(SDV_OP_VERIFY_HEAD, head->n, head->k, S, 0, 0) == 0) return SDV_ERR_INVALID_ARG;
  // The least scratch a head call uses -- status word, ticket and per-CTA argmax
  // partials, the same for every weight (a one-row head asks for exactly that).
  // Windows whose rows need the reduction split for the tensor-core plan run in
  // row chunks here instead: the fixed scratch cannot hold partial logits.
  const size_t need = sdv_workspace_bytes(SDV_OP_VERIFY_HEAD, 1, 32, S, 0, 0);
  if (need == 0 || need > kScratchBytes) return SDV_ERR_WORKSPACE;  // beyond the fixed scratch
  void* ws = nullptr;
  const sdv_status st = scratch_address(&ws);
  if (st != SDV_OK) return st;
  // The scratch keeps the previous call's contents.  The ticket must start at
  // zero (every completed call leaves it there; clearing it costs nothing).  The
  // status word is left alone: a bounded wait that gave up stays visible until
  // sdv_noalloc_device_status reads it.
  if (cudaMemsetAsync(static_cast<char*>(ws) + kTicketOffset, 0, 4, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return SDV_ERR_CUDA;
  return sdv_verify_head(head, x, S, drafts, n_valid, logits_or_null, argmax, accepted, next_a0, ws,
                         kScratchBytes, stream);
}

extern "C" SDV_API sdv_status sdv_noalloc_device_status(sdv_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return SDV_ERR_CUDA;
  void* ws = nullptr;
  const sdv_status st = scratch_address(&ws);
  if (st != SDV_OK) return st;
  int word = 0;
  if (cudaMemcpy(&word, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SDV_ERR_CUDA;
  if (word == 0) return SDV_OK;
  const int zero = 0;
  if (cudaMemcpy(ws, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return SDV_ERR_CUDA;
  return (word & sdv::kDevErrTimeout) ? SDV_ERR_TIMEOUT : SDV_ERR_CUDA;
}
