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
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sdv.h"

namespace {

// 256-byte header (status word, ticket) + per-CTA (max, index) partials:
// room for grid * S <= 8192, i.e. S <= 32 on devices with up to 256 SMs.
constexpr size_t kScratchBytes = 256 + 64 * 1024;

// One copy per device that loads the library; it stays resident until the
// process exits.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_scratch on the current device.  In host code the name
// g_scratch is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached.
sdv_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SDV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SDV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return SDV_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SDV_OK;
}

}  // namespace

extern "C" SDV_API sdv_status sdv_verify_head_noalloc(const sdv_qweight* head, const uint16_t* x,
                                                      int32_t S, const int32_t* drafts,
                                                      int32_t n_valid, float* logits_or_null,
                                                      int32_t* argmax, int32_t* accepted,
                                                      int32_t* next_a0, sdv_stream_t stream) {
  if (head == nullptr) return SDV_ERR_INVALID_ARG;
  if (S < 1) return SDV_ERR_INVALID_ARG;
  if (S > 32) return SDV_ERR_UNSUPPORTED;
  const size_t need = sdv_workspace_bytes(SDV_OP_VERIFY_HEAD, head->n, head->k, S, 0, 0);
  if (need == 0) return SDV_ERR_CUDA;
  if (need > kScratchBytes) return SDV_ERR_WORKSPACE;  // beyond the fixed scratch
  void* ws = nullptr;
  const sdv_status st = scratch_address(&ws);
  if (st != SDV_OK) return st;
  // The scratch keeps the previous call's contents: clear the status word and
  // the ticket, which must start at zero.
  if (cudaMemsetAsync(ws, 0, 256, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SDV_ERR_CUDA;
  return sdv_verify_head(head, x, S, drafts, n_valid, logits_or_null, argmax, accepted, next_a0, ws,
                         kScratchBytes, stream);
}
