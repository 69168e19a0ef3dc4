// Test infrastructure: a stand-in for the CUDA runtime that lets libsdv's host
// code run on a machine without a GPU and records every launch it makes.
//
// The library's translation units are compiled as usual and linked against
// these definitions instead of libcudart.  Device queries answer with a chosen
// SM count and shared-memory limit, the tensor-map encoder records each map's
// box, and each kernel launch prints one line: the kernel (by the name the
// compiler registered for it), grid, block, dynamic shared memory and, for the
// tcgen05 GEMM, its launch arguments.  Nothing is computed and no device
// memory exists: the pointers the test passes are never dereferenced here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <map>
#include <string>

#include "sdv_kernels.h"

namespace {

int g_sms = 152, g_smem = 232448;

// kernel host function -> registered device name (a function-local static:
// registration runs from other translation units' static initialisers)
std::map<const void*, std::string>& names() {
  static std::map<const void*, std::string> m;
  return m;
}

dim3 g_grid, g_block;
size_t g_shmem = 0;

unsigned long long low(const void* p) { return reinterpret_cast<unsigned long long>(p) & 0xFFFFFFFull; }

CUresult record_tensor_map(CUtensorMap* m, CUtensorMapDataType dt, cuuint32_t, void*, const cuuint64_t* dims,
                           const cuuint64_t* strides, const cuuint32_t* box, const cuuint32_t*,
                           CUtensorMapInterleave, CUtensorMapSwizzle sw, CUtensorMapL2promotion,
                           CUtensorMapFloatOOBfill) {
  std::printf("tmap dtype=%d dims=%llu,%llu stride=%llu box=%u,%u swizzle=%d\n", (int)dt,
              (unsigned long long)dims[0], (unsigned long long)dims[1], (unsigned long long)strides[0], box[0],
              box[1], (int)sw);
  std::memset(m, 0, sizeof(*m));
  return CUDA_SUCCESS;
}

}  // namespace

extern "C" void trace_set_device(int sms, int smem) {
  g_sms = sms;
  g_smem = smem;
}

extern "C" {

// ---- registration of the translation units' kernels ----
void** __cudaRegisterFatBinary(void*) {
  static void* handle[4];
  return handle;
}
void __cudaRegisterFatBinaryEnd(void**) {}
void __cudaUnregisterFatBinary(void**) {}
void __cudaRegisterFunction(void**, const char* host_fn, char*, const char* device_name, int, void*, void*, void*,
                            void*, int*) {
  names()[host_fn] = device_name;
}
void __cudaRegisterVar(void**, char*, char*, const char*, int, size_t, int, int) {}

// ---- <<<...>>> launches: the configuration is recorded when it is pushed ----
unsigned __cudaPushCallConfiguration(dim3 grid, dim3 block, size_t shmem, void*) {
  g_grid = grid;
  g_block = block;
  g_shmem = shmem;
  std::printf("launch kind=chevron grid=%u,%u block=%u smem=%zu\n", grid.x, grid.y, block.x, shmem);
  return 0;
}
cudaError_t __cudaPopCallConfiguration(dim3* grid, dim3* block, size_t* shmem, void*) {
  *grid = g_grid;
  *block = g_block;
  *shmem = g_shmem;
  return cudaSuccess;
}
int __cudaLaunchKernel() { return 0; }
int __cudaGetKernel() { return 0; }

CUresult fake_ctx_get_current(CUcontext* c) {
  *c = reinterpret_cast<CUcontext>(0x1000);
  return CUDA_SUCCESS;
}
CUresult fake_ctx_get_id(CUcontext, unsigned long long* id) {
  *id = 1;
  return CUDA_SUCCESS;
}

// ---- the public runtime calls the library makes ----
cudaError_t cudaGetDevice(int* d) {
  *d = 0;
  return cudaSuccess;
}
cudaError_t cudaDeviceGetAttribute(int* v, cudaDeviceAttr attr, int) {
  *v = attr == cudaDevAttrMultiProcessorCount ? g_sms : attr == cudaDevAttrMaxSharedMemoryPerBlockOptin ? g_smem : 0;
  return cudaSuccess;
}
cudaError_t cudaGetDriverEntryPointByVersion(const char* sym, void** fn, unsigned int, unsigned long long,
                                             cudaDriverEntryPointQueryResult* q) {
  if (std::strcmp(sym, "cuTensorMapEncodeTiled") == 0) {
    *fn = reinterpret_cast<void*>(&record_tensor_map);
    *q = cudaDriverEntryPointSuccess;
    return cudaSuccess;
  }
  if (std::strcmp(sym, "cuCtxGetCurrent") == 0) {  // one fixed context
    *fn = reinterpret_cast<void*>(&fake_ctx_get_current);
    *q = cudaDriverEntryPointSuccess;
    return cudaSuccess;
  }
  if (std::strcmp(sym, "cuCtxGetId") == 0) {
    *fn = reinterpret_cast<void*>(&fake_ctx_get_id);
    *q = cudaDriverEntryPointSuccess;
    return cudaSuccess;
  }
  *fn = nullptr;
  *q = cudaDriverEntryPointSymbolNotFound;
  return cudaErrorUnknown;
}
cudaError_t cudaFuncSetAttribute(const void*, cudaFuncAttribute, int) { return cudaSuccess; }
cudaError_t cudaLaunchKernelExC(const cudaLaunchConfig_t* c, const void* fn, void** args) {
  const auto it = names().find(fn);
  const std::string name = it == names().end() ? "?" : it->second;
  std::printf("launch kind=ex name=%s grid=%u,%u block=%u smem=%zu", name.c_str(), c->gridDim.x, c->gridDim.y,
              c->blockDim.x, c->dynamicSmemBytes);
  if (name.find("tc_gemm_kernel") != std::string::npos) {
    const sdv::GemmArgs& a = *static_cast<const sdv::GemmArgs*>(args[4]);
    std::printf(" S=%d N=%d K=%d k_chunk=%d splits=%d depth=%d scales_tma=%d n_valid=%d dual=%d seg_k=%d"
                " rows_per_expert=%d y=%llx h=%llx part_v=%llx part_s=%llx x=%llx route=%d route_E=%d"
                " route_top_k=%d listed=%d",
                a.S, a.N, a.K, a.k_chunk, a.splits, a.depth, a.scales_tma, a.n_valid, a.dual, a.seg_k,
                a.rows_per_expert, low(a.y), low(a.h), low(a.part_v), low(a.part_s), low(a.x),
                a.route_logits != nullptr ? 1 : 0, a.route_E, a.route_top_k, a.n_hit != nullptr ? 1 : 0);
  }
  if (name.find("splitk_reduce_kernel") != std::string::npos ||
      name.find("swiglu_reduce_kernel") != std::string::npos)  // first argument: the partials
    std::printf(" part=%llx", low(*static_cast<const float* const*>(args[0])));
  std::printf("\n");
  return cudaSuccess;
}
cudaError_t cudaGetLastError() { return cudaSuccess; }
cudaError_t cudaGetSymbolAddress(void** p, const void*) {
  *p = reinterpret_cast<void*>(0x7000000000ull);
  return cudaSuccess;
}
cudaError_t cudaMemcpy(void* dst, const void*, size_t n, cudaMemcpyKind kind) {
  // the only device-to-host read is the status word: report "no error"
  if (kind == cudaMemcpyDeviceToHost && n <= 64) std::memset(dst, 0, n);
  return cudaSuccess;
}
cudaError_t cudaMemcpyAsync(void*, const void*, size_t n, cudaMemcpyKind, cudaStream_t) {
  std::printf("memcpy bytes=%zu\n", n);
  return cudaSuccess;
}
cudaError_t cudaMemsetAsync(void*, int, size_t n, cudaStream_t) {
  std::printf("memset bytes=%zu\n", n);
  return cudaSuccess;
}
cudaError_t cudaStreamSynchronize(cudaStream_t) { return cudaSuccess; }

}  // extern "C"
