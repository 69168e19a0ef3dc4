// Test infrastructure: drives libsdv's C ABI from commands on standard input,
// with the stand-in runtime of stub_runtime.cpp, and prints each call's
// launches.  Commands (one per line):
//   device <sms> <smem_optin>             the device the queries describe
//   path <0|1|2>                          sdv_set_gemm_path
//   head <qtype> <n> <k> <S> <n_valid> <logits 0|1>
//   sample <qtype> <n> <k> <S> <n_valid>
//   qlinear <qtype> <n> <k> <S>
//   swiglu <qtype> <n> <k> <S>
//   moe <qtype> <E> <I> <H> <top_k> <S>
//   noalloc <qtype> <n> <k> <S> <n_valid>
//   ws <op> <n> <k> <S> <E> <top_k>
//   count   (prints sdv_launch_count())
// Output: "call <command>", the call's trace lines, then "status <code>" (or
// "ws bytes=<n>").  Pointers are distinct 16-byte-aligned addresses that are
// never dereferenced.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>

#include "sdv.h"

extern "C" void trace_set_device(int sms, int smem);

namespace {

void* addr(uint64_t off) { return reinterpret_cast<void*>(0x100000000ull + off); }

sdv_qweight weight(int qtype, int n, int k, uint64_t base) {
  sdv_qweight w;
  w.qtype = static_cast<sdv_qtype>(qtype);
  w.n = n;
  w.k = k;
  w.codes = addr(base);
  w.scales = static_cast<const uint16_t*>(addr(base + 0x8000000));
  return w;
}

const uint16_t* X = static_cast<const uint16_t*>(addr(0x20000000));
const int32_t* DRAFTS = static_cast<const int32_t*>(addr(0x21000000));
float* OUT = static_cast<float*>(addr(0x22000000));
int32_t* ARGMAX = static_cast<int32_t*>(addr(0x23000000));
int32_t* ACCEPTED = static_cast<int32_t*>(addr(0x23001000));
int32_t* NEXT = static_cast<int32_t*>(addr(0x23002000));
void* WS = addr(0x30000000);

}  // namespace

int main() {
  char line[512];
  while (std::fgets(line, sizeof line, stdin)) {
    char cmd[32] = {0};
    int a[8] = {0};
    const int got = std::sscanf(line, "%31s %d %d %d %d %d %d %d %d", cmd, &a[0], &a[1], &a[2], &a[3], &a[4], &a[5],
                                &a[6], &a[7]);
    if (got < 1) continue;
    line[std::strcspn(line, "\n")] = 0;
    std::printf("call %s\n", line);
    const std::string c = cmd;
    int st = -1;
    if (c == "device") {
      trace_set_device(a[0], a[1]);
      st = 0;
    } else if (c == "path") {
      st = sdv_set_gemm_path(a[0]) < 0 ? -1 : 0;
    } else if (c == "head") {
      const sdv_qweight w = weight(a[0], a[1], a[2], 0x1000);
      const size_t ws = sdv_workspace_bytes(SDV_OP_VERIFY_HEAD, a[1], a[2], a[3], 0, 0);
      st = sdv_verify_head(&w, X, a[3], DRAFTS, a[4], a[5] ? OUT : nullptr, ARGMAX, ACCEPTED, NEXT, WS, ws, nullptr);
    } else if (c == "sample") {
      const sdv_qweight w = weight(a[0], a[1], a[2], 0x1000);
      const size_t ws = sdv_workspace_bytes(SDV_OP_VERIFY_SAMPLE, a[1], a[2], a[3], 0, 0);
      st = sdv_verify_sample(&w, X, a[3], DRAFTS, a[4], 0.7f, 11, 3, nullptr, ARGMAX, ACCEPTED, NEXT, WS, ws,
                             nullptr);
    } else if (c == "qlinear") {
      const sdv_qweight w = weight(a[0], a[1], a[2], 0x1000);
      const size_t ws = sdv_workspace_bytes(SDV_OP_QLINEAR, a[1], a[2], a[3], 0, 0);
      st = sdv_qlinear(&w, X, a[3], OUT, WS, ws, nullptr);
    } else if (c == "swiglu") {
      const sdv_qweight g = weight(a[0], a[1], a[2], 0x1000), u = weight(a[0], a[1], a[2], 0x40000000);
      const size_t ws = sdv_workspace_bytes(SDV_OP_QLINEAR_SWIGLU, a[1], a[2], a[3], 0, 0);
      st = sdv_qlinear_swiglu(&g, &u, X, a[3], reinterpret_cast<uint16_t*>(OUT), WS, ws, nullptr);
    } else if (c == "moe") {
      const int E = a[1], I = a[2], H = a[3], top_k = a[4], S = a[5];
      const sdv_qweight g = weight(a[0], E * I, H, 0x1000), u = weight(a[0], E * I, H, 0x40000000),
                        d = weight(a[0], E * H, I, 0x80000000);
      const size_t ws = sdv_workspace_bytes(SDV_OP_MOE, I, H, S, E, top_k);
      st = sdv_moe_gather_qmm(&g, &u, &d, E, I, H, top_k, X, static_cast<const float*>(addr(0x24000000)), S, OUT,
                              nullptr, nullptr, WS, ws, nullptr);
    } else if (c == "noalloc") {
      const sdv_qweight w = weight(a[0], a[1], a[2], 0x1000);
      st = sdv_verify_head_noalloc(&w, X, a[3], DRAFTS, a[4], nullptr, ARGMAX, ACCEPTED, NEXT, nullptr);
    } else if (c == "count") {  // the library's own launch counter
      std::printf("count n=%llu\n", static_cast<unsigned long long>(sdv_launch_count()));
    } else if (c == "ws") {
      std::printf("ws bytes=%zu\n", sdv_workspace_bytes(a[0], a[1], a[2], a[3], a[4], a[5]));
      continue;
    }
    std::printf("status %d\n", st);
  }
  return 0;
}
