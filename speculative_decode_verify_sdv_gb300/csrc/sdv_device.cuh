// Device-side building blocks shared by the libsdv kernels: mbarriers, TMA
// (cp.async.bulk.tensor) loads with bounded waits, exact integer-code -> fp16
// conversions, the m16n8k16 tensor-core MMA and the (value, index) argmax order.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

namespace sdv {

// Give up on an asynchronous copy after this long (nanoseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of an mbarrier, giving up after `limit_ns`.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// L2 policy for data read exactly once (weights): evict first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 2-D tiled TMA load of the box at (x = inner element, y = row) into shared
// memory, completing on `bar` (transaction bytes).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Four signed int8 codes e0..e3 (e0 in bits 0-7) -> exact fp16 pairs
// lo = (e0, e2), hi = (e1, e3).  Each byte, xor 0x80, is placed in the mantissa
// of 1024 (1024 + e + 128 is exact for e in [-128, 127]) and the bias removed.
__device__ __forceinline__ void i8x4_to_h2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const __half2 bias = u32_as_h2(0x64806480u);  // (1152, 1152)
  const uint32_t t0 = (w & 0x00FF00FFu) ^ 0x64806480u;
  const uint32_t t1 = ((w >> 8) & 0x00FF00FFu) ^ 0x64806480u;
  lo = h2_as_u32(__hsub2(u32_as_h2(t0), bias));
  hi = h2_as_u32(__hsub2(u32_as_h2(t1), bias));
}

// Four signed int8 codes -> the fp16 pairs of e * s (same pairing as
// i8x4_to_h2x2) with scale and bias in one HFMA2 per pair.  One xor of the word
// turns each code into u = e + 128 in [0, 255], which in bits 0-7 of an fp16
// half reads as the subnormal u * 2^-24 (exact); fma(u * 2^-24, m, c) with
// m = s * 2^24 and c = -128 s is u * s - 128 s = e * s computed exactly and
// rounded once: the bits of fp16(e) * s.  Valid while m is finite
// (s <= 65504 * 2^-24); m and c in both halves.
__device__ __forceinline__ void i8x4_to_h2x2_scaled(uint32_t w, __half2 m, __half2 c, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;
  // bytes 0, 2 and bytes 1, 3 into the low byte of each half, the rest zero:
  // one byte permute each (with a zero second operand)
  lo = h2_as_u32(__hfma2(u32_as_h2(__byte_perm(x, 0u, 0x4240u)), m, c));  // (e0, e2)
  hi = h2_as_u32(__hfma2(u32_as_h2(__byte_perm(x, 0u, 0x4341u)), m, c));  // (e1, e3)
}

// Eight signed int4 codes n0..n7 (n0 in bits 0-3) -> exact fp16 pairs
// p0 = (n0, n4), p1 = (n1, n5), p2 = (n2, n6), p3 = (n3, n7).
// Nibbles at bits 0-3 of each 16-bit half land as 1024 + (n + 8); nibbles at
// bits 4-7 land as 1024 + 16 (n + 8) and are rescaled by 1/16 (exact).
__device__ __forceinline__ void i4x8_to_h2x4(uint32_t w, uint32_t& p0, uint32_t& p1, uint32_t& p2,
                                             uint32_t& p3) {
  const __half2 b_lo = u32_as_h2(0x64086408u);       // (1032, 1032)
  const __half2 sixteenth = u32_as_h2(0x2C002C00u);  // (1/16, 1/16)
  const __half2 b_hi = u32_as_h2(0xD480D480u);       // (-72, -72)
  const uint32_t y = w >> 8;
  const uint32_t t0 = (w & 0x000F000Fu) ^ 0x64086408u;
  const uint32_t t1 = (w & 0x00F000F0u) ^ 0x64806480u;
  const uint32_t t2 = (y & 0x000F000Fu) ^ 0x64086408u;
  const uint32_t t3 = (y & 0x00F000F0u) ^ 0x64806480u;
  p0 = h2_as_u32(__hsub2(u32_as_h2(t0), b_lo));
  p1 = h2_as_u32(__hfma2(u32_as_h2(t1), sixteenth, b_hi));
  p2 = h2_as_u32(__hsub2(u32_as_h2(t2), b_lo));
  p3 = h2_as_u32(__hfma2(u32_as_h2(t3), sixteenth, b_hi));
}

// (a & mask) ^ flip in one LOP3: mask an immediate, flip a register.
template <uint32_t kMask>
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t flip) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(d) : "r"(a), "n"(kMask), "r"(flip));
  return d;
}

// The tcgen05 converters' int4 forms.  Eight signed int4 codes n0..n7 of a
// 32-bit word give the fp16 pairs (n0, n4), (n1, n5), (n2, n6), (n3, n7) -- the
// pairing of i4x8_to_h2x4 -- with (n0, n4) and (n2, n6) scaled by 2^-4: those
// codes sit at bits 0-3 of each half of w and of w >> 8, and taking them there
// needs the 2^-4 (their accumulators are scaled back by 16 in the epilogue).
// The LOP3 that masks a code also flips its top bit, giving u = n + 8 in
// [0, 15].  One-FMA form: a code at bits 4-7 reads as the subnormal u * 2^-20,
// one at bits 0-3 as u * 2^-24 (both exact); fma with m = s * 2^20 and
// c = -8 s, resp. c_lo = -s / 2, gives n * s, resp. n * s / 16, computed
// exactly and rounded once.  Valid while m is finite (s <= 65504 * 2^-20) and
// s / 2 is exact (s = 0 or s >= 2^-13); m, c, c_lo in both halves.
__device__ __forceinline__ void i4x8_to_h2x4_split(uint32_t w, __half2 m, __half2 c, __half2 c_lo, uint32_t& p0,
                                                   uint32_t& p1, uint32_t& p2, uint32_t& p3) {
  const uint32_t flip_hi = 0x00800080u, flip_lo = 0x00080008u;  // the top bit of a code at bits 4-7 / 0-3
  const uint32_t y = w >> 8;
  p0 = h2_as_u32(__hfma2(u32_as_h2(and_xor<0x000F000Fu>(w, flip_lo)), m, c_lo));  // (n0, n4) / 16
  p1 = h2_as_u32(__hfma2(u32_as_h2(and_xor<0x00F000F0u>(w, flip_hi)), m, c));     // (n1, n5)
  p2 = h2_as_u32(__hfma2(u32_as_h2(and_xor<0x000F000Fu>(y, flip_lo)), m, c_lo));  // (n2, n6) / 16
  p3 = h2_as_u32(__hfma2(u32_as_h2(and_xor<0x00F000F0u>(y, flip_hi)), m, c));     // (n3, n7)
}

// The same pairs as exact fp16 values before the scale, (n0, n4) and (n2, n6)
// as n / 16: the exponent-bias form of i4x8_to_h2x4 with (1024 + u) / 16 - 64.5
// = n / 16 (exact) for those two pairs; times s (HMUL2) they round once, to the
// bits of the one-FMA form.
__device__ __forceinline__ void i4x8_to_h2x4_split_exact(uint32_t w, uint32_t& p0, uint32_t& p1, uint32_t& p2,
                                                         uint32_t& p3) {
  const __half2 sixteenth = u32_as_h2(0x2C002C00u);  // (1/16, 1/16)
  const __half2 b_lo = u32_as_h2(0xD408D408u);       // (-64.5, -64.5)
  const __half2 b_hi = u32_as_h2(0xD480D480u);       // (-72, -72)
  const uint32_t y = w >> 8;
  const uint32_t t0 = (w & 0x000F000Fu) ^ 0x64086408u;
  const uint32_t t1 = (w & 0x00F000F0u) ^ 0x64806480u;
  const uint32_t t2 = (y & 0x000F000Fu) ^ 0x64086408u;
  const uint32_t t3 = (y & 0x00F000F0u) ^ 0x64806480u;
  p0 = h2_as_u32(__hfma2(u32_as_h2(t0), sixteenth, b_lo));
  p1 = h2_as_u32(__hfma2(u32_as_h2(t1), sixteenth, b_hi));
  p2 = h2_as_u32(__hfma2(u32_as_h2(t2), sixteenth, b_lo));
  p3 = h2_as_u32(__hfma2(u32_as_h2(t3), sixteenth, b_hi));
}

// Counter stream of the sampling verify: SplitMix64 (Steele, Lea & Flood,
// OOPSLA 2014; finaliser constants as published by Vigna) keyed by
// key = mix(seed + (counter + 1) * G); output c = mix(key + (c + 1) * G) carries
// elements 2c (low 32 bits) and 2c + 1 (high 32 bits).
constexpr unsigned long long kSplitMixG = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ unsigned long long splitmix_mix(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// u = (2 * (h >> 9) + 1) * 2^-24 for a 32-bit half h: in (0, 1), exact in fp32.
__device__ __forceinline__ float half_uniform(unsigned h) {
  return (float)(2u * (h >> 9) + 1u) * 5.9604644775390625e-8f;
}

__device__ __forceinline__ unsigned long long counter_pair(unsigned long long key, unsigned long long c) {
  return splitmix_mix(key + (c + 1ull) * kSplitMixG);
}

// u(e) of element e.
__device__ __forceinline__ float counter_uniform(unsigned long long key, unsigned long long e) {
  const unsigned long long w = counter_pair(key, e >> 1);
  return half_uniform((e & 1ull) ? (unsigned)(w >> 32) : (unsigned)w);
}

// Standard Gumbel from u: -log(-log(u)), with -log(u) = -log1p(-(1 - u)) (1 - u
// is exact) so that the upper tail (u near 1) keeps its accuracy; the outer log
// is the fast hardware one (absolute error ~1e-6, below what the draws compare).
__device__ __forceinline__ float gumbel_of(float u) { return -__logf(-log1pf(-(1.f - u))); }

// Top 1 under the argmax order (value desc, index asc).
__device__ __forceinline__ void top1_add(float& z1, int& v1, float z, int v) {
  if (z > z1 || (z == z1 && v < v1)) {
    z1 = z;
    v1 = v;
  }
}

// Online softmax statistics: m = max, s = sum exp(x - m); -inf entries are absent.
__device__ __forceinline__ void softmax_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
  } else if (m2 > m) {
    s = s * expf(m - m2) + s2;
    m = m2;
  } else {
    s += s2 * expf(m2 - m);
  }
}

// FP4 (E2M1, OCP Microscaling): 8 codes of w (byte j holds codes 2j in its low,
// 2j + 1 in its high nibble) to f16x2 pairs (k0, k1), (k2, k3), (k4, k5),
// (k6, k7) by the hardware conversion; every E2M1 value is exact in fp16.
__device__ __forceinline__ void e2m1x8_to_h2x4(uint32_t w, uint32_t& p0, uint32_t& p1, uint32_t& p2,
                                               uint32_t& p3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(p0), "=r"(p1), "=r"(p2), "=r"(p3)
      : "r"(w));
}

// D = A * B + C, m16n8k16, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}

// Total order for the argmax: larger value first, then lower index.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__device__ __forceinline__ void argmax_merge(float& v, int& i, float ov, int oi) {
  if (better(ov, oi, v, i)) {
    v = ov;
    i = oi;
  }
}

}  // namespace sdv

// ---- tcgen05 (5th-generation tensor core, tensor memory) ------------------------

namespace sdv {

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The 16 MMAs of one 256-column stage under a single elect.sync (one lane
// issues, the warp stays converged): MMA m multiplies A columns a + 8m by the
// B descriptor b + 16m (16-byte units) into accumulator m % NACC at d + N (m % NACC);
// the first NACC MMAs overwrite their accumulator unless `accumulate`.
#define SDV_MMA1(D, P) "@e tcgen05.mma.cta_group::1.kind::f16 [" D "], [ta], tb, %3, " P ";\n\t" \
                        "add.u32 ta, ta, 8;\n\tadd.u64 tb, tb, 16;\n\t"
template <int NACC>
__device__ __forceinline__ void tc_mma_stage16(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t n,
                                               uint32_t accumulate) {
  static_assert(NACC == 2 || NACC == 4, "accumulators per tile");
  if (NACC == 2) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b32 ta, d0, d1;\n\t.reg .b64 tb;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
        "mov.b32 ta, %1;\n\tmov.b64 tb, %2;\n\tmov.b32 d0, %0;\n\tadd.u32 d1, %0, %5;\n\t"
        SDV_MMA1("d0", "p") SDV_MMA1("d1", "p")
        SDV_MMA1("d0", "t") SDV_MMA1("d1", "t") SDV_MMA1("d0", "t") SDV_MMA1("d1", "t")
        SDV_MMA1("d0", "t") SDV_MMA1("d1", "t") SDV_MMA1("d0", "t") SDV_MMA1("d1", "t")
        SDV_MMA1("d0", "t") SDV_MMA1("d1", "t") SDV_MMA1("d0", "t") SDV_MMA1("d1", "t")
        SDV_MMA1("d0", "t") SDV_MMA1("d1", "t")
        "}" ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(n)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b32 ta, d0, d1, d2, d3;\n\t.reg .b64 tb;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
        "mov.b32 ta, %1;\n\tmov.b64 tb, %2;\n\tmov.b32 d0, %0;\n\tadd.u32 d1, %0, %5;\n\t"
        "add.u32 d2, d1, %5;\n\tadd.u32 d3, d2, %5;\n\t"
        SDV_MMA1("d0", "p") SDV_MMA1("d1", "p") SDV_MMA1("d2", "p") SDV_MMA1("d3", "p")
        SDV_MMA1("d0", "t") SDV_MMA1("d1", "t") SDV_MMA1("d2", "t") SDV_MMA1("d3", "t")
        SDV_MMA1("d0", "t") SDV_MMA1("d1", "t") SDV_MMA1("d2", "t") SDV_MMA1("d3", "t")
        SDV_MMA1("d0", "t") SDV_MMA1("d1", "t") SDV_MMA1("d2", "t") SDV_MMA1("d3", "t")
        "}" ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(n)
        : "memory");
  }
}
#undef SDV_MMA1

// tcgen05.commit from a warp-uniform context (one elected lane).
__device__ __forceinline__ void tc_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// Arrive on an mbarrier once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major, no swizzle: core matrices of
// 8 rows x 16 bytes; lbo = byte distance between core matrices adjacent along K,
// sbo = byte distance between 8-row groups.
__device__ __forceinline__ uint64_t smem_desc_kmajor(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version of this tensor-core generation
  return d;                // base offset 0, layout type 0 (no swizzle)
}

// Instruction descriptor of kind::f16: fp16 A and B (K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Programmatic dependent launch: wait until the previous grid in the stream has
// completed and its memory is visible (a no-op without the launch attribute), and
// let the next grid's CTAs be scheduled as this grid's CTAs finish.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace sdv
