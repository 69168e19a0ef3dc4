// Plain, slow CPU oracle of the speculative-decoding verify path.
//
// TEST INFRASTRUCTURE ONLY.  Loaded (through oracle/_native.py) by the tests,
// __graft_entry__.smoke() and the CPU legs of bench.py; never by the product.
// It shares no code, header, table or constant generator with the CUDA path:
// the two meet only in the seeded input bytes that synth/ generates.
//
// Every function states the definition it follows, with the page and section
// it comes from.  Floating point: products and sums in IEEE binary64 (double),
// one multiply and one add per term (built with -ffp-contract=off, so no fused
// multiply-add changes a rounding), reductions in index order.  Work is spread
// over output rows only (OpenMP, static schedule): every output element is
// computed by one thread with exactly the same operations in the same order,
// so results do not depend on the thread count.
//
// Pages:
//  [Q] "Riding Apple's pipelined GPU engine -- 3.5x over a hand-rolled loop, zero
//      custom kernels", section "Quantization on the GPU delegate": per-block-32
//      absmax symmetric linear int8 (ship configuration) and int4 (q4_0 is
//      per-block-32 absmax symmetric int4); big-vocabulary heads plain absmax.
//  [V] "Spec-decode on GDN hybrids (Qwen3.5/3.6 family) -- static-S verify
//      design", sections "Verify graph = STATIC S=K+1" (one forward over the
//      S-row window gives logits for every position) and "Hybrid state
//      discipline" (a0 committed first; the row after the last accepted draft is
//      the next a0; the window is padded to exactly S).
//  [D] "Stream C -- Speculative decoding: feasibility verdict + implementation
//      plan", sections "The delta" (batched argmax [K, vocab] -> [K]; accept
//      while the draft equals the argmax; correction on the first miss, bonus on
//      all-accept), "Control-logic proof" (a_i = argmax(prefix + draft[:i])) and
//      "Deferred / harder" (sampling verify; tree verify).
//  [F] "Flagship dramatic-speedup plan -- the full stackable tuning set",
//      sections "Baseline byte model" (lm_head matvec; routed experts gathered
//      top-8 of 256), "Axis 1" lever 1c (FP4 E2M1 weights) and "Axis 4" (the
//      fused SwiGLU MLP).
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

constexpr int kBlock = 32;  // [Q]: one scale per 32 consecutive weights of a row

// ---------------------------------------------------------------------------
// IEEE binary16 <-> binary32/64 conversions (written from the format: 1 sign
// bit, 5 exponent bits with bias 15, 10 fraction bits; subnormals below 2^-14).
// ---------------------------------------------------------------------------

double half_to_double(uint16_t h) {
  const int sign = h >> 15, e = (h >> 10) & 31, f = h & 1023;
  double v;
  if (e == 0) {
    v = std::ldexp((double)f, -24);  // subnormal (or zero): f * 2^-24
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = std::ldexp((double)(1024 + f), e - 25);  // 1.f * 2^(e-15)
  }
  return sign ? -v : v;
}

// Round a double to the nearest binary16, ties to even (one rounding).
uint16_t double_to_half(double d) {
  const uint16_t sign = std::signbit(d) ? 0x8000 : 0;
  if (std::isnan(d)) return sign | 0x7E00;
  const double a = std::fabs(d);
  // 65520 = halfway between the largest finite half (65504) and 2^16: the tie
  // goes to the even neighbour, which is infinity.
  if (a >= 65520.0) return sign | 0x7C00;
  if (a < std::ldexp(1.0, -14)) {
    // subnormal range: the value in units of 2^-24, rounded to an integer
    // (nearbyint rounds ties to even in the default rounding mode); 1024 units
    // is the smallest normal and is encoded by the same bits
    return sign | (uint16_t)std::nearbyint(std::ldexp(a, 24));
  }
  int e2 = 0;
  std::frexp(a, &e2);  // a = m * 2^e2, m in [0.5, 1)
  int e = e2 - 1;      // a in [2^e, 2^(e+1))
  double r = std::nearbyint(std::ldexp(a, 10 - e));  // significand in units of 2^(e-10): [1024, 2048]
  if (r == 2048.0) {
    r = 1024.0;
    ++e;
  }
  if (e + 15 >= 31) return sign | 0x7C00;
  return sign | (uint16_t)((e + 15) << 10) | (uint16_t)(r - 1024.0);
}

// ---------------------------------------------------------------------------
// FP4 (E2M1) values ([F] Axis 1, lever 1c; the encoding of the OCP
// Microscaling Formats spec v1.0): sign bit 3, magnitude index 0..7 for
// 0, 0.5, 1, 1.5, 2, 3, 4, 6.  The mantissa bit of index i is i & 1.
// ---------------------------------------------------------------------------

double e2m1_magnitude(int idx) {
  // exponent field idx >> 1 (bias 1), mantissa bit idx & 1; field 0 is subnormal
  const int ef = idx >> 1, m = idx & 1;
  if (ef == 0) return 0.5 * m;
  return std::ldexp(1.0 + 0.5 * m, ef - 1);
}

double e2m1_value(int code) {
  const double v = e2m1_magnitude(code & 7);
  return (code & 8) ? -v : v;
}

// The code of r: the nearest E2M1 magnitude to |r| (ties to the even mantissa
// bit), saturating at 6; the sign bit is set for r < 0 unless the magnitude is 0.
uint8_t e2m1_encode(float r) {
  const double a = std::fabs((double)r);
  int best = 0;
  double best_d = a;  // distance to magnitude 0
  for (int i = 1; i < 8; ++i) {
    const double d = std::fabs(a - e2m1_magnitude(i));
    if (d < best_d || (d == best_d && (i & 1) == 0 && (best & 1) == 1)) {
      best = i;
      best_d = d;
    }
  }
  if (best != 0 && r < 0.f) best |= 8;
  return (uint8_t)best;
}

int threads_of(int t) { return t > 0 ? t : 1; }

// Value of weight (row, h) before its scale, for the three code layouts the
// oracle accepts: 0 = int8 integer codes, 1 = E2M1 codes (one per byte, 0..15),
// 2 = the values themselves in float64.
inline double code_value(int kind, const void* codes, int64_t idx) {
  if (kind == 0) return (double)static_cast<const int8_t*>(codes)[idx];
  if (kind == 1) return e2m1_value(static_cast<const uint8_t*>(codes)[idx]);
  return static_cast<const double*>(codes)[idx];
}

// y[s][r] = sum over h of x[s][h] * (q[r][h] * s16[r][h / 32]), h = 0, 1, ...,
// in float64 ([V] "Verify graph = STATIC S=K+1": every window row meets every
// weight once).  x is given as float64 [S][k] (fp16 values widened exactly, or
// float64 activations inside the MoE); the product q * s16 is exact for the
// integer and E2M1 codes (at most 8 + 11 significant bits), and so is its
// product with an fp16 x.
void gemm64(int kind, const void* codes, const uint16_t* scales, int64_t n, int64_t k, const double* x, int S,
            double* y, int threads) {
  std::vector<double> xt((size_t)k * S);  // x transposed to [h][s]: the row loop reads it in order
  for (int s = 0; s < S; ++s)
    for (int64_t h = 0; h < k; ++h) xt[(size_t)h * S + s] = x[(size_t)s * k + h];
  const int64_t nb = k / kBlock;
#pragma omp parallel num_threads(threads_of(threads))
  {
    std::vector<double> acc(S);
#pragma omp for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
      for (int s = 0; s < S; ++s) acc[s] = 0.0;
      for (int64_t b = 0; b < nb; ++b) {
        const double sc = half_to_double(scales[r * nb + b]);
        for (int64_t h = b * kBlock; h < (b + 1) * kBlock; ++h) {
          const double w = code_value(kind, codes, r * k + h) * sc;
          const double* xh = &xt[(size_t)h * S];
          for (int s = 0; s < S; ++s) acc[s] += xh[s] * w;
        }
      }
      for (int s = 0; s < S; ++s) y[(size_t)s * n + r] = acc[s];
    }
  }
}

std::vector<double> widen_halves(const uint16_t* x, int64_t count) {
  std::vector<double> v((size_t)count);
  for (int64_t i = 0; i < count; ++i) v[(size_t)i] = half_to_double(x[i]);
  return v;
}

double silu(double t) { return t / (1.0 + std::exp(-t)); }  // [F] Axis 4: SiLU(t) = t / (1 + e^-t)

// ---------------------------------------------------------------------------
// SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014; finaliser constants as published by Vigna) used as
// a counter-based generator for the sampling verify.
// ---------------------------------------------------------------------------
constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// u(e): element e of the stream keyed by `key`; elements 2c and 2c+1 are the
// low and high halves of output c = mix(key + (c + 1) G); u = (2 (h >> 9) + 1) 2^-24.
double uniform_of(uint64_t key, uint64_t e) {
  const uint64_t w = mix64(key + ((e >> 1) + 1) * kGolden);
  const uint64_t h = (e & 1) ? (w >> 32) : (w & 0xFFFFFFFFull);
  return (2.0 * (double)(h >> 9) + 1.0) * std::ldexp(1.0, -24);
}

// Standard Gumbel from u: -log(-log(u)), with -log(u) = -log1p(-(1 - u)).
double gumbel_of(double u) { return -std::log(-std::log1p(-(1.0 - u))); }

constexpr uint64_t kMaxRows = 32;  // element index of row i, entry v: 32 v + i

}  // namespace

extern "C" {

int orc_version(void) { return 1; }

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_num_procs();
#else
  return 1;
#endif
}

// ---- fp16 ------------------------------------------------------------------
void orc_half_to_double(const uint16_t* h, int64_t count, double* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = half_to_double(h[i]);
}
void orc_double_to_half(const double* d, int64_t count, uint16_t* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = double_to_half(d[i]);
}

// ---- quantisation ([Q]) -------------------------------------------------------
// Per row r and block b of 32 along k: m = max |w|; s32 = m / Q in fp32 (IEEE
// division); the stored scale s16 = fp16(s32), nearest even; every code
// q = clamp(rint(w / s16), -Q, Q) with the division in fp32 and rint rounding
// ties to even; s16 == 0 gives zero codes.  Q = 127 (bits 8) or 7 (bits 4);
// int4 codes are returned one per byte (see orc_pack_nibbles).
int orc_quantize_block32(const float* w, int64_t n, int64_t k, int bits, int8_t* codes, uint16_t* scales,
                         int threads) {
  if (k % kBlock != 0 || (bits != 8 && bits != 4)) return 1;
  const float qmax = bits == 8 ? 127.f : 7.f;
  const int64_t nb = k / kBlock;
#pragma omp parallel for num_threads(threads_of(threads)) schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* blk = w + r * k + b * kBlock;
      float m = 0.f;
      for (int i = 0; i < kBlock; ++i) m = std::fmax(m, std::fabs(blk[i]));
      const float s32 = m / qmax;
      const uint16_t s16 = double_to_half((double)s32);
      scales[r * nb + b] = s16;
      const float sf = (float)half_to_double(s16);
      for (int i = 0; i < kBlock; ++i) {
        int8_t q = 0;
        if (sf != 0.f) {
          float v = std::rint(blk[i] / sf);
          v = std::fmin(std::fmax(v, -qmax), qmax);
          q = (int8_t)v;
        }
        codes[r * k + b * kBlock + i] = q;
      }
    }
  }
  return 0;
}

// FP4 ([F] Axis 1, lever 1c) with the integer types' block layout: s32 = m / 6,
// s16 = fp16(s32); the code of r = w / s16 (fp32 division) is e2m1_encode(r);
// s16 == 0 gives zero codes.  Codes returned one per byte (0..15).
int orc_quantize_fp4_block32(const float* w, int64_t n, int64_t k, uint8_t* codes, uint16_t* scales, int threads) {
  if (k % kBlock != 0) return 1;
  const int64_t nb = k / kBlock;
#pragma omp parallel for num_threads(threads_of(threads)) schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* blk = w + r * k + b * kBlock;
      float m = 0.f;
      for (int i = 0; i < kBlock; ++i) m = std::fmax(m, std::fabs(blk[i]));
      const uint16_t s16 = double_to_half((double)(m / 6.f));
      scales[r * nb + b] = s16;
      const float sf = (float)half_to_double(s16);
      for (int i = 0; i < kBlock; ++i)
        codes[r * k + b * kBlock + i] = sf == 0.f ? 0 : e2m1_encode(blk[i] / sf);
    }
  }
  return 0;
}

void orc_e2m1_values(const uint8_t* codes, int64_t count, double* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = e2m1_value(codes[i] & 15);
}
void orc_e2m1_encode(const float* r, int64_t count, uint8_t* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = e2m1_encode(r[i]);
}

// Two 4-bit codes per byte: byte i of a row holds element 2i in bits 0-3 and
// element 2i+1 in bits 4-7 (two's-complement nibbles for int4).
int orc_pack_nibbles(const uint8_t* codes, int64_t n, int64_t k, uint8_t* out) {
  if (k % 2 != 0) return 1;
  for (int64_t r = 0; r < n; ++r)
    for (int64_t i = 0; i < k / 2; ++i)
      out[r * (k / 2) + i] = (uint8_t)((codes[r * k + 2 * i] & 15) | ((codes[r * k + 2 * i + 1] & 15) << 4));
  return 0;
}
void orc_unpack_int4(const uint8_t* packed, int64_t n, int64_t k, int8_t* out) {
  for (int64_t r = 0; r < n; ++r)
    for (int64_t i = 0; i < k; ++i) {
      const int nib = (packed[r * (k / 2) + i / 2] >> (4 * (i & 1))) & 15;
      out[r * k + i] = (int8_t)(nib >= 8 ? nib - 16 : nib);
    }
}

// w[r][h] = q[r][h] * s16[r][h / 32] in float64.
void orc_dequantize(int kind, const void* codes, const uint16_t* scales, int64_t n, int64_t k, double* out) {
  for (int64_t r = 0; r < n; ++r)
    for (int64_t h = 0; h < k; ++h)
      out[r * k + h] = code_value(kind, codes, r * k + h) * half_to_double(scales[r * (k / kBlock) + h / kBlock]);
}

// ---- the dequantised GEMM ([V], [F] "Baseline byte model") --------------------
// y[s][r] (float64 [S][n]) for fp16 activations x [S][k].
int orc_dequant_gemm64(int kind, const void* codes, const uint16_t* scales, int64_t n, int64_t k,
                       const uint16_t* x, int S, double* y, int threads) {
  if (k % kBlock != 0 || S < 1) return 1;
  const std::vector<double> xd = widen_halves(x, (int64_t)S * k);
  gemm64(kind, codes, scales, n, k, xd.data(), S, y, threads);
  return 0;
}

// The same for float64 activations.
int orc_dequant_gemm64_x64(int kind, const void* codes, const uint16_t* scales, int64_t n, int64_t k,
                           const double* x, int S, double* y, int threads) {
  if (k % kBlock != 0 || S < 1) return 1;
  gemm64(kind, codes, scales, n, k, x, S, y, threads);
  return 0;
}

// ---- argmax, top-2 gap, accept ([D] "The delta") --------------------------------
// Per row: the largest value, ties to the lowest index (+0 and -0 are equal).
void orc_argmax_rows_f32(const float* v, int S, int64_t n, int32_t* out) {
  for (int s = 0; s < S; ++s) {
    int64_t best = 0;
    for (int64_t i = 1; i < n; ++i)
      if (v[(size_t)s * n + i] > v[(size_t)s * n + best]) best = i;
    out[s] = (int32_t)best;
  }
}

void orc_argmax_rows_f64(const double* v, int S, int64_t n, int32_t* out) {
  for (int s = 0; s < S; ++s) {
    int64_t best = 0;
    for (int64_t i = 1; i < n; ++i)
      if (v[(size_t)s * n + i] > v[(size_t)s * n + best]) best = i;
    out[s] = (int32_t)best;
  }
}

// Per row: the largest value minus the largest over the other indices (0 for a
// duplicated maximum; +inf for a single entry).
void orc_top2_gap(const double* v, int S, int64_t n, double* out) {
  for (int s = 0; s < S; ++s) {
    const double* row = v + (size_t)s * n;
    if (n < 2) {
      out[s] = INFINITY;
      continue;
    }
    int64_t best = 0;
    for (int64_t i = 1; i < n; ++i)
      if (row[i] > row[best]) best = i;
    double second = -INFINITY;
    for (int64_t i = 0; i < n; ++i)
      if (i != best && row[i] > second) second = row[i];
    out[s] = row[best] - second;
  }
}

// Greedy accept over one window [a0, d_1 .. d_{S-1}] ([D] "The delta",
// "Control-logic proof"; [V] "Hybrid state discipline"): argmax[i] is the
// target's token after window position i; draft i (drafts[i], the token at
// position i+1) is accepted iff every earlier draft was and drafts[i] ==
// argmax[i]; drafts at i >= n_valid are pad, never accepted.
// accepted = the accepted count j, next_a0 = argmax[j].
int orc_greedy_accept(const int32_t* argmax, int S, const int32_t* drafts, int n_valid, int32_t* accepted,
                      int32_t* next_a0) {
  if (S < 1 || n_valid < 0 || n_valid > S - 1) return 1;
  int j = 0;
  while (j < n_valid && drafts[j] == argmax[j]) ++j;
  *accepted = j;
  *next_a0 = argmax[j];
  return 0;
}

// Tree accept ([D] "Deferred / harder", the tree verify): node 0 is the root;
// node i > 0 carries tokens[i] below parent[i] (absent unless 0 <= parent[i] < i).
// Node i is accepted iff its parent is and tokens[i] == argmax[parent[i]].  The
// commit is the path to the deepest accepted node, the lowest index among
// equally deep ones: path[0 .. *depth-1] from the root's child down,
// next_a0 = argmax[that node].
int orc_tree_accept(const int32_t* argmax, int S, const int32_t* tokens, const int32_t* parent, int32_t* path,
                    int32_t* depth_out, int32_t* next_a0) {
  if (S < 1) return 1;
  std::vector<int> acc(S, 0), depth(S, 0);
  acc[0] = 1;
  for (int i = 1; i < S; ++i) {
    const int p = parent[i];
    if (p >= 0 && p < i && acc[p] && tokens[i] == argmax[p]) {
      acc[i] = 1;
      depth[i] = depth[p] + 1;
    }
  }
  int best = 0;
  for (int i = 1; i < S; ++i)
    if (acc[i] && depth[i] > depth[best]) best = i;
  *depth_out = depth[best];
  for (int i = best, d = depth[best]; i != 0; i = parent[i]) path[--d] = i;
  *next_a0 = argmax[best];
  return 0;
}

// The whole greedy verify of one window: logits (float64 GEMM rounded once to
// float32), per-row argmax of the float32 logits, the top-2 gap of the float64
// values, and the accept.  logits_or_null: float32 [S][n].
int orc_verify_head(int kind, const void* codes, const uint16_t* scales, int64_t n, int64_t k, const uint16_t* x,
                    int S, const int32_t* drafts, int n_valid, float* logits_or_null, int32_t* argmax, double* gap,
                    int32_t* accepted, int32_t* next_a0, int threads) {
  if (S < 1 || n_valid < 0 || n_valid > S - 1) return 1;
  std::vector<double> y((size_t)S * n);
  if (orc_dequant_gemm64(kind, codes, scales, n, k, x, S, y.data(), threads) != 0) return 1;
  std::vector<float> lf((size_t)S * n);
  for (size_t i = 0; i < lf.size(); ++i) lf[i] = (float)y[i];
  orc_argmax_rows_f32(lf.data(), S, n, argmax);
  orc_top2_gap(y.data(), S, n, gap);
  if (logits_or_null != nullptr) std::memcpy(logits_or_null, lf.data(), lf.size() * sizeof(float));
  return orc_greedy_accept(argmax, S, drafts, n_valid, accepted, next_a0);
}

// ---- SwiGLU ([F] Axis 4) ----------------------------------------------------------
void orc_silu(const double* t, int64_t count, double* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = silu(t[i]);
}

// h = SiLU(x G^T) * (x U^T), float64 [S][n]; h16 (when not null) = fp16(h),
// one rounding -- the dense projection's API output.
int orc_swiglu64(int kind, const void* g_codes, const uint16_t* g_scales, const void* u_codes,
                 const uint16_t* u_scales, int64_t n, int64_t k, const uint16_t* x, int S, double* h, uint16_t* h16,
                 int threads) {
  std::vector<double> u((size_t)S * n);
  if (orc_dequant_gemm64(kind, g_codes, g_scales, n, k, x, S, h, threads) != 0) return 1;
  if (orc_dequant_gemm64(kind, u_codes, u_scales, n, k, x, S, u.data(), threads) != 0) return 1;
  for (size_t i = 0; i < u.size(); ++i) h[i] = silu(h[i]) * u[i];
  if (h16 != nullptr)
    for (size_t i = 0; i < u.size(); ++i) h16[i] = double_to_half(h[i]);
  return 0;
}

// ---- gathered-expert MoE ([F] "Baseline byte model": top-8 of 256 routed experts) --
// Per row: the top_k experts by logit (larger first, ties to the lower id) and
// their weights softmax over the selected logits: exp(l - l_max) / sum, the sum
// over the selection in selection order.
int orc_route_topk(const float* logits, int S, int E, int top_k, int32_t* ids, double* w) {
  if (top_k < 1 || top_k > E) return 1;
  for (int s = 0; s < S; ++s) {
    const float* l = logits + (size_t)s * E;
    std::vector<int> taken(E, 0);
    for (int j = 0; j < top_k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;  // strict: the lower id keeps a tie
      taken[best] = 1;
      ids[s * top_k + j] = best;
    }
    const double lmax = (double)l[ids[s * top_k]];
    double sum = 0.0;
    for (int j = 0; j < top_k; ++j) {
      w[s * top_k + j] = std::exp((double)l[ids[s * top_k + j]] - lmax);
      sum += w[s * top_k + j];
    }
    for (int j = 0; j < top_k; ++j) w[s * top_k + j] /= sum;
  }
  return 0;
}

// Counting sort of the (row, slot) selections by expert; rows ascending within
// an expert: expert e owns entries offsets[e] .. offsets[e+1]-1 of rows / slots.
int orc_group_by_expert(const int32_t* ids, int S, int top_k, int E, int32_t* offsets, int32_t* rows,
                        int32_t* slots) {
  std::vector<int64_t> count(E, 0);
  for (int i = 0; i < S * top_k; ++i) {
    if (ids[i] < 0 || ids[i] >= E) return 1;
    ++count[ids[i]];
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + (int32_t)count[e];
  std::vector<int64_t> fill(offsets, offsets + E);
  for (int s = 0; s < S; ++s)
    for (int j = 0; j < top_k; ++j) {
      const int e = ids[s * top_k + j];
      rows[fill[e]] = s;
      slots[fill[e]] = j;
      ++fill[e];
    }
  return 0;
}

// One expert's SwiGLU MLP on R fp16 rows x [R][H]: h = SiLU(x G_e^T) * (x U_e^T)
// (float64 [R][I]), y = h D_e^T (float64 [R][H]).  Stacked weights: gate/up
// [E*I][H] (expert e owns rows e*I ..), down [E*H][I] (rows e*H ..).
int orc_expert_swiglu64(int kind, const void* gc, const uint16_t* gs, const void* uc, const uint16_t* us,
                        const void* dc, const uint16_t* ds, int e, int I, int H, const uint16_t* x, int R, double* y,
                        int threads) {
  const size_t cb = kind == 0 || kind == 1 ? 1 : sizeof(double);  // bytes per code
  const char* g = static_cast<const char*>(gc) + (size_t)e * I * H * cb;
  const char* u = static_cast<const char*>(uc) + (size_t)e * I * H * cb;
  const char* d = static_cast<const char*>(dc) + (size_t)e * H * I * cb;
  std::vector<double> h((size_t)R * I);
  if (orc_swiglu64(kind, g, gs + (size_t)e * I * (H / kBlock), u, us + (size_t)e * I * (H / kBlock), I, H, x, R,
                   h.data(), nullptr, threads) != 0)
    return 1;
  return orc_dequant_gemm64_x64(kind, d, ds + (size_t)e * H * (I / kBlock), H, I, h.data(), R, y, threads);
}

// out[s] = sum over the row's selections j (selection order) of
// w[s][j] * expert_swiglu(x[s]) of expert ids[s][j], float64, rounded once to float32.
int orc_moe_forward(int kind, const void* gc, const uint16_t* gs, const void* uc, const uint16_t* us, const void* dc,
                    const uint16_t* ds, int E, int I, int H, int top_k, const uint16_t* x, const float* router, int S,
                    float* out, int32_t* ids, double* w, int threads) {
  if (orc_route_topk(router, S, E, top_k, ids, w) != 0) return 1;
  std::vector<double> acc((size_t)H), y((size_t)H);
  for (int s = 0; s < S; ++s) {
    for (int c = 0; c < H; ++c) acc[c] = 0.0;
    for (int j = 0; j < top_k; ++j) {
      if (orc_expert_swiglu64(kind, gc, gs, uc, us, dc, ds, ids[s * top_k + j], I, H, x + (size_t)s * H, 1,
                              y.data(), threads) != 0)
        return 1;
      for (int c = 0; c < H; ++c) acc[c] += w[s * top_k + j] * y[c];
    }
    for (int c = 0; c < H; ++c) out[(size_t)s * H + c] = (float)acc[c];
  }
  return 0;
}

// ---- sampling verify ([D] "Deferred / harder"; speculative sampling, Leviathan,
// Kalman & Matias, ICML 2023, with a drafter that proposes each token
// deterministically) -------------------------------------------------------------
uint64_t orc_mix(uint64_t z) { return mix64(z); }
void orc_mix_array(const uint64_t* z, int64_t count, uint64_t* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = mix64(z[i]);
}
uint64_t orc_rng_key(uint64_t seed, uint64_t counter) { return mix64(seed + (counter + 1) * kGolden); }
void orc_uniforms(uint64_t key, const uint64_t* idx, int64_t count, double* out) {
  for (int64_t i = 0; i < count; ++i) out[i] = uniform_of(key, idx[i]);
}
// Gumbel noise [S][V]: row i, entry v uses element 32 v + i.
void orc_gumbel(uint64_t key, int S, int64_t V, double* out) {
  for (int i = 0; i < S; ++i)
    for (int64_t v = 0; v < V; ++v) out[(size_t)i * V + v] = gumbel_of(uniform_of(key, kMaxRows * (uint64_t)v + i));
}

// One window: p_i = softmax(L_i / T); each row's draw samples[i] = argmax of
// L_i / T + g_i (ties to the lower entry; Gumbel-max); draft i is kept iff
// u_i < p_i(d_i) with u_i = element 32 V + i; at the first rejection (row j) the
// token is the argmax over v != d_j (a draw from the residual distribution),
// if every draft is kept it is samples[n_valid].  Also returns, for the
// tolerance decisions of the parity tests: p_draft [n_valid], u [S], z_gap [S]
// (top-2 gap of L/T + g), z_gap_res [S] (the same without the draft's entry, for
// the rows the scan read; +inf elsewhere), *u_margin (the smallest |u_i - p_i(d_i)|
// over those rows) and probs [S][V] when not null.
int orc_verify_sample(const double* logits, int S, int64_t V, const int32_t* drafts, int n_valid, double temperature,
                      uint64_t seed, uint64_t counter, int32_t* accepted, int32_t* token, int32_t* samples,
                      double* p_draft, double* u, double* z_gap, double* z_gap_res, double* u_margin, double* probs) {
  if (!(temperature > 0.0) || S < 1 || S > (int)kMaxRows || n_valid < 0 || n_valid > S - 1) return 1;
  const uint64_t key = orc_rng_key(seed, counter);
  std::vector<double> z((size_t)S * V), l((size_t)S * V);
  for (int i = 0; i < S; ++i)
    for (int64_t v = 0; v < V; ++v) {
      const size_t o = (size_t)i * V + v;
      l[o] = logits[o] / temperature;
      z[o] = l[o] + gumbel_of(uniform_of(key, kMaxRows * (uint64_t)v + i));
    }
  for (int i = 0; i < S; ++i) u[i] = uniform_of(key, kMaxRows * (uint64_t)V + i);
  auto first_argmax = [&](const double* row, int64_t skip) {
    int64_t best = -1;
    for (int64_t v = 0; v < V; ++v)
      if (v != skip && (best < 0 || row[v] > row[best])) best = v;
    return best;
  };
  // largest minus second largest over the entries v != skip (0 for a duplicated
  // maximum; +inf with fewer than two entries)
  auto gap_of = [&](const double* row, int64_t skip) {
    double a = -INFINITY, b = -INFINITY;
    int64_t entries = 0;
    for (int64_t v = 0; v < V; ++v) {
      if (v == skip) continue;
      ++entries;
      if (row[v] > a) {
        b = a;
        a = row[v];
      } else if (row[v] > b) {
        b = row[v];
      }
    }
    return entries < 2 ? INFINITY : a - b;
  };
  for (int i = 0; i < S; ++i) {
    samples[i] = (int32_t)first_argmax(&z[(size_t)i * V], -1);
    z_gap[i] = gap_of(&z[(size_t)i * V], -1);
    z_gap_res[i] = INFINITY;
  }
  std::vector<double> p((size_t)V);
  for (int i = 0; i < S; ++i) {
    const double* li = &l[(size_t)i * V];
    double m = li[0];
    for (int64_t v = 1; v < V; ++v) m = std::fmax(m, li[v]);
    double sum = 0.0;
    for (int64_t v = 0; v < V; ++v) sum += (p[v] = std::exp(li[v] - m));
    for (int64_t v = 0; v < V; ++v) p[v] /= sum;
    if (i < n_valid) p_draft[i] = p[drafts[i]];
    if (probs != nullptr) std::memcpy(probs + (size_t)i * V, p.data(), (size_t)V * sizeof(double));
  }
  int j = n_valid;
  int32_t tok = samples[n_valid];
  double margin = INFINITY;
  for (int i = 0; i < n_valid; ++i) {
    margin = std::fmin(margin, std::fabs(u[i] - p_draft[i]));
    const double* zi = &z[(size_t)i * V];
    z_gap_res[i] = gap_of(zi, drafts[i]);
    if (!(u[i] < p_draft[i])) {
      j = i;
      tok = (int32_t)first_argmax(zi, drafts[i]);
      break;
    }
  }
  *accepted = j;
  *token = tok;
  *u_margin = margin;
  return 0;
}

}  // extern "C"
