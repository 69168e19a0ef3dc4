#pragma once
// Routing of the gathered-expert MoE ("Flagship dramatic-speedup plan -- the
// full stackable tuning set", section "Baseline byte model": routed experts
// through gather_qmm, top-8 of 256): the top k of a row's router logits (larger
// logit first, ties to the lower expert id) and their softmax-renormalised
// weights.  Shared by the routing kernel and by the MoE gate/up launch that
// routes the window in its own prologue.
#include <cstdint>

#include "sdv_device.cuh"

namespace sdv {

// Order-preserving 32-bit key of a routing logit: a larger logit has a larger
// key, -0 and +0 share one key (they compare equal), and NaN sorts below -inf.
__device__ __forceinline__ uint32_t route_key(float v) {
  if (v != v) return 0u;
  const uint32_t u = __float_as_uint(v + 0.f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float route_key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One warp routes one row of E logits (E <= 32 SLOTS): its lanes hold the
// experts lane + 32 m in registers, each lane keeps its best untaken expert, and
// every selection round is one warp max over the keys plus one warp min over the
// ids of the lanes holding that key.  On return (after a __syncwarp) ids[i] and
// w[i], i < top_k, hold the i-th pick and its weight
// exp(l_i - l_0) / sum_j exp(l_j - l_0); `ids` and `w` are the row's arrays in
// shared memory.
template <int SLOTS>
__device__ __forceinline__ void route_row(const float* __restrict__ row, int E, int top_k, int lane, int* ids,
                                          float* w) {
  uint32_t key[SLOTS];
  int idx[SLOTS];  // slot m of key[] holds expert lane + 32 idx[m]
#pragma unroll
  for (int m = 0; m < SLOTS; ++m) {
    const int e = lane + 32 * m;
    key[m] = (e < E) ? route_key(__ldg(row + e)) : 0u;
    idx[m] = m;
  }
  // With up to 8 experts a lane sorts its list once (key descending, then id
  // ascending; a bitonic network on registers) and each pick pops the head;
  // with more, the lane recomputes its best untaken expert after each pick.
  constexpr bool kSorted = SLOTS <= 8;
  if (kSorted) {
#pragma unroll
    for (int k = 2; k <= SLOTS; k <<= 1)
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
        for (int i = 0; i < SLOTS; ++i) {
          const int l = i ^ j;
          if (l <= i) continue;
          // in the block (i & k) == 0 the better entry goes first, else last
          const bool l_better = key[l] > key[i] || (key[l] == key[i] && idx[l] < idx[i]);
          const bool swap = ((i & k) == 0) ? l_better : !l_better;
          const uint32_t ki = key[i], kl = key[l];
          const int ii = idx[i], il = idx[l];
          key[i] = swap ? kl : ki;
          key[l] = swap ? ki : kl;
          idx[i] = swap ? il : ii;
          idx[l] = swap ? ii : il;
        }
  }
  uint32_t taken = 0u;
  // the lane's best untaken expert: highest key, then lowest m (= lowest id)
  auto local_best = [&](uint32_t& bk, int& bm) {
    if (kSorted) {
      bk = key[0];
      bm = (lane + 32 * idx[0] < E) ? idx[0] : -1;
      return;
    }
    bk = 0u;
    bm = -1;
#pragma unroll
    for (int m = 0; m < SLOTS; ++m) {
      const bool live = (lane + 32 * m < E) && !((taken >> m) & 1u);
      if (live && (bm < 0 || key[m] > bk)) {
        bk = key[m];
        bm = m;
      }
    }
  };
  uint32_t bk;
  int bm;
  local_best(bk, bm);
  float first = 0.f;
  for (int i = 0; i < top_k; ++i) {
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bm >= 0 ? bk : 0u);
    const unsigned cand = (bm >= 0 && bk == kmax) ? (unsigned)(lane + 32 * bm) : 0xFFFFFFFFu;
    const int win = (int)__reduce_min_sync(0xffffffffu, cand);
    const float v = route_key_value(kmax);
    if (i == 0) first = v;
    if (lane == 0) {
      ids[i] = win;
      w[i] = v;
    }
    if ((win & 31) == lane) {
      if (kSorted) {  // pop the head
#pragma unroll
        for (int m = 0; m + 1 < SLOTS; ++m) {
          key[m] = key[m + 1];
          idx[m] = idx[m + 1];
        }
        key[SLOTS - 1] = 0u;
        idx[SLOTS - 1] = SLOTS;  // expert lane + 32 SLOTS >= E: never live
      } else {
        taken |= 1u << (win >> 5);
      }
      local_best(bk, bm);
    }
  }
  __syncwarp();
  // softmax over the selection (the first selected logit is the largest)
  float sum = 0.f;
  for (int i = 0; i < top_k; ++i) sum += expf(w[i] - first);
  __syncwarp();
  if (lane < top_k) w[lane] = expf(w[lane] - first) / sum;
  __syncwarp();
}

}  // namespace sdv
