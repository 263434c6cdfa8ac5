// Device-side gating pieces shared by the gating kernel (routing.cu) and the
// fused small-batch routing kernel (align.cu).
// mlc-llm moe_misc.py, gating_topk / gating_softmax_topk.
#pragma once

#include <float.h>

#include "common.cuh"

namespace moe {
namespace gate {

constexpr int kNone = 0x7fffffff;   // "no candidate" index

// (value, index) order of the page's top-k: larger value first; equal values
// keep the lower expert index first. kNone loses to everything.
__device__ __forceinline__ bool better(float av, int ai, float bv, int bi) {
  if (ai == kNone) return false;
  if (bi == kNone) return true;
  return av > bv || (av == bv && ai < bi);
}

// Lanes of this thread's group of L (L a power of two, groups aligned in the warp).
template <int L>
__device__ __forceinline__ unsigned group_mask() {
  if constexpr (L == 32) {
    return 0xffffffffu;
  } else {
    const unsigned lane = threadIdx.x & 31;
    return ((1u << L) - 1u) << (lane & ~(unsigned)(L - 1));
  }
}

// exp(a - b) with the rounding error of the float subtraction folded back in
// (a - b = s + err exactly, exp(s + err) ~= exp(s) * (1 + err)).
__device__ __forceinline__ float exp_diff(float a, float b) {
  const float s = a - b;
  const float bb = s - a;
  const float err = (a - (s - bb)) + (-b - bb);
  const float e = expf(s);
  return fmaf(e, err, e);
}

// Order-preserving map of a finite float to an unsigned key (larger float ->
// larger key; -0 and +0 share a key; 0 is below every finite float's key).
__device__ __forceinline__ unsigned okey(float x) {
  const unsigned u = __float_as_uint(x + 0.0f);   // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float okey_value(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// (hi, lo) += x with the rounding error of the add kept in lo (TwoSum).
__device__ __forceinline__ void two_sum_add(float& hi, float& lo, float x) {
  const float s = hi + x;
  const float bb = s - hi;
  lo += (hi - (s - bb)) + (x - bb);
  hi = s;
}

// One arg-max round over the 32 lanes of a warp, each holding V candidates
// (expert g + 32 i, key 0 = none): largest key, then lowest expert among equal
// keys. Returns the winning expert (every lane gets it) and its key in *kout.
template <int V>
__device__ __forceinline__ int warp_argmax_round(const unsigned (&key)[V], unsigned taken, int g,
                                                 unsigned* kout) {
  unsigned best = 0;
#pragma unroll
  for (int i = 0; i < V; ++i)
    if (!((taken >> i) & 1u)) best = max(best, key[i]);
  const unsigned m = __reduce_max_sync(0xffffffffu, best);
  unsigned cand = 0xffffffffu;
#pragma unroll
  for (int i = V - 1; i >= 0; --i)
    if (!((taken >> i) & 1u) && key[i] == m) cand = (unsigned)(g + 32 * i);
  *kout = m;
  return (int)__reduce_min_sync(0xffffffffu, cand);
}

// Top-k and softmax of one token's logits row, by the L lanes of a group
// (lane g of the group holds experts g, g + L, ...; E <= L * V, k <= L).
// Lane j < k of the group writes output slot j. The softmax denominator is a
// compensated float32 sum; each weight is one correctly rounded division.
template <int L, int V>
__device__ __forceinline__ void gate_one_token(const float* __restrict__ logits, long t, int E, int k,
                                               int norm, float* __restrict__ w_out,
                                               int32_t* __restrict__ idx_out) {
  const int g = threadIdx.x & (L - 1);
  const unsigned gm = group_mask<L>();
  const float* row = logits + t * (long)E;
  float v[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = g + i * L;
    v[i] = e < E ? __ldg(row + e) : 0.0f;
  }
  unsigned taken = 0;
#pragma unroll
  for (int i = 0; i < V; ++i)
    if (g + i * L >= E) taken |= 1u << i;

  float my_v = 0.0f, row_max = 0.0f;
  int my_i = -1;
  if constexpr (L == 32) {
    unsigned key[V];
#pragma unroll
    for (int i = 0; i < V; ++i) key[i] = okey(v[i]);
    for (int j = 0; j < k; ++j) {
      unsigned m;
      const int bi = warp_argmax_round<V>(key, taken, g, &m);
      if ((bi & 31) == g) taken |= 1u << (bi >> 5);
      const float bv = okey_value(m);
      if (j == 0) row_max = bv;
      if (g == j) { my_v = bv; my_i = bi; }
    }
  } else {
    for (int j = 0; j < k; ++j) {
      float bv = 0.0f;
      int bi = kNone;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int e = g + i * L;
        if (!((taken >> i) & 1u) && better(v[i], e, bv, bi)) { bv = v[i]; bi = e; }
      }
#pragma unroll
      for (int off = L / 2; off >= 1; off >>= 1) {
        const float ov = __shfl_xor_sync(gm, bv, off, L);
        const int oi = __shfl_xor_sync(gm, bi, off, L);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if ((bi & (L - 1)) == g) taken |= 1u << (bi / L);
      if (j == 0) row_max = bv;
      if (g == j) { my_v = bv; my_i = bi; }
    }
  }

  // denominator: the k selected (norm) or the whole row
  float hi = 0.0f, lo = 0.0f;
  if (norm) {
    if (g < k) hi = exp_diff(my_v, row_max);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (g + i * L < E) two_sum_add(hi, lo, exp_diff(v[i], row_max));
  }
#pragma unroll
  for (int off = L / 2; off >= 1; off >>= 1) {
    const float ohi = __shfl_xor_sync(gm, hi, off, L);
    const float olo = __shfl_xor_sync(gm, lo, off, L);
    two_sum_add(hi, lo, ohi);
    lo += olo;
  }

  if (g < k) {
    const float num = exp_diff(my_v, row_max);
    w_out[t * k + g] = __fdiv_rn(num, hi + lo);
    idx_out[t * k + g] = my_i;
  }
}

}  // namespace gate
}  // namespace moe

// Dispatch on E: L lanes per row, V = ceil(E / L) values per lane.
#define MOE_DISPATCH_LV(E, FN, ...)                                        \
  do {                                                                     \
    if ((E) <= 1) return FN<1, 1>(__VA_ARGS__);                            \
    if ((E) <= 2) return FN<2, 1>(__VA_ARGS__);                            \
    if ((E) <= 4) return FN<4, 1>(__VA_ARGS__);                            \
    if ((E) <= 8) return FN<8, 1>(__VA_ARGS__);                            \
    if ((E) <= 16) return FN<16, 1>(__VA_ARGS__);                          \
    if ((E) <= 32) return FN<32, 1>(__VA_ARGS__);                          \
    if ((E) <= 64) return FN<32, 2>(__VA_ARGS__);                          \
    if ((E) <= 128) return FN<32, 4>(__VA_ARGS__);                         \
    if ((E) <= 256) return FN<32, 8>(__VA_ARGS__);                         \
    if ((E) <= 512) return FN<32, 16>(__VA_ARGS__);                        \
    return FN<32, 32>(__VA_ARGS__);                                        \
  } while (0)
