// Routing kernels: gating softmax-top-k, indices -> multihot, multihot -> indices.
//
// gating: mlc-llm moe_misc.py, gating_topk / gating_softmax_topk.
// multihot: Megatron-LM fused_indices_converter.py, _indices_to_multihot_kernel
//           and _multihot_to_indices_kernel.
//
// Layout: a token's row is handled by a group of L lanes (L = next power of two
// of E, capped at 32), so small-E rows pack several tokens per warp and every
// row is read with coalesced loads (lane g holds experts g, g+L, g+2L, ...).
#include <float.h>
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kBlock = 256;
constexpr int kNone = 0x7fffffff;   // "no candidate" index

// (value, index) order of the page's top-k: larger value first; equal values
// keep the lower expert index first. kNone loses to everything.
__device__ __forceinline__ bool better(float av, int ai, float bv, int bi) {
  if (ai == kNone) return false;
  if (bi == kNone) return true;
  return av > bv || (av == bv && ai < bi);
}

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

template <int L, int V>
__global__ void __launch_bounds__(kBlock) gating_kernel(const float* __restrict__ logits, int T,
                                                        int E, int k, int norm,
                                                        float* __restrict__ w_out,
                                                        int32_t* __restrict__ idx_out) {
  const int g = threadIdx.x & (L - 1);
  const long t = (long)blockIdx.x * (kBlock / L) + threadIdx.x / L;
  if (t >= T) return;   // whole groups leave together
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

  // denominator: the k selected (norm) or the whole row, summed in double
  double part = 0.0;
  if (norm) {
    if (g < k) part = (double)exp_diff(my_v, row_max);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (g + i * L < E) part += (double)exp_diff(v[i], row_max);
  }
#pragma unroll
  for (int off = L / 2; off >= 1; off >>= 1) part += __shfl_xor_sync(gm, part, off, L);

  if (g < k) {
    const float num = exp_diff(my_v, row_max);
    w_out[t * k + g] = (float)((double)num / part);
    idx_out[t * k + g] = my_i;
  }
}

template <int L, int V>
int launch_gating_t(const float* logits, int T, int E, int k, int norm, float* w, int32_t* idx,
                    cudaStream_t s) {
  const int tpb = kBlock / L;
  const int grid = (T + tpb - 1) / tpb;
  gating_kernel<L, V><<<grid, kBlock, 0, s>>>(logits, T, E, k, norm, w, idx);
  return check_launch("gating_softmax_topk");
}

// ---------------------------------------------------------------------------
// indices -> multihot: one thread writes 4 consecutive experts of one row.

__global__ void __launch_bounds__(kBlock) indices_to_multihot_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ probs, int T, int k, int E,
    uint8_t* __restrict__ mh, float* __restrict__ pm, int32_t* __restrict__ pos) {
  const int E4 = (E + 3) >> 2;
  const long tid = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (tid >= (long)T * E4) return;
  const long t = tid / E4;
  const int e0 = (int)(tid - t * E4) * 4;
  unsigned m[4] = {0, 0, 0, 0};
  float p[4] = {0.f, 0.f, 0.f, 0.f};
  int q[4] = {-1, -1, -1, -1};
  for (int j = k - 1; j >= 0; --j) {       // descending, so the lowest j is kept on a repeat
    const int e = __ldg(idx + t * k + j);
    const int d = e - e0;
    if (e >= 0 && e < E && d >= 0 && d < 4) {
      m[d] = 1;
      p[d] = __ldg(probs + t * k + j);
      q[d] = j;
    }
  }
  const long base = t * (long)E + e0;
  if ((E & 3) == 0) {
    *reinterpret_cast<uchar4*>(mh + base) = make_uchar4(m[0], m[1], m[2], m[3]);
    *reinterpret_cast<float4*>(pm + base) = make_float4(p[0], p[1], p[2], p[3]);
    *reinterpret_cast<int4*>(pos + base) = make_int4(q[0], q[1], q[2], q[3]);
  } else {
    for (int d = 0; d < 4 && e0 + d < E; ++d) {
      mh[base + d] = (uint8_t)m[d];
      pm[base + d] = p[d];
      pos[base + d] = q[d];
    }
  }
}

// ---------------------------------------------------------------------------
// multihot -> indices: a group of L lanes per row; each output slot is written
// once, by the lane that owns its expert or (unfilled) by lane j % L.

template <int L, int V>
__global__ void __launch_bounds__(kBlock) multihot_to_indices_kernel(
    const float* __restrict__ pm, const int32_t* __restrict__ pos, int T, int E, int k,
    float* __restrict__ probs, int32_t* __restrict__ idx_out) {
  const int g = threadIdx.x & (L - 1);
  const long t = (long)blockIdx.x * (kBlock / L) + threadIdx.x / L;
  if (t >= T) return;
  const unsigned gm = group_mask<L>();
  unsigned filled = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = g + i * L;
    if (e < E) {
      const int p = __ldg(pos + t * E + e);
      if (p >= 0 && p < k) {
        probs[t * k + p] = __ldg(pm + t * E + e);
        if (idx_out) idx_out[t * k + p] = e;
        filled |= 1u << p;
      }
    }
  }
#pragma unroll
  for (int off = L / 2; off >= 1; off >>= 1) filled |= __shfl_xor_sync(gm, filled, off, L);
  for (int j = g; j < k; j += L) {
    if (!((filled >> j) & 1u)) {
      probs[t * k + j] = 0.0f;
      if (idx_out) idx_out[t * k + j] = -1;
    }
  }
}

template <int L, int V>
int launch_m2i_t(const float* pm, const int32_t* pos, int T, int E, int k, float* probs,
                 int32_t* idx, cudaStream_t s) {
  const int tpb = kBlock / L;
  multihot_to_indices_kernel<L, V><<<(T + tpb - 1) / tpb, kBlock, 0, s>>>(pm, pos, T, E, k, probs, idx);
  return check_launch("multihot_to_indices");
}

}  // namespace

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

int launch_gating(const float* logits, int T, int E, int k, int norm, float* w, int32_t* idx,
                  cudaStream_t s) {
  if (T == 0) return MOE_OK;
  ProfScope ps("gating_softmax_topk", s);
  MOE_DISPATCH_LV(E, launch_gating_t, logits, T, E, k, norm, w, idx, s);
}

int launch_indices_to_multihot(const int32_t* idx, const float* probs, int T, int k, int E,
                               uint8_t* mh, float* pm, int32_t* pos, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  ProfScope ps("indices_to_multihot", s);
  const long n = (long)T * ((E + 3) / 4);
  indices_to_multihot_kernel<<<(unsigned)((n + kBlock - 1) / kBlock), kBlock, 0, s>>>(
      idx, probs, T, k, E, mh, pm, pos);
  return check_launch("indices_to_multihot");
}

int launch_multihot_to_indices(const float* pm, const int32_t* pos, int T, int E, int k,
                               float* probs, int32_t* idx, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  ProfScope ps("multihot_to_indices", s);
  MOE_DISPATCH_LV(E, launch_m2i_t, pm, pos, T, E, k, probs, idx, s);
}

}  // namespace moe
