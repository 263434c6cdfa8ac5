// Expert-parallel exchange: the index work on both sides of the two
// all-to-all steps when each of G ranks owns E/G consecutive experts.
//
// Megatron-LM fused_indices_converter.py, _indices_to_multihot_kernel masks
// the indices to a rank's local experts (idx < num_of_local_experts); the
// grouped FFN each owner runs is project_6 moe_expert_gemm.cpp
// moe_prefill_experts on the rows routed to its experts, and the weighted sum
// over k is mlc-llm moe_misc.py scatter_output + moe_sum.
//
// Sender: the align step orders slots expert-major, so the rows for owner r
// are the contiguous range [offsets[E_r.lo], offsets[E_r.hi]) of x_sorted
// (moe_gather_rows writes it); they go out in rank order.
//
// Receiver: the rows arrive source-major (all of source 0, then source 1, ...),
// each source's rows expert-major. ep_receive_index turns the G x E_local table
// of counts into the local counts / exclusive offsets and the permutation
// perm[p] (expert-major position p -> received row), expert-major with the
// sources in rank order inside an expert. The grouped FFN then runs with k = 1
// on the received rows, gathering through perm and writing each result back to
// the received row it came from (reverse = perm), so the returned rows are in
// the layout they arrived in.
//
// Return: the y rows come back in the sender's x_sorted order; ep_combine
// inverts `reverse` (pos[slot] = sorted row) and forms
// out[t] = sum_j w[t, j] * y[pos[t*k + j]] in fp32, j ascending, rounded once.
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kTabThreads = 1024;

// One CTA: block starts of every (source g, local expert e) in both layouts
// (ws: src_start[B], dst_start[B], B = G * El, flat index g * El + e), local
// counts [El] and exclusive offsets [El + 1].
__global__ void __launch_bounds__(kTabThreads) ep_tables_kernel(const int32_t* __restrict__ rc, int G, int El,
                                                                int32_t* __restrict__ src_start,
                                                                int32_t* __restrict__ dst_start,
                                                                int32_t* __restrict__ counts,
                                                                int32_t* __restrict__ offsets) {
  extern __shared__ int32_t sh[];   // [El] column sums, then [El + 1] offsets
  int32_t* col = sh;
  int32_t* off = sh + El;
  const int tid = threadIdx.x;
  for (int e = tid; e < El; e += blockDim.x) {
    int s = 0;
    for (int g = 0; g < G; ++g) s += __ldg(rc + (long)g * El + e);
    col[e] = s;
    counts[e] = s;
  }
  __syncthreads();
  if (tid == 0) {   // El <= a few thousand: a serial scan is cheap next to the exchange
    int acc = 0;
    for (int e = 0; e < El; ++e) {
      off[e] = acc;
      acc += col[e];
    }
    off[El] = acc;
  }
  __syncthreads();
  for (int e = tid; e <= El; e += blockDim.x) offsets[e] = off[e];
  // expert-major position of block (g, e): off[e] + sum of the same expert's blocks of earlier sources
  for (int e = tid; e < El; e += blockDim.x) {
    int acc = off[e];
    for (int g = 0; g < G; ++g) {
      dst_start[g * El + e] = acc;
      acc += __ldg(rc + (long)g * El + e);
    }
  }
  // source-major position: a running sum over the flat (g, e) order, one source per thread
  for (int g = tid; g < G; g += blockDim.x) {
    int acc = 0;
    for (int g2 = 0; g2 < g; ++g2)
      for (int e = 0; e < El; ++e) acc += __ldg(rc + (long)g2 * El + e);
    for (int e = 0; e < El; ++e) {
      src_start[g * El + e] = acc;
      acc += __ldg(rc + (long)g * El + e);
    }
  }
}

// CTA b fills perm for block b = (g, e).
__global__ void __launch_bounds__(256) ep_fill_perm_kernel(const int32_t* __restrict__ rc,
                                                           const int32_t* __restrict__ src_start,
                                                           const int32_t* __restrict__ dst_start,
                                                           int32_t* __restrict__ perm) {
  const int b = blockIdx.x;
  const int n = __ldg(rc + b), s0 = __ldg(src_start + b), d0 = __ldg(dst_start + b);
  for (int i = threadIdx.x; i < n; i += blockDim.x) perm[d0 + i] = s0 + i;
}

// pos[reverse[p]] = p for the routed rows p < offsets[E] (pos was set to -1).
__global__ void __launch_bounds__(256) ep_invert_kernel(const int32_t* __restrict__ reverse,
                                                        const int32_t* __restrict__ offsets, int E,
                                                        int32_t* __restrict__ pos) {
  const int n = __ldg(offsets + E);
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < n; p += gridDim.x * blockDim.x) pos[__ldg(reverse + p)] = p;
}

template <class T>
struct Vec;   // 16 bytes of T widened to float
template <>
struct Vec<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void load(const void* p, float (&v)[4]) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  }
  static __device__ __forceinline__ void store(void* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void load(const void* p, float (&v)[8]) {
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ uint32_t pack(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  static __device__ __forceinline__ void store(void* p, const float (&v)[8]) {
    *reinterpret_cast<uint4*>(p) = make_uint4(pack(v[0], v[1]), pack(v[2], v[3]), pack(v[4], v[5]), pack(v[6], v[7]));
  }
};

// out[t] = sum_j w[t,j] * y[pos[t*k+j]] (dropped slots, pos < 0, add nothing); one
// thread per 16 bytes of an output row.
template <class T>
__global__ void __launch_bounds__(256) ep_combine_kernel(const T* __restrict__ y, const float* __restrict__ w,
                                                         const int32_t* __restrict__ pos, long n_tok, int k, int HV,
                                                         T* __restrict__ out, int sh) {
  constexpr int N = Vec<T>::N;
  const long n = n_tok * HV;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const long t = div_idx(i, HV, sh);
    const int c = (int)(i - t * HV);
    float acc[N], v[N];
#pragma unroll
    for (int q = 0; q < N; ++q) acc[q] = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int p = __ldg(pos + t * k + j);
      if (p < 0) continue;
      const float wj = __ldg(w + t * k + j);
      Vec<T>::load(y + ((long)p * HV + c) * N, v);
#pragma unroll
      for (int q = 0; q < N; ++q) acc[q] += wj * v[q];
    }
    Vec<T>::store(out + i * N, acc);
  }
}

}  // namespace

size_t ep_receive_workspace_bytes(int G, int El) { return (size_t)2 * G * El * sizeof(int32_t); }

int launch_ep_receive_index(const int32_t* recv_counts, int G, int El, int32_t* counts, int32_t* offsets,
                            int32_t* perm, void* ws, cudaStream_t s) {
  int32_t* src_start = static_cast<int32_t*>(ws);
  int32_t* dst_start = src_start + (long)G * El;
  {
    ProfScope ps("ep_receive_tables", s);
    const size_t smem = (size_t)(2 * El + 1) * sizeof(int32_t);
    if (int rc = ensure_smem_limit(ep_tables_kernel, smem, "ep_receive_index")) return rc;
    ep_tables_kernel<<<1, kTabThreads, smem, s>>>(recv_counts, G, El, src_start, dst_start, counts, offsets);
    if (int rc = check_launch("ep_receive_index")) return rc;
  }
  ProfScope ps("ep_receive_perm", s);
  ep_fill_perm_kernel<<<G * El, 256, 0, s>>>(recv_counts, src_start, dst_start, perm);
  return check_launch("ep_receive_index");
}

int launch_ep_combine(const void* y, const float* w, const int32_t* reverse, const int32_t* offsets, int dtype,
                      int T, int k, int H, int E, void* out, int32_t* pos, cudaStream_t s) {
  const long S = (long)T * k;
  const int esz = dtype == MOE_F32 ? 4 : 2;
  if ((long)H * esz % 16 != 0) return fail(MOE_ERR_UNSUPPORTED, "ep_combine: rows of %ld bytes (need a multiple of 16)",
                                           (long)H * esz);
  ProfScope ps("ep_combine", s);
  cudaError_t e = cudaMemsetAsync(pos, 0xff, (size_t)S * sizeof(int32_t), s);   // -1: slot not routed
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "ep_combine: %s", cudaGetErrorString(e));
  const int g1 = (int)std::max(1L, std::min((long)num_sms() * 4, (S + 255) / 256));
  ep_invert_kernel<<<g1, 256, 0, s>>>(reverse, offsets, E, pos);
  if (int rc = check_launch("ep_combine")) return rc;
  const int HV = H * esz / 16;
  const long units = (long)T * HV;
  const int g2 = (int)std::max(1L, std::min((long)num_sms() * 8, (units + 255) / 256));
  if (dtype == MOE_F32)
    ep_combine_kernel<float><<<g2, 256, 0, s>>>(static_cast<const float*>(y), w, pos, (long)T, k, HV,
                                                static_cast<float*>(out), pow2_shift(HV));
  else
    ep_combine_kernel<__nv_bfloat16><<<g2, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(y), w, pos, (long)T, k,
                                                        HV, static_cast<__nv_bfloat16*>(out), pow2_shift(HV));
  return check_launch("ep_combine");
}

}  // namespace moe
