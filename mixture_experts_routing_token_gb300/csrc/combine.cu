// Weighted combine: out[t] = sum_{j<k} staging[t*k + j], j ascending, fp32,
// one rounding to the output dtype.
// mlc-llm moe_misc.py moe_sum (sum of the [T, k, H] expert outputs over k);
// the routing weight was already applied by the FC2 epilogue. The staging rows
// are float32 (CUDA-core and decode paths, backward) or bfloat16 (tensor-core
// prefill path: the weighted slot rows in the hidden dtype, as project_6
// moe_prefill_experts accumulates them; the sum over k stays fp32).
// HBM-bound streaming kernel: 16-byte loads, one thread per 16 bytes of each
// of the token's k rows. Launched with programmatic dependency on the FC2
// kernel (waits before reading).
#include <algorithm>
#include <type_traits>

#include "common.cuh"

namespace moe {
namespace {

// One 16-byte vector of the staging dtype, widened to float.
template <class InT>
struct Vec16;
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void load(const void* p, float (&v)[4]) {
    const float4 x = __ldcs(reinterpret_cast<const float4*>(p));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  }
};
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void load(const void* p, float (&v)[8]) {
    const uint4 x = __ldcs(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // bf16 -> f32 is exact: the bits move to the high half
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

template <class OutT, int N>
__device__ __forceinline__ void store_out(OutT* o, const float (&v)[N]);
template <>
__device__ __forceinline__ void store_out<float, 4>(float* o, const float (&v)[4]) {
  *reinterpret_cast<float4*>(o) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void store_out<float, 8>(float* o, const float (&v)[8]) {
  reinterpret_cast<float4*>(o)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(o)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16, 4>(__nv_bfloat16* o, const float (&v)[4]) {
  *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]));
}
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16, 8>(__nv_bfloat16* o, const float (&v)[8]) {
  *reinterpret_cast<uint4*>(o) =
      make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
}

// One thread per N = 16 / sizeof(InT) columns of a token (HV = H / N units per row).
// K > 0: k == K known at compile time, and all K loads are issued before the sum
// (the same j order); K == 0: any k.
template <class InT, class OutT, int K>
__global__ void __launch_bounds__(256) combine_vec_kernel(const InT* __restrict__ staging, long T, int k,
                                                          int HV, OutT* __restrict__ out, int sh) {
  constexpr int N = Vec16<InT>::N;
  pdl_wait();
  pdl_trigger();
  const long n = T * HV;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const long t = div_idx(i, HV, sh);
    const int c = (int)(i - t * HV);
    const InT* src = staging + (t * k * HV + c) * N;
    float acc[N];
    if constexpr (K > 0) {
      float v[K][N];
#pragma unroll
      for (int j = 0; j < K; ++j) Vec16<InT>::load(src + (long)j * HV * N, v[j]);
#pragma unroll
      for (int q = 0; q < N; ++q) acc[q] = v[0][q];
#pragma unroll
      for (int j = 1; j < K; ++j)
#pragma unroll
        for (int q = 0; q < N; ++q) acc[q] += v[j][q];
    } else {
      float v[N];
      Vec16<InT>::load(src, acc);
      for (int j = 1; j < k; ++j) {
        Vec16<InT>::load(src + (long)j * HV * N, v);
#pragma unroll
        for (int q = 0; q < N; ++q) acc[q] += v[q];
      }
    }
    store_out<OutT, N>(out + i * N, acc);
  }
}

template <class OutT>
__global__ void __launch_bounds__(256) combine_scalar_kernel(const float* __restrict__ staging, long T,
                                                             int k, int H, OutT* __restrict__ out, int sh) {
  pdl_wait();
  pdl_trigger();
  const long n = T * H;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const long t = div_idx(i, H, sh);
    const int h = (int)(i - t * H);
    float acc = staging[t * k * H + h];
    for (int j = 1; j < k; ++j) acc += staging[(t * k + j) * H + h];
    out[i] = from_float<OutT>(acc);
  }
}

// Slots dropped by the align step (expert index outside [0, E)) are in no
// expert's rows, so no FFN epilogue writes their staging rows. When any slot
// was dropped (offsets[E] < S) the whole staging buffer is zeroed before the
// FFN writes the routed rows; otherwise the kernel exits at once.
__global__ void __launch_bounds__(256) zero_dropped_kernel(const int32_t* __restrict__ offsets, int E, long S,
                                                           long n16, long n2, uint4* __restrict__ staging) {
  pdl_wait();
  pdl_trigger();
  if (__ldg(offsets + E) >= S) return;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (long)gridDim.x * blockDim.x)
    staging[i] = make_uint4(0u, 0u, 0u, 0u);
  // a tail shorter than 16 bytes (2-byte units)
  uint16_t* tail = reinterpret_cast<uint16_t*>(staging + n16);
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n2; i += (long)gridDim.x * blockDim.x) tail[i] = 0;
}

template <class InT, class OutT>
int launch_t(const InT* staging, int T, int k, int H, OutT* out, cudaStream_t s) {
  constexpr int N = Vec16<InT>::N;
  ProfScope ps("combine", s);
  const bool vec = H % N == 0;
  const long units = (long)T * (vec ? H / N : H);
  const long cap = (long)num_sms() * 8;
  const int grid = (int)std::max(1L, std::min(cap, (units + 255) / 256));
  cudaError_t e;
  if (vec && k == 8)
    e = launch_pdl(combine_vec_kernel<InT, OutT, 8>, grid, 256, 0, s, staging, (long)T, k, H / N, out,
                   pow2_shift(H / N));
  else if (vec && k == 2)
    e = launch_pdl(combine_vec_kernel<InT, OutT, 2>, grid, 256, 0, s, staging, (long)T, k, H / N, out,
                   pow2_shift(H / N));
  else if (vec)
    e = launch_pdl(combine_vec_kernel<InT, OutT, 0>, grid, 256, 0, s, staging, (long)T, k, H / N, out,
                   pow2_shift(H / N));
  else if constexpr (std::is_same<InT, float>::value)
    e = launch_pdl(combine_scalar_kernel<OutT>, grid, 256, 0, s, staging, (long)T, k, H, out, pow2_shift(H));
  else
    return fail(MOE_ERR_UNSUPPORTED, "combine: bf16 staging needs H %% 8 == 0 (H=%d)", H);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "combine: %s", cudaGetErrorString(e));
  return check_launch("combine");
}

}  // namespace

int launch_zero_dropped(const int32_t* offsets, int E, long S, int H, void* staging, int elem_bytes,
                        cudaStream_t s) {
  const long bytes = S * H * elem_bytes;
  if (bytes == 0) return MOE_OK;
  ProfScope ps("zero_dropped", s);
  const long n16 = bytes / 16, n2 = (bytes - n16 * 16) / 2;
  const int grid = (int)std::max(1L, std::min((long)num_sms() * 4, (n16 + 255) / 256));
  const cudaError_t e =
      launch_pdl(zero_dropped_kernel, grid, 256, 0, s, offsets, E, S, n16, n2, static_cast<uint4*>(staging));
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "zero_dropped: %s", cudaGetErrorString(e));
  return check_launch("zero_dropped");
}

int launch_combine(const void* staging, int staging_bf16, int T, int k, int H, int dtype, void* out,
                   cudaStream_t s) {
  if ((long)T * H == 0) return MOE_OK;
  if (staging_bf16) {
    const __nv_bfloat16* st = static_cast<const __nv_bfloat16*>(staging);
    return dtype == MOE_F32 ? launch_t(st, T, k, H, static_cast<float*>(out), s)
                            : launch_t(st, T, k, H, static_cast<__nv_bfloat16*>(out), s);
  }
  const float* st = static_cast<const float*>(staging);
  return dtype == MOE_F32 ? launch_t(st, T, k, H, static_cast<float*>(out), s)
                          : launch_t(st, T, k, H, static_cast<__nv_bfloat16*>(out), s);
}

}  // namespace moe
