// Weighted combine: out[t] = sum_{j<k} staging[t*k + j], j ascending, fp32,
// one rounding to the output dtype.
// mlc-llm moe_misc.py moe_sum (sum of the [T, k, H] expert outputs over k);
// the routing weight was already applied by the FC2 epilogue.
// HBM-bound streaming kernel: 16-byte loads, one thread per 4 output columns.
// Launched with programmatic dependency on the FC2 kernel (waits before reading).
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace {

template <class OutT>
struct Out4;
template <>
struct Out4<float> {
  static __device__ __forceinline__ void store(float* o, float4 v) {
    *reinterpret_cast<float4*>(o) = v;
  }
};
template <>
struct Out4<__nv_bfloat16> {
  static __device__ __forceinline__ void store(__nv_bfloat16* o, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(o) = u;
  }
};

template <class OutT>
__global__ void __launch_bounds__(256) combine_vec_kernel(const float4* __restrict__ staging, long T,
                                                          int k, int H4, OutT* __restrict__ out, int sh) {
  pdl_wait();
  pdl_trigger();
  const long n = T * H4;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
    const long t = div_idx(i, H4, sh);
    const int c = (int)(i - t * H4);
    const float4* src = staging + t * k * H4 + c;
    float4 acc = __ldcs(src);
    for (int j = 1; j < k; ++j) {
      const float4 v = __ldcs(src + (long)j * H4);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    Out4<OutT>::store(out + i * 4, acc);
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
                                                           int H4, float4* __restrict__ staging) {
  pdl_wait();
  pdl_trigger();
  if (__ldg(offsets + E) >= S) return;
  const long n = S * H4;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x)
    staging[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(256) zero_dropped_scalar_kernel(const int32_t* __restrict__ offsets, int E,
                                                                  long S, int H, float* __restrict__ staging) {
  pdl_wait();
  pdl_trigger();
  if (__ldg(offsets + E) >= S) return;
  const long n = S * H;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x)
    staging[i] = 0.0f;
}

template <class OutT>
int launch_t(const float* staging, int T, int k, int H, OutT* out, cudaStream_t s) {
  ProfScope ps("combine", s);
  const long units = (long)T * (H % 4 == 0 ? H / 4 : H);
  const long cap = (long)num_sms() * 8;
  const int grid = (int)std::max(1L, std::min(cap, (units + 255) / 256));
  cudaError_t e;
  if (H % 4 == 0)
    e = launch_pdl(combine_vec_kernel<OutT>, grid, 256, 0, s, reinterpret_cast<const float4*>(staging), (long)T, k,
                   H / 4, out, pow2_shift(H / 4));
  else
    e = launch_pdl(combine_scalar_kernel<OutT>, grid, 256, 0, s, staging, (long)T, k, H, out, pow2_shift(H));
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "combine: %s", cudaGetErrorString(e));
  return check_launch("combine");
}

}  // namespace

int launch_zero_dropped(const int32_t* offsets, int E, long S, int H, float* staging, cudaStream_t s) {
  if (S * H == 0) return MOE_OK;
  ProfScope ps("zero_dropped", s);
  const long units = S * (H % 4 == 0 ? H / 4 : H);
  const int grid = (int)std::max(1L, std::min((long)num_sms() * 4, (units + 255) / 256));
  const cudaError_t e =
      H % 4 == 0 ? launch_pdl(zero_dropped_kernel, grid, 256, 0, s, offsets, E, S, H / 4,
                              reinterpret_cast<float4*>(staging))
                 : launch_pdl(zero_dropped_scalar_kernel, grid, 256, 0, s, offsets, E, S, H, staging);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "zero_dropped: %s", cudaGetErrorString(e));
  return check_launch("zero_dropped");
}

int launch_combine(const float* staging, int T, int k, int H, int dtype, void* out, cudaStream_t s) {
  if ((long)T * H == 0) return MOE_OK;
  return dtype == MOE_F32 ? launch_t<float>(staging, T, k, H, static_cast<float*>(out), s)
                          : launch_t<__nv_bfloat16>(staging, T, k, H, static_cast<__nv_bfloat16*>(out), s);
}

}  // namespace moe
