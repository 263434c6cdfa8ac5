// Prefill path of the grouped expert FFN on the 5th-generation tensor cores.
//
// project_6 moe_expert_gemm.cpp, moe_prefill_experts: for every expert with
// tokens, gather its token rows, FC1 (x @ w13[e]^T), silu_and_mul, FC2
// (act @ w2[e]^T), scale by the routing weight and accumulate into the
// token's row; mlc-llm moe_misc.py, scatter_output and moe_sum.
//
// Steps on the caller's stream, no host synchronisation:
//   1. gather_rows_kernel copies the expert-sorted token rows of `hidden`
//      into x_sorted (the FC1 A operand; one tiled TMA load per pipeline
//      stage then feeds the MMA; a fused four-row TMA gather per stage was
//      measured 3.4x slower on GB300);
//   2. FC1 and FC2 run as persistent 2-SM grouped GEMMs (ffn_tc_pair.cu);
//   3. the combine kernel sums each token's k weighted rows (combine.cu).
// Batches of at most kDecodeMaxTokens tokens take the weight-streaming
// kernels of ffn_decode.cu instead.
#include <cuda.h>

#include "common.cuh"

namespace moe {
namespace {

// Copies the expert-sorted token rows of `hidden` into x_sorted, the FC1 A operand
// (16-byte vectors; rows p < offsets[E]).
__global__ void gather_rows_kernel(const uint4* __restrict__ hidden, const int32_t* __restrict__ ids,
                                   const int32_t* __restrict__ offsets, int E, int H16, int sh,
                                   uint4* __restrict__ xs) {
  pdl_wait();
  pdl_trigger();
  const int n = __ldg(offsets + E);
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < (long)n * H16;
       i += (long)gridDim.x * blockDim.x) {
    const long p = div_idx(i, H16, sh);
    const int c = (int)(i - p * H16);
    xs[i] = __ldg(hidden + (long)__ldg(ids + p) * H16 + c);
  }
}

// ---- host -------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

// bf16 matrix [rows, cols] row-major; box = box_rows x 64 columns, 128-byte swizzle.
int make_tmap(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MOE_OK;
}

bool ffn_uses_tensor_cores(int dtype, int H, int I) {
  return dtype == MOE_BF16 && H % 64 == 0 && I % 64 == 0 && H > 0 && I > 0;
}

size_t ffn_tc_extra_bytes(long S, int H) { return (size_t)S * H * 2; }

int launch_ffn_tc(const FfnArgs& a, cudaStream_t s) {
  const long S = (long)a.T * a.k;
  if (S == 0) return MOE_OK;
  if (a.T <= kDecodeMaxTokens) return launch_ffn_decode(a, s);
  CUtensorMap tA1, tB1, tA2, tB2, tS2;
  int rc;
  {
    ProfScope ps("gather_rows", s);
    const cudaError_t e = launch_pdl(gather_rows_kernel, num_sms() * 4, 256, 0, s,
                                     static_cast<const uint4*>(a.hidden), a.sorted_ids, a.offsets, a.E,
                                     a.H / 8, pow2_shift(a.H / 8), static_cast<uint4*>(a.xs));
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "gather_rows: %s", cudaGetErrorString(e));
    if ((rc = check_launch("gather_rows"))) return rc;
  }
  if ((rc = make_tmap(&tA1, a.xs, (uint64_t)S, (uint64_t)a.H, 128))) return rc;
  if ((rc = make_tmap(&tB1, a.w13, (uint64_t)a.E * 2 * a.I, (uint64_t)a.H, 128))) return rc;
  if ((rc = make_tmap(&tA2, a.act, (uint64_t)S, (uint64_t)a.I, 128))) return rc;
  if ((rc = make_tmap(&tB2, a.w2, (uint64_t)a.E * a.H, (uint64_t)a.I, 128))) return rc;
  if ((rc = make_tmap(&tS2, a.act, (uint64_t)S, (uint64_t)a.I, 32))) return rc;

  if ((rc = launch_ffn_pair_gemms(a, tA1, tB1, tA2, tB2, tS2, s))) return rc;
  return launch_combine(a.staging, a.T, a.k, a.H, a.dtype, a.out, s);
}

}  // namespace moe
