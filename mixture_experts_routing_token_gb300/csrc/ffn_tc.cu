// Prefill path of the grouped expert FFN on the 5th-generation tensor cores.
//
// project_6 moe_expert_gemm.cpp, moe_prefill_experts: for every expert with
// tokens, gather its token rows, FC1 (x @ w13[e]^T), silu_and_mul, FC2
// (act @ w2[e]^T), scale by the routing weight and accumulate into the
// token's row; mlc-llm moe_misc.py, scatter_output and moe_sum.
//
// Steps on the caller's stream, no host synchronisation:
//   1. gather_rows_bulk_kernel (rows up to 16 KB; else gather_rows_kernel)
//      copies the expert-sorted token rows of `hidden` into x_sorted (the
//      FC1 A operand; one tiled TMA load per pipeline stage then feeds the
//      MMA; a fused four-row TMA gather per stage was measured 3.4x slower
//      on GB300);
//   2. FC1 and FC2 run as persistent 2-SM grouped GEMMs (ffn_tc_pair.cu);
//   3. the combine kernel sums each token's k weighted rows (combine.cu).
// Batches of at most kDecodeMaxTokens tokens take the weight-streaming
// kernels of ffn_decode.cu instead.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "sm100_ptx.cuh"

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

// The same copy with TMA bulk transfers (rows of at most kBulkRowMax bytes):
// warp w takes batches of R consecutive sorted rows; its lane 0 loads the R
// token rows of `hidden` into the warp's shared-memory slots (one mbarrier per
// slot, bounded waits), then writes the batch to x_sorted as ONE contiguous
// bulk store, and reuses the slots once that store has read them. The copy
// engine moves the bytes, so R whole rows per warp are in flight with almost
// no instructions.
constexpr int kBulkWarps = 8;
constexpr int kBulkMaxR = 4;
constexpr int kBulkSmem = 128 * 1024;
constexpr int kBulkRowMax = kBulkSmem / kBulkWarps;
constexpr uint64_t kBulkWaitNs = 2000000000ull;

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__global__ void __launch_bounds__(kBulkWarps * 32) gather_rows_bulk_kernel(
    const uint8_t* __restrict__ hidden, const int32_t* __restrict__ ids, const int32_t* __restrict__ offsets,
    int E, int row_bytes, int R, uint8_t* __restrict__ xs, int32_t* status) {
  extern __shared__ __align__(128) uint8_t slots[];   // [kBulkWarps][R][row_bytes]
  __shared__ __align__(8) uint64_t bar[kBulkWarps][kBulkMaxR];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) abort_flag = 0;
  if (lane == 0)
    for (int r = 0; r < R; ++r) ptx::mbar_init(ptx::smem_u32(&bar[warp][r]), 1);
  ptx::fence_mbar_init();
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (lane != 0) return;
  volatile int* abort_p = &abort_flag;
  const int n = __ldg(offsets + E);
  const int nw = gridDim.x * kBulkWarps;
  const uint32_t my = ptx::smem_u32(slots) + (uint32_t)(warp * R * row_bytes);
  uint32_t ph = 0;
  for (long p0 = (long)(blockIdx.x * kBulkWarps + warp) * R; p0 < n; p0 += (long)nw * R) {
    const int nr = (int)min((long)R, n - p0);
    for (int r = 0; r < nr; ++r) {
      const uint32_t b = ptx::smem_u32(&bar[warp][r]);
      ptx::mbar_arrive_expect_tx(b, (uint32_t)row_bytes);
      bulk_load(my + (uint32_t)(r * row_bytes), hidden + (long)__ldg(ids + p0 + r) * row_bytes, (uint32_t)row_bytes, b);
    }
    bool ok = true;
    for (int r = 0; r < nr && ok; ++r) ok = ptx::mbar_wait(ptx::smem_u32(&bar[warp][r]), ph, abort_p, kBulkWaitNs);
    if (!ok) {   // let the loads still in flight land (bounded) before the slots go away
      for (int r = 0; r < nr; ++r) {
        int dummy = 0;
        ptx::mbar_wait(ptx::smem_u32(&bar[warp][r]), ph, &dummy, kBulkWaitNs / 2);
      }
      if (status) atomicOr(status, MOE_STATUS_TIMEOUT);
      break;
    }
    bulk_store(xs + p0 * row_bytes, my, (uint32_t)(nr * row_bytes));
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");   // the slots may be refilled
    ph ^= 1u;
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// pos[reverse[p]] = p for the routed rows p < offsets[E]: the sorted row of every
// slot. Slots the align step dropped keep whatever the buffer held; readers check
// reverse[pos[s]] == s before they use an entry.
__global__ void __launch_bounds__(256) slot_rows_kernel(const int32_t* __restrict__ reverse,
                                                        const int32_t* __restrict__ offsets, int E,
                                                        int32_t* __restrict__ pos) {
  pdl_wait();
  pdl_trigger();
  const int n = __ldg(offsets + E);
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < n; p += gridDim.x * blockDim.x)
    pos[__ldg(reverse + p)] = p;
}

// The expert-sorted copy of the token rows in token order: warp w takes batches
// of R consecutive tokens; lane 0 loads their rows of `hidden` into the warp's
// shared-memory slots with bulk copies (one mbarrier per slot, bounded waits),
// then each lane writes one of the batch's R*k slots: a bulk store of the
// token's row to x_sorted[pos[slot]]. Every row of `hidden` is read once (a
// walk over the sorted rows reads a token's row once per slot, k times, mostly
// from DRAM when `hidden` exceeds L2).
__global__ void __launch_bounds__(kBulkWarps * 32) gather_by_token_kernel(
    const uint8_t* __restrict__ hidden, const int32_t* __restrict__ pos, const int32_t* __restrict__ reverse,
    const int32_t* __restrict__ offsets, int E, int T, int k, int row_bytes, int R, uint8_t* __restrict__ xs,
    int32_t* status) {
  extern __shared__ __align__(128) uint8_t slots[];   // [kBulkWarps][R][row_bytes]
  __shared__ __align__(8) uint64_t bar[kBulkWarps][kBulkMaxR];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) abort_flag = 0;
  if (lane == 0)
    for (int r = 0; r < R; ++r) ptx::mbar_init(ptx::smem_u32(&bar[warp][r]), 1);
  ptx::fence_mbar_init();
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  volatile int* abort_p = &abort_flag;
  const int n = __ldg(offsets + E);
  const int nw = gridDim.x * kBulkWarps;
  const uint32_t my = ptx::smem_u32(slots) + (uint32_t)(warp * R * row_bytes);
  const int kshift = (k & (k - 1)) == 0 ? __ffs(k) - 1 : -1;
  uint32_t ph = 0;
  for (int t0 = (blockIdx.x * kBulkWarps + warp) * R; t0 < T; t0 += nw * R) {
    const int nr = min(R, T - t0);
    if (lane == 0)
      for (int r = 0; r < nr; ++r) {
        const uint32_t b = ptx::smem_u32(&bar[warp][r]);
        ptx::mbar_arrive_expect_tx(b, (uint32_t)row_bytes);
        bulk_load(my + (uint32_t)(r * row_bytes), hidden + (long)(t0 + r) * row_bytes, (uint32_t)row_bytes, b);
      }
    bool ok = true;   // every lane sees the rows land before it stores from them
    for (int r = 0; r < nr && ok; ++r) ok = ptx::mbar_wait(ptx::smem_u32(&bar[warp][r]), ph, abort_p, kBulkWaitNs);
    if (!__all_sync(0xffffffffu, ok)) {   // let the loads still in flight land (bounded) before the slots go away
      if (lane == 0) {
        for (int r = 0; r < nr; ++r) {
          int dummy = 0;
          ptx::mbar_wait(ptx::smem_u32(&bar[warp][r]), ph, &dummy, kBulkWaitNs / 2);
        }
        if (status) atomicOr(status, MOE_STATUS_TIMEOUT);
      }
      break;
    }
    for (int l = lane; l < nr * k; l += 32) {
      const int r = kshift >= 0 ? l >> kshift : l / k;
      const int s = (t0 + r) * k + (l - r * k);
      const int p = __ldg(pos + s);
      if (p >= 0 && p < n && __ldg(reverse + p) == s)
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(xs + (long)p * row_bytes),
                     "r"(my + (uint32_t)(r * row_bytes)), "r"((uint32_t)row_bytes)
                     : "memory");
    }
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");   // this lane's stores have read the slots
    __syncwarp();                                                      // ... and every lane's: refill
    ph ^= 1u;
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
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

int launch_gather_rows(const void* hidden, const int32_t* sorted_ids, const int32_t* offsets, int E, int row_bytes,
                       void* xs, int32_t* status, cudaStream_t s) {
  if (row_bytes % 16 != 0) return fail(MOE_ERR_UNSUPPORTED, "gather_rows: rows of %d bytes (need a multiple of 16)", row_bytes);
  ProfScope ps("gather_rows", s);
  cudaError_t e;
  if (row_bytes <= kBulkRowMax) {
    if (int rc = ensure_smem_limit(gather_rows_bulk_kernel, kBulkSmem, "gather_rows")) return rc;
    const int R = std::min(kBulkMaxR, kBulkRowMax / row_bytes);
    e = launch_pdl(gather_rows_bulk_kernel, num_sms(), kBulkWarps * 32, (size_t)kBulkWarps * R * row_bytes, s,
                   static_cast<const uint8_t*>(hidden), sorted_ids, offsets, E, row_bytes, R,
                   static_cast<uint8_t*>(xs), status);
  } else {
    const int r16 = row_bytes / 16;
    e = launch_pdl(gather_rows_kernel, num_sms() * 4, 256, 0, s, static_cast<const uint4*>(hidden), sorted_ids,
                   offsets, E, r16, pow2_shift(r16), static_cast<uint4*>(xs));
  }
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "gather_rows: %s", cudaGetErrorString(e));
  return check_launch("gather_rows");
}

// bf16 matrix [rows, cols] row-major; box = box_rows x 64 columns, 128-byte swizzle.
// The encoded maps of recent (base, rows, cols, box) keys are kept: a layer call
// with the same buffers reuses them instead of encoding again.
namespace {
struct TmapEntry {
  const void* base;
  uint64_t rows, cols;
  uint32_t box_rows;
  bool used;
  CUtensorMap map;
};
std::mutex g_tmap_mu;
TmapEntry g_tmaps[64];
}  // namespace

int make_tmap(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  const size_t slot = ((reinterpret_cast<uintptr_t>(base) >> 8) ^ rows * 31 ^ cols * 131 ^ box_rows * 7) % 64;
  {
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    const TmapEntry& c = g_tmaps[slot];
    if (c.used && c.base == base && c.rows == rows && c.cols == cols && c.box_rows == box_rows) {
      *m = c.map;
      return MOE_OK;
    }
  }
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
  std::lock_guard<std::mutex> lk(g_tmap_mu);
  g_tmaps[slot] = TmapEntry{base, rows, cols, box_rows, true, *m};
  return MOE_OK;
}

int make_tmap_rows128(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, int elem_bytes,
                      uint32_t box_rows) {
  if (elem_bytes != 2 && elem_bytes != 4) return fail(MOE_ERR_UNSUPPORTED, "make_tmap_rows128: %d-byte elements", elem_bytes);
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (cuuint64_t)elem_bytes};
  const cuuint32_t box[2] = {128u / (cuuint32_t)elem_bytes, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  const CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MOE_OK;
}

bool ffn_uses_tensor_cores(int dtype, int H, int I) {
  return dtype == MOE_BF16 && H % 64 == 0 && I % 64 == 0 && H > 0 && I > 0;
}

bool staging_is_bf16(int dtype, int T, int H, int I) {
  return ffn_uses_tensor_cores(dtype, H, I) && T > kDecodeMaxTokens;
}

size_t ffn_tc_extra_bytes(long S, int H) { return (size_t)S * H * 2; }
size_t ffn_tc_pos_bytes(long S) { return (size_t)S * sizeof(int32_t); }

int launch_ffn_tc(const FfnArgs& a, cudaStream_t s) {
  const long S = (long)a.T * a.k;
  if (S == 0) return MOE_OK;
  if (a.T <= kDecodeMaxTokens) return launch_ffn_decode(a, s);
  CUtensorMap tA1, tB1, tA2, tB2, tS2;
  int rc;
  const int row_bytes = a.H * 2;
  if (row_bytes <= kBulkRowMax) {
    {
      ProfScope ps("slot_rows", s);
      const int grid = (int)std::max(1L, std::min((long)num_sms() * 4, (S + 255) / 256));
      const cudaError_t e = launch_pdl(slot_rows_kernel, grid, 256, 0, s, a.reverse, a.offsets, a.E, a.pos);
      if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "slot_rows: %s", cudaGetErrorString(e));
      if ((rc = check_launch("slot_rows"))) return rc;
    }
    ProfScope ps("gather_rows", s);
    if ((rc = ensure_smem_limit(gather_by_token_kernel, kBulkSmem, "gather_rows"))) return rc;
    const int R = std::min(kBulkMaxR, kBulkRowMax / row_bytes);
    const cudaError_t e =
        launch_pdl(gather_by_token_kernel, num_sms(), kBulkWarps * 32, (size_t)kBulkWarps * R * row_bytes, s,
                   static_cast<const uint8_t*>(a.hidden), a.pos, a.reverse, a.offsets, a.E, a.T, a.k, row_bytes, R,
                   static_cast<uint8_t*>(a.xs), a.status);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "gather_rows: %s", cudaGetErrorString(e));
    if ((rc = check_launch("gather_rows"))) return rc;
  } else if ((rc = launch_gather_rows(a.hidden, a.sorted_ids, a.offsets, a.E, row_bytes, a.xs, a.status, s))) {
    return rc;
  }
  if ((rc = make_tmap(&tA1, a.xs, (uint64_t)S, (uint64_t)a.H, 128))) return rc;
  if ((rc = make_tmap(&tB1, a.w13, (uint64_t)a.E * 2 * a.I, (uint64_t)a.H, 128))) return rc;
  if ((rc = make_tmap(&tA2, a.act, (uint64_t)S, (uint64_t)a.I, 128))) return rc;
  if ((rc = make_tmap(&tB2, a.w2, (uint64_t)a.E * a.H, (uint64_t)a.I, 128))) return rc;
  if ((rc = make_tmap(&tS2, a.act, (uint64_t)S, (uint64_t)a.I, 32))) return rc;

  if ((rc = launch_ffn_pair_gemms(a, tA1, tB1, tA2, tB2, tS2, s))) return rc;
  return launch_combine(a.staging, 1, a.T, a.k, a.H, a.dtype, a.out, s);
}

}  // namespace moe
