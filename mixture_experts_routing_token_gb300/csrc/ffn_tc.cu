// Grouped expert FFN on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// project_6 moe_expert_gemm.cpp, moe_prefill_experts: for every expert with
// tokens, FC1 (x @ w13[e]^T), silu_and_mul, FC2 (act @ w2[e]^T), scale by the
// routing weight and accumulate into the token's row; mlc-llm moe_misc.py,
// scatter_output (sorted row p belongs to slot reverse_indices[p]).
//
// One persistent kernel per GEMM (FC1, FC2) walks a device-built tile list:
// tiles are (expert e, 128 sorted rows of e, one N tile), built in each CTA
// from the expert counts (no host sync), N tile major within an expert so that
// concurrently running CTAs share the same weight tile through L2.
//
// CTA = 6 warps, one CTA per SM:
//   warp 0      TMA producer: A tile (128 x 64 bf16) and B tile (256 x 64 bf16)
//               per k-step into a 4-stage ring. FC1's A operand is the
//               expert-sorted copy of the token rows written by
//               gather_rows_kernel (one tiled TMA load per stage; a fused
//               4-row TMA gather per stage measured 3.4x slower on GB300).
//   warp 1      MMA issuer: 4 x tcgen05.mma (M=128, N=256, K=16) per k-step into
//               one of two TMEM accumulators (2 x 256 columns), so the
//               epilogue of tile i overlaps the main loop of tile i+1.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator rows;
//               FC1: B rows 0..127 are gate rows n0.., rows 128..255 the
//                    matching up rows I+n0.., so act = silu(g) * u is formed
//                    in registers and stored as bf16 in sorted row order;
//               FC2: y * routing weight, stored as float32 to the slot's
//                    staging row reverse_indices[p] (no atomics).
// Every wait is bounded; on expiry the CTA drains, frees TMEM, and reports
// MOE_STATUS_TIMEOUT.
#include <cuda.h>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN = 256;                   // MMA N: B rows per tile
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int B_BYTES = BN * BK * 2;      // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int DSMEM_BYTES = STAGES * STAGE_BYTES + 1024;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // 2 s
constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, BN);

enum { MODE_FC1 = 0, MODE_FC2 = 1 };

struct TcParams {
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* sorted_ids;
  const float* sorted_w;
  const int32_t* reverse;
  int E;
  int K;            // reduction length (H for FC1, I for FC2)
  int N_out;        // output columns (I for FC1, H for FC2)
  int NT;           // N tiles per expert
  int b_rows;       // rows of one expert's weight matrix (2I or H)
  void* out;        // FC1: act bf16 [S, I]; FC2: staging f32 [S, H]
  int32_t* status;
};

struct TileInfo {
  int e, m_tile, n_tile;
};

__device__ __forceinline__ TileInfo decode_tile(int t, const int* tile_start, int E, int NT) {
  int lo = 0, hi = E;                    // last e with tile_start[e] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int local = t - tile_start[lo];
  const int mt = (tile_start[lo + 1] - tile_start[lo]) / NT;
  TileInfo ti;
  ti.e = lo;
  ti.n_tile = local / mt;
  ti.m_tile = local - ti.n_tile * mt;
  return ti;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    ffn_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const TcParams P) {
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int tile_start[MOE_MAX_EXPERTS + 1];
  extern __shared__ uint8_t dsmem_raw[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t dsmem = (ptx::smem_u32(dsmem_raw) + 1023u) & ~1023u;
  auto sA = [&](int s) { return dsmem + (uint32_t)(s * STAGE_BYTES); };
  auto sB = [&](int s) { return dsmem + (uint32_t)(s * STAGE_BYTES + A_BYTES); };
  volatile int* abort_p = &abort_flag;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&tfull_bar[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&tempty_bar[b]), 128);
    }
    ptx::mbar_init(ptx::smem_u32(&drain_bar), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
  }
  if (warp == 1) ptx::tmem_alloc(ptx::smem_u32(&tmem_slot), TMEM_COLS);
  if (warp == 2) {   // tile list: tile_start[e] = sum over e' < e of ceil(count/BM) * NT
    const int per = (P.E + 31) / 32;
    const int e0 = min(P.E, lane * per), e1 = min(P.E, e0 + per);
    int run = 0;
    for (int e = e0; e < e1; ++e) run += (__ldg(P.counts + e) + BM - 1) / BM * P.NT;
    int incl = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int acc = incl - run;
    for (int e = e0; e < e1; ++e) {
      tile_start[e] = acc;
      acc += (__ldg(P.counts + e) + BM - 1) / BM * P.NT;
    }
    if (lane == 31) tile_start[P.E] = incl;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = tmem_slot;
  const int total = tile_start[P.E];

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t ph = 0;
    int issued_parity[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
    const int KB = P.K / BK;
    if (lane == 0) {
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const TileInfo ti = decode_tile(t, tile_start, P.E, P.NT);
        const int a_row0 = __ldg(P.offsets + ti.e) + ti.m_tile * BM;
        int b_row0, b_row1;
        if (MODE == MODE_FC1) {
          b_row0 = ti.e * P.b_rows + ti.n_tile * 128;
          b_row1 = b_row0 + P.N_out;            // up rows: I + n0
        } else {
          b_row0 = ti.e * P.b_rows + ti.n_tile * BN;
          b_row1 = b_row0 + 128;
        }
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&empty_bar[stage]), ph ^ 1u, abort_p, WAIT_LIMIT_NS))
            goto producer_done;
          const uint32_t fb = ptx::smem_u32(&full_bar[stage]);
          ptx::mbar_arrive_expect_tx(fb, STAGE_BYTES);
          ptx::tma_load_2d(sA(stage), &tmA, kb * BK, a_row0, fb);
          ptx::tma_load_2d(sB(stage), &tmB, kb * BK, b_row0, fb);
          ptx::tma_load_2d(sB(stage) + 128 * 128, &tmB, kb * BK, b_row1, fb);
          issued_parity[stage] = (int)ph;
          if (++stage == STAGES) { stage = 0; ph ^= 1u; }
        }
      }
    producer_done:
      // wait until every copy this thread issued has landed
      int dummy = 0;
      for (int s = 0; s < STAGES; ++s)
        if (issued_parity[s] >= 0)
          ptx::mbar_wait(ptx::smem_u32(&full_bar[s]), (uint32_t)issued_parity[s], &dummy, WAIT_LIMIT_NS);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      const int KB = P.K / BK;
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        if (!ptx::mbar_wait(ptx::smem_u32(&tempty_bar[acc]), aph ^ 1u, abort_p, WAIT_LIMIT_NS)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&full_bar[stage]), ph, abort_p, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = sA(stage), b0 = sB(stage);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            ptx::mma_bf16(d_tmem, ptx::sdesc_k128(a0 + kk * 32), ptx::sdesc_k128(b0 + kk * 32), IDESC,
                          (kb | kk) != 0);
          ptx::mma_commit(ptx::smem_u32(&empty_bar[stage]));
          if (++stage == STAGES) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
        ptx::mma_commit(ptx::smem_u32(&tfull_bar[acc]));
        if (++acc == 2) { acc = 0; aph ^= 1u; }
      }
      // all issued MMAs complete before TMEM is released
      ptx::mma_commit(ptx::smem_u32(&drain_bar));
      int dummy = 0;
      ptx::mbar_wait(ptx::smem_u32(&drain_bar), 0, &dummy, WAIT_LIMIT_NS);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const TileInfo ti = decode_tile(t, tile_start, P.E, P.NT);
      if (!ptx::mbar_wait(ptx::smem_u32(&tfull_bar[acc]), aph, abort_p, WAIT_LIMIT_NS)) break;
      ptx::tc_fence_after();
      const int cnt = __ldg(P.counts + ti.e);
      const int r = ti.m_tile * BM + row;
      const bool valid = r < cnt;
      const long p = (long)__ldg(P.offsets + ti.e) + r;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      if (MODE == MODE_FC1) {
        const int I = P.N_out;
        __nv_bfloat16* act = static_cast<__nv_bfloat16*>(P.out);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          ptx::tmem_ld32(taddr + c * 32, g);
          ptx::tmem_ld32(taddr + 128 + c * 32, u);
          ptx::tmem_ld_wait();
          const int col0 = ti.n_tile * 128 + c * 32;
          if (valid && col0 < I) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float a0 = silu(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
              const float a1 = silu(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
              pk[i] = pack_bf16x2(a0, a1);
            }
            uint4* dst = reinterpret_cast<uint4*>(act + p * I + col0);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      } else {
        const int H = P.N_out;
        float* staging = static_cast<float*>(P.out);
        const float wt = valid ? __ldg(P.sorted_w + p) : 0.0f;
        const long dst_row = valid ? (long)__ldg(P.reverse + p) : 0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t y[32];
          ptx::tmem_ld32(taddr + c * 32, y);
          ptx::tmem_ld_wait();
          const int col0 = ti.n_tile * BN + c * 32;
          if (valid && col0 < H) {
            float4* dst = reinterpret_cast<float4*>(staging + dst_row * H + col0);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(y[4 * i]) * wt, __uint_as_float(y[4 * i + 1]) * wt,
                                   __uint_as_float(y[4 * i + 2]) * wt, __uint_as_float(y[4 * i + 3]) * wt);
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&tempty_bar[acc]));
      if (++acc == 2) { acc = 0; aph ^= 1u; }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if (tid == 0 && abort_flag && P.status) atomicOr(P.status, MOE_STATUS_TIMEOUT);
}

// Copies the expert-sorted token rows of `hidden` into x_sorted, the FC1 A operand
// (16-byte vectors; rows p < offsets[E]).
__global__ void gather_rows_kernel(const uint4* __restrict__ hidden, const int32_t* __restrict__ ids,
                                   const int32_t* __restrict__ offsets, int E, int H16,
                                   uint4* __restrict__ xs) {
  const int n = __ldg(offsets + E);
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < (long)n * H16;
       i += (long)gridDim.x * blockDim.x) {
    const long p = i / H16;
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

namespace {

template <int MODE>
int launch_tc(const CUtensorMap& a, const CUtensorMap& b, const TcParams& p, long S, cudaStream_t s,
              const char* name) {
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr[dev]) {
    if (cudaFuncSetAttribute(ffn_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             DSMEM_BYTES) != cudaSuccess)
      return check_launch(name);
    attr[dev] = true;
  }
  const long max_tiles = ((S + BM - 1) / BM + p.E) * (long)p.NT;
  const int grid = (int)(max_tiles < num_sms() ? max_tiles : num_sms());
  if (grid <= 0) return MOE_OK;
  ProfScope ps(name, s);
  ffn_tc_kernel<MODE><<<grid, THREADS, DSMEM_BYTES, s>>>(a, b, p);
  return check_launch(name);
}

}  // namespace

bool ffn_uses_tensor_cores(int dtype, int H, int I) {
  return dtype == MOE_BF16 && H % 64 == 0 && I % 64 == 0 && H > 0 && I > 0;
}

size_t ffn_tc_extra_bytes(long S, int H) { return (size_t)S * H * 2; }

int launch_ffn_tc(const FfnArgs& a, cudaStream_t s) {
  const long S = (long)a.T * a.k;
  if (S == 0) return MOE_OK;
  if (a.T <= kDecodeMaxTokens) return launch_ffn_decode(a, s);
  CUtensorMap tA1, tB1, tA2, tB2;
  int rc;
  {
    ProfScope ps("gather_rows", s);
    gather_rows_kernel<<<num_sms() * 4, 256, 0, s>>>(static_cast<const uint4*>(a.hidden), a.sorted_ids,
                                                     a.offsets, a.E, a.H / 8, static_cast<uint4*>(a.xs));
    if ((rc = check_launch("gather_rows"))) return rc;
  }
  if ((rc = make_tmap(&tA1, a.xs, (uint64_t)S, (uint64_t)a.H, BM))) return rc;
  if ((rc = make_tmap(&tB1, a.w13, (uint64_t)a.E * 2 * a.I, (uint64_t)a.H, 128))) return rc;
  if ((rc = make_tmap(&tA2, a.act, (uint64_t)S, (uint64_t)a.I, BM))) return rc;
  if ((rc = make_tmap(&tB2, a.w2, (uint64_t)a.E * a.H, (uint64_t)a.I, 128))) return rc;

  TcParams p1{a.counts, a.offsets, a.sorted_ids, a.sorted_w, a.reverse, a.E, a.H, a.I,
              (a.I + 127) / 128, 2 * a.I, a.act, a.status};
  if ((rc = launch_tc<MODE_FC1>(tA1, tB1, p1, S, s, "ffn_fc1_tc"))) return rc;
  TcParams p2{a.counts, a.offsets, a.sorted_ids, a.sorted_w, a.reverse, a.E, a.I, a.H,
              (a.H + BN - 1) / BN, a.H, a.staging, a.status};
  if ((rc = launch_tc<MODE_FC2>(tA2, tB2, p2, S, s, "ffn_fc2_tc"))) return rc;
  return launch_combine(a.staging, a.T, a.k, a.H, a.dtype, a.out, s);
}

}  // namespace moe
