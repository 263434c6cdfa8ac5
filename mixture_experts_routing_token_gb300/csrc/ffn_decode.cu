// Weight-streaming expert FFN for small token counts (decode, T <= 64).
//
// project_6 moe_expert_gemm.cpp, moe_decode_experts: per routed expert, FC1
// (x @ w13[e]^T), silu_and_mul, FC2 (act @ w2[e]^T), scale by the routing
// weight and accumulate; here for all experts of a small batch at once.
//
// At decode sizes an expert sees at most T tokens, so the roles of the GEMM
// operands are swapped: weight rows are the MMA's M = 128 operand, the
// expert's tokens (padded to NTOK = 16, 32 or 64) are N. Each weight tile is
// streamed from HBM once per chunk of NTOK tokens (once in total when
// T <= NTOK), and only experts with tokens are touched.
//
// CTA = 6 warps, one per SM, persistent over (expert, token chunk, weight
// tile) tiles built on the device from the counts:
//   warp 0      TMA producer: 128 weight rows (FC1: 64 gate rows over the 64
//               matching up rows, i.e. 64 activation columns per tile; FC2: 128
//               rows of w2[e]) and the chunk's token rows (FC1: 4-row TMA
//               gathers from `hidden`; FC2: a tiled load of the expert-sorted
//               activation rows), 8-stage ring;
//   warp 1      MMA issuer: tcgen05.mma M=128, N=NTOK, K=16;
//   warps 2..5  epilogue: FC1: the two warps holding the up rows pass them
//               through shared memory to the two warps holding the gate rows
//               (bounded mbarrier hand-off), which form act = silu(g) * u and
//               store bf16 activation rows; FC2: y * routing weight -> float32
//               staging row of the slot.
// All waits are bounded as in the prefill kernel.
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

constexpr int DM = 128;          // weight rows per tile (MMA M)
constexpr int DK = 64;           // K per stage (one 128-byte swizzle row)
constexpr int DSTAGES_MAX = 8;
constexpr int DTHREADS = 192;
constexpr uint64_t DWAIT_NS = 2000000000ull;

enum { DEC_FC1 = 0, DEC_FC2 = 1 };

struct DecParams {
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* sorted_ids;
  const float* sorted_w;
  const int32_t* reverse;
  int E;
  int K;          // reduction length: H (FC1) or I (FC2)
  int N_out;      // output columns: I (FC1) or H (FC2)
  int NTW;        // weight tiles per expert: I / 64 (FC1) or ceil(H / 128) (FC2)
  int w_rows;     // rows of one expert's weight matrix: 2I or H
  void* out;      // FC1: act bf16 [S, I]; FC2: staging f32 [S, H]
  int32_t* status;
};

template <int MODE, int NTOK>
struct DecCfg {
  static constexpr int A_BYTES = DM * DK * 2;
  static constexpr int B_BYTES = NTOK * DK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;            // multiple of 1024
  static constexpr int STAGES = 8;
  static constexpr int XBUF = MODE == DEC_FC1 ? 64 * NTOK * 4 : 0;   // up-row hand-off
  static constexpr int DSMEM = STAGES * STAGE + XBUF + 1024;
  static constexpr int ACC_COLS = NTOK;                      // one accumulator buffer
  static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS < 32 ? 32 : 2 * ACC_COLS;
  static_assert(STAGE % 1024 == 0, "stage must keep 1024-byte alignment");
  static_assert(STAGES <= DSTAGES_MAX && DSMEM <= 209 * 1024, "shared memory budget");
  static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM allocation must be a power of two");
};

struct DecTile {
  int e, chunk, wt;
};

__device__ __forceinline__ DecTile dec_tile(int t, const int* tile_start, int E, int NTW) {
  int lo = 0, hi = E;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int local = t - tile_start[lo];
  DecTile d;
  d.e = lo;
  d.chunk = local / NTW;
  d.wt = local - d.chunk * NTW;
  return d;
}

template <int MODE, int NTOK>
__global__ void __launch_bounds__(DTHREADS, 1)
    ffn_decode_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const DecParams P) {
  using C = DecCfg<MODE, NTOK>;
  constexpr uint32_t IDESC = ptx::idesc_bf16_f32(DM, NTOK);
  __shared__ __align__(8) uint64_t full_bar[DSTAGES_MAX], empty_bar[DSTAGES_MAX];
  __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2], drain_bar, xfull_bar, xempty_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int tile_start[MOE_MAX_EXPERTS + 1];
  extern __shared__ uint8_t dsmem_raw[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t dsmem = (ptx::smem_u32(dsmem_raw) + 1023u) & ~1023u;
  auto sA = [&](int s) { return dsmem + (uint32_t)(s * C::STAGE); };
  auto sB = [&](int s) { return dsmem + (uint32_t)(s * C::STAGE + C::A_BYTES); };
  // up-row hand-off buffer [NTOK][64] floats, after the ring
  float* xbuf = reinterpret_cast<float*>(dsmem_raw + (dsmem - ptx::smem_u32(dsmem_raw)) + C::STAGES * C::STAGE);
  volatile int* abort_p = &abort_flag;

  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&xfull_bar), 64);
    ptx::mbar_init(ptx::smem_u32(&xempty_bar), 64);
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&tfull_bar[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&tempty_bar[b]), 128);
    }
    ptx::mbar_init(ptx::smem_u32(&drain_bar), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmW);
    ptx::prefetch_tmap(&tmX);
  }
  if (warp == 1) ptx::tmem_alloc(ptx::smem_u32(&tmem_slot), C::TMEM_COLS);
  if (warp == 2) {   // tile_start[e] = sum over e' < e of ceil(count / NTOK) * NTW
    const int per = (P.E + 31) / 32;
    const int e0 = min(P.E, lane * per), e1 = min(P.E, e0 + per);
    int run = 0;
    for (int e = e0; e < e1; ++e) run += (__ldg(P.counts + e) + NTOK - 1) / NTOK * P.NTW;
    int incl = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int acc = incl - run;
    for (int e = e0; e < e1; ++e) {
      tile_start[e] = acc;
      acc += (__ldg(P.counts + e) + NTOK - 1) / NTOK * P.NTW;
    }
    if (lane == 31) tile_start[P.E] = incl;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = tmem_slot;
  const int total = tile_start[P.E];
  const int KB = P.K / DK;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t ph = 0;
    int issued_parity[C::STAGES];
#pragma unroll
    for (int s = 0; s < C::STAGES; ++s) issued_parity[s] = -1;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const DecTile d = dec_tile(t, tile_start, P.E, P.NTW);
      const int cnt = __ldg(P.counts + d.e);
      const int p0 = __ldg(P.offsets + d.e) + d.chunk * NTOK;
      // FC1: 64 gate rows of the tile's activation columns, then the 64 matching up rows
      const int w0 = MODE == DEC_FC1 ? d.e * P.w_rows + d.wt * 64 : d.e * P.w_rows + d.wt * DM;
      const int w1 = w0 + P.N_out;
      int rid[4] = {0, 0, 0, 0};
      if (MODE == DEC_FC1 && lane < NTOK / 4) {
        const int valid = min(NTOK, cnt - d.chunk * NTOK);
        const int first = __ldg(P.sorted_ids + p0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = lane * 4 + i;
          rid[i] = r < valid ? __ldg(P.sorted_ids + p0 + r) : first;
        }
      }
      for (int kb = 0; kb < KB; ++kb) {
        int ok = 1;
        if (lane == 0)
          ok = ptx::mbar_wait(ptx::smem_u32(&empty_bar[stage]), ph ^ 1u, abort_p, DWAIT_NS);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) goto producer_done;
        {
          const uint32_t fb = ptx::smem_u32(&full_bar[stage]);
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(fb, C::STAGE);
            ptx::tma_load_2d(sA(stage), &tmW, kb * DK, w0, fb);
            if (MODE == DEC_FC1) ptx::tma_load_2d(sA(stage) + 64 * 128, &tmW, kb * DK, w1, fb);
            if (MODE == DEC_FC2) ptx::tma_load_2d(sB(stage), &tmX, kb * DK, p0, fb);
          }
          if (MODE == DEC_FC1) {
            __syncwarp();
            if (lane < NTOK / 4)
              ptx::tma_gather4(sB(stage) + lane * 512, &tmX, kb * DK, rid[0], rid[1], rid[2], rid[3], fb);
          }
          issued_parity[stage] = (int)ph;
          if (++stage == C::STAGES) { stage = 0; ph ^= 1u; }
        }
      }
    }
  producer_done:
    if (lane == 0) {
      int dummy = 0;
      for (int s = 0; s < C::STAGES; ++s)
        if (issued_parity[s] >= 0)
          ptx::mbar_wait(ptx::smem_u32(&full_bar[s]), (uint32_t)issued_parity[s], &dummy, DWAIT_NS);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        if (!ptx::mbar_wait(ptx::smem_u32(&tempty_bar[acc]), aph ^ 1u, abort_p, DWAIT_NS)) break;
        ptx::tc_fence_after();
        const uint32_t d0 = tmem_base + (uint32_t)(acc * C::ACC_COLS);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&full_bar[stage]), ph, abort_p, DWAIT_NS)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = sA(stage), b0 = sB(stage);
#pragma unroll
          for (int kk = 0; kk < DK / 16; ++kk)
            ptx::mma_bf16(d0, ptx::sdesc_k128(a0 + kk * 32), ptx::sdesc_k128(b0 + kk * 32), IDESC,
                          (kb | kk) != 0);
          ptx::mma_commit(ptx::smem_u32(&empty_bar[stage]));
          if (++stage == C::STAGES) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
        ptx::mma_commit(ptx::smem_u32(&tfull_bar[acc]));
        if (++acc == 2) { acc = 0; aph ^= 1u; }
      }
      ptx::mma_commit(ptx::smem_u32(&drain_bar));
      int dummy = 0;
      ptx::mbar_wait(ptx::smem_u32(&drain_bar), 0, &dummy, DWAIT_NS);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;     // weight row within the tile
    int acc = 0;
    uint32_t aph = 0, xph = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const DecTile d = dec_tile(t, tile_start, P.E, P.NTW);
      if (!ptx::mbar_wait(ptx::smem_u32(&tfull_bar[acc]), aph, abort_p, DWAIT_NS)) break;
      ptx::tc_fence_after();
      const int cnt = __ldg(P.counts + d.e);
      const int valid = min(NTOK, cnt - d.chunk * NTOK);
      const long p0 = (long)__ldg(P.offsets + d.e) + d.chunk * NTOK;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::ACC_COLS);
      bool ok = true;
      if (MODE == DEC_FC1) {
        // rows 0..63: gate of activation column wt*64 + row; rows 64..127: up of column wt*64 + row - 64
        const bool up = row >= 64;
        const int r64 = row & 63;
        if (up && !ptx::mbar_wait(ptx::smem_u32(&xempty_bar), xph ^ 1u, abort_p, DWAIT_NS)) ok = false;
        const int col = d.wt * 64 + r64;
#pragma unroll
        for (int c0 = 0; c0 < NTOK; c0 += 16) {
          uint32_t v[16];
          ptx::tmem_ld16(taddr + c0, v);
          ptx::tmem_ld_wait();
          if (up) {
            if (ok) {
#pragma unroll
              for (int i = 0; i < 16; ++i) xbuf[(c0 + i) * 64 + r64] = __uint_as_float(v[i]);
            }
          } else {
            if (c0 == 0 && !ptx::mbar_wait(ptx::smem_u32(&xfull_bar), xph, abort_p, DWAIT_NS)) ok = false;
            if (ok) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int c = c0 + i;
                if (c < valid) {
                  const float a = silu(__uint_as_float(v[i])) * xbuf[c * 64 + r64];
                  static_cast<__nv_bfloat16*>(P.out)[(p0 + c) * P.N_out + col] = __float2bfloat16_rn(a);
                }
              }
            }
          }
          if (up && c0 + 16 >= NTOK && ok) ptx::mbar_arrive(ptx::smem_u32(&xfull_bar));
        }
        if (!up && ok) ptx::mbar_arrive(ptx::smem_u32(&xempty_bar));
        xph ^= 1u;
      } else {
        const int col = d.wt * DM + row;
#pragma unroll
        for (int c0 = 0; c0 < NTOK; c0 += 16) {
          uint32_t v[16];
          ptx::tmem_ld16(taddr + c0, v);
          ptx::tmem_ld_wait();
          if (col < P.N_out) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int c = c0 + i;
              if (c < valid) {
                const float w = __ldg(P.sorted_w + p0 + c);
                const long dst = (long)__ldg(P.reverse + p0 + c);
                static_cast<float*>(P.out)[dst * P.N_out + col] = __uint_as_float(v[i]) * w;
              }
            }
          }
        }
      }
      if (!ok) break;
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&tempty_bar[acc]));
      if (++acc == 2) { acc = 0; aph ^= 1u; }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  if (tid == 0 && abort_flag && P.status) atomicOr(P.status, MOE_STATUS_TIMEOUT);
}

template <int MODE, int NTOK>
int launch_dec(const CUtensorMap& w, const CUtensorMap& x, const DecParams& p, long S, cudaStream_t s,
               const char* name) {
  using C = DecCfg<MODE, NTOK>;
  static bool attr[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr[dev]) {
    if (cudaFuncSetAttribute(ffn_decode_kernel<MODE, NTOK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::DSMEM) != cudaSuccess)
      return check_launch(name);
    attr[dev] = true;
  }
  const long max_tiles = ((S + NTOK - 1) / NTOK + p.E) * (long)p.NTW;
  const int grid = (int)(max_tiles < num_sms() ? max_tiles : num_sms());
  if (grid <= 0) return MOE_OK;
  ProfScope ps(name, s);
  ffn_decode_kernel<MODE, NTOK><<<grid, DTHREADS, C::DSMEM, s>>>(w, x, p);
  return check_launch(name);
}

template <int NTOK>
int run_decode(const FfnArgs& a, cudaStream_t s) {
  const long S = (long)a.T * a.k;
  CUtensorMap w1, x1, w2, x2;
  int rc;
  if ((rc = make_tmap(&w1, a.w13, (uint64_t)a.E * 2 * a.I, (uint64_t)a.H, 64))) return rc;
  if ((rc = make_tmap(&x1, a.hidden, (uint64_t)a.T, (uint64_t)a.H, 1))) return rc;
  if ((rc = make_tmap(&w2, a.w2, (uint64_t)a.E * a.H, (uint64_t)a.I, DM))) return rc;
  if ((rc = make_tmap(&x2, a.act, (uint64_t)S, (uint64_t)a.I, NTOK))) return rc;
  DecParams p1{a.counts, a.offsets, a.sorted_ids, a.sorted_w, a.reverse, a.E, a.H, a.I,
               a.I / 64, 2 * a.I, a.act, a.status};
  if ((rc = launch_dec<DEC_FC1, NTOK>(w1, x1, p1, S, s, "ffn_fc1_decode"))) return rc;
  DecParams p2{a.counts, a.offsets, a.sorted_ids, a.sorted_w, a.reverse, a.E, a.I, a.H,
               (a.H + DM - 1) / DM, a.H, a.staging, a.status};
  if ((rc = launch_dec<DEC_FC2, NTOK>(w2, x2, p2, S, s, "ffn_fc2_decode"))) return rc;
  return launch_combine(a.staging, a.T, a.k, a.H, a.dtype, a.out, s);
}

}  // namespace

int launch_ffn_decode(const FfnArgs& a, cudaStream_t s) {
  if ((long)a.T * a.k == 0) return MOE_OK;
  if (a.T <= 16) return run_decode<16>(a, s);
  if (a.T <= 32) return run_decode<32>(a, s);
  return run_decode<64>(a, s);
}

}  // namespace moe
