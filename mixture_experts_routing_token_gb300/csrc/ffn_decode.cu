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
//   warp 0      TMA producer: weight rows (FC1: 128 gate rows and the matching
//               128 up rows; FC2: 128 rows of w2[e]) and the chunk's token rows
//               (FC1: 4-row TMA gathers from `hidden`; FC2: a tiled load of the
//               expert-sorted activation rows), a ring of as many stages as
//               fit in ~205 KB (5-11) to keep enough weight bytes in flight;
//   warp 1      MMA issuer: tcgen05.mma M=128, N=NTOK, K=16 (FC1: two MMAs per
//               step, gate and up into separate accumulators, so one TMEM lane
//               holds the gate and up value of the same activation column);
//   warps 2..5  epilogue: FC1 act = silu(g) * u -> bf16 act row of each token;
//               FC2 y * routing weight -> float32 staging row of the slot.
// All waits are bounded as in the prefill kernel.
//
// Inside the layer call (router logits given, E <= 64, T <= 16) the
// FC1 kernel does not wait for the routing kernel before it streams weights:
// every CTA repeats the top-k selection of the batch's tokens (the same
// comparisons, ties toward the lower expert, so the same experts) and the
// stable expert order of the align step in shared memory, and takes its tiles,
// token ids and activation rows from that. Its epilogue warps wait for the
// routing kernel (griddepcontrol.wait) before they release FC2, which reads
// the routing kernel's outputs, so FC1 also ends after it.
#include "common.cuh"
#include "gating_device.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

constexpr int DM = 128;          // weight rows per tile (MMA M)
constexpr int DK = 64;           // K per stage (one 128-byte swizzle row)
constexpr int DSTAGES_MAX = 12;
constexpr int DTHREADS = 192;
constexpr uint64_t DWAIT_NS = 2000000000ull;   // drains (copies and MMAs already issued)
constexpr int kLocalExperts = 64;   // local routing: a warp per token, two experts per lane (E <= 64),
constexpr int kLocalTokens = 16;    // for at most this many tokens (more cost FC1 what the overlap gains)
constexpr int kLocalSlots = kLocalTokens * kLocalExperts;

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
  int NTW;        // weight tiles per expert: ceil(I / 128) or ceil(H / 128)
  int w_rows;     // rows of one expert's weight matrix: 2I or H
  void* out;      // FC1: act bf16 [S, I]; FC2: staging f32 [S, H]
  int32_t* status;
  const float* logits;   // FC1 only, or null: route the tokens locally (see above)
  int norm, T, k;
  uint64_t wait_ns;       // limit of the waits on the other roles (moe_set_wait_limit_ns)
};

template <int MODE, int NTOK>
struct DecCfg {
  static constexpr int NA = MODE == DEC_FC1 ? 2 : 1;       // weight boxes (and MMAs) per stage
  static constexpr int A_BYTES = NA * DM * DK * 2;
  static constexpr int B_BYTES = NTOK * DK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;            // multiple of 1024
  static constexpr int STAGES_FIT = (205 * 1024) / STAGE;    // ring within ~205 KB of shared memory
  static constexpr int STAGES = STAGES_FIT < 12 ? STAGES_FIT : 12;
  static constexpr int DSMEM = STAGES * STAGE + 1024;
  static constexpr int ACC_COLS = NA * NTOK;                 // one accumulator buffer
  static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS < 32 ? 32 : 2 * ACC_COLS;
  static_assert(STAGE % 1024 == 0, "stage must keep 1024-byte alignment");
  static_assert(STAGES >= 4 && STAGES <= DSTAGES_MAX && DSMEM <= 206 * 1024, "shared memory budget");
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
  __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int tile_start[MOE_MAX_EXPERTS + 1];
  // local routing (FC1 with logits): selected experts, counts, offsets and the
  // expert-sorted token ids
  constexpr bool kCanRoute = MODE == DEC_FC1 && NTOK == kLocalTokens;
  __shared__ int32_t l_idx[kCanRoute ? kLocalSlots : 1];
  __shared__ int32_t l_ids[kCanRoute ? kLocalSlots : 1];
  __shared__ int32_t l_cnt[kCanRoute ? kLocalExperts : 1], l_off[kCanRoute ? kLocalExperts + 1 : 1];
  __shared__ int32_t l_run[kCanRoute ? kLocalExperts : 1];
  extern __shared__ uint8_t dsmem_raw[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool local = kCanRoute && P.logits != nullptr;
  const int32_t* counts = local ? l_cnt : P.counts;
  const int32_t* offsets = local ? l_off : P.offsets;
  const int32_t* sorted_ids = local ? l_ids : P.sorted_ids;
  auto rd = [&](const int32_t* q) -> int { return local ? *q : __ldg(q); };   // shared or global
  const uint32_t dsmem = (ptx::smem_u32(dsmem_raw) + 1023u) & ~1023u;
  auto sA = [&](int s) { return dsmem + (uint32_t)(s * C::STAGE); };
  auto sB = [&](int s) { return dsmem + (uint32_t)(s * C::STAGE + C::A_BYTES); };
  volatile int* abort_p = &abort_flag;

  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
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
    ptx::prefetch_tmap(&tmW);
    ptx::prefetch_tmap(&tmX);
  }
  if (warp == 1) ptx::tmem_alloc(ptx::smem_u32(&tmem_slot), C::TMEM_COLS);
  // Programmatic dependency: FC1 follows the routing kernel, whose counts, offsets
  // and ids it reads from here on. FC2 follows FC1 and reads only its activations
  // (after pdl_wait in the producer); the routing outputs it reads earlier come
  // from two launches back and are complete once FC1 has triggered.
  if (MODE == DEC_FC1 && !local) pdl_wait();
  if (!local) pdl_trigger();
  // the routing of the batch, as the routing kernel computes it
  if (kCanRoute && local) gate::route_block(P.logits, P.T, P.E, P.k, l_idx, l_cnt, l_off, l_ids, l_run);
  if (warp == 2) {   // tile_start[e] = sum over e' < e of ceil(count / NTOK) * NTW
    const int per = (P.E + 31) / 32;
    const int e0 = min(P.E, lane * per), e1 = min(P.E, e0 + per);
    int run = 0;
    for (int e = e0; e < e1; ++e) run += (rd(counts + e) + NTOK - 1) / NTOK * P.NTW;
    int incl = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int acc = incl - run;
    for (int e = e0; e < e1; ++e) {
      tile_start[e] = acc;
      acc += (rd(counts + e) + NTOK - 1) / NTOK * P.NTW;
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
    // FC2: the weight rows of the first stages of this CTA's first tile do not
    // depend on FC1, so they are requested before waiting for its activations.
    int pre = 0;
    if (MODE == DEC_FC2) {
      if ((int)blockIdx.x < total) {
        const DecTile d = dec_tile(blockIdx.x, tile_start, P.E, P.NTW);
        const int w0 = d.e * P.w_rows + d.wt * DM;
        pre = KB < C::STAGES ? KB : C::STAGES;
        if (lane == 0)
          for (int kb = 0; kb < pre; ++kb) {     // fresh ring: stage kb is free
            const uint32_t fb = ptx::smem_u32(&full_bar[kb]);
            ptx::mbar_arrive_expect_tx(fb, C::STAGE);
            ptx::tma_load_2d(sA(kb), &tmW, kb * DK, w0, fb);
          }
      }
      pdl_wait();
    }
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const DecTile d = dec_tile(t, tile_start, P.E, P.NTW);
      const int cnt = rd(counts + d.e);
      const int p0 = rd(offsets + d.e) + d.chunk * NTOK;
      const int w0 = d.e * P.w_rows + d.wt * DM;           // FC1: gate rows; FC2: w2 rows
      const int w1 = w0 + P.N_out;                          // FC1: matching up rows (I further)
      int rid[4] = {0, 0, 0, 0};
      if (MODE == DEC_FC1 && lane < NTOK / 4) {
        const int valid = min(NTOK, cnt - d.chunk * NTOK);
        const int first = rd(sorted_ids + p0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = lane * 4 + i;
          rid[i] = r < valid ? rd(sorted_ids + p0 + r) : first;
        }
      }
      for (int kb = 0; kb < KB; ++kb) {
        const bool preloaded = t == (int)blockIdx.x && kb < pre;   // weights already requested
        int ok = 1;
        if (lane == 0 && !preloaded)
          ok = ptx::mbar_wait(ptx::smem_u32(&empty_bar[stage]), ph ^ 1u, abort_p, P.wait_ns);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) goto producer_done;
        {
          const uint32_t fb = ptx::smem_u32(&full_bar[stage]);
          if (lane == 0) {
            if (!preloaded) {
              ptx::mbar_arrive_expect_tx(fb, C::STAGE);
              ptx::tma_load_2d(sA(stage), &tmW, kb * DK, w0, fb);
            }
            if (MODE == DEC_FC1) ptx::tma_load_2d(sA(stage) + DM * 128, &tmW, kb * DK, w1, fb);
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
        if (!ptx::mbar_wait(ptx::smem_u32(&tempty_bar[acc]), aph ^ 1u, abort_p, P.wait_ns)) break;
        ptx::tc_fence_after();
        const uint32_t d0 = tmem_base + (uint32_t)(acc * C::ACC_COLS);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&full_bar[stage]), ph, abort_p, P.wait_ns)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = sA(stage), b0 = sB(stage);
#pragma unroll
          for (int kk = 0; kk < DK / 16; ++kk) {
            const uint64_t bd = ptx::sdesc_k128(b0 + kk * 32);
            ptx::mma_bf16(d0, ptx::sdesc_k128(a0 + kk * 32), bd, IDESC, (kb | kk) != 0);
            if (MODE == DEC_FC1)
              ptx::mma_bf16(d0 + NTOK, ptx::sdesc_k128(a0 + DM * 128 + kk * 32), bd, IDESC, (kb | kk) != 0);
          }
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
    const int row = q * 32 + lane;     // weight row within the tile = output column offset
    int acc = 0;
    uint32_t aph = 0;
    if (local) {   // FC2 reads the routing kernel's outputs: release it only once they exist
      pdl_wait();
      pdl_trigger();
    }
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const DecTile d = dec_tile(t, tile_start, P.E, P.NTW);
      if (!ptx::mbar_wait(ptx::smem_u32(&tfull_bar[acc]), aph, abort_p, P.wait_ns)) break;
      ptx::tc_fence_after();
      const int cnt = rd(counts + d.e);
      const int valid = min(NTOK, cnt - d.chunk * NTOK);
      const long p0 = (long)rd(offsets + d.e) + d.chunk * NTOK;
      const int col = d.wt * DM + row;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::ACC_COLS);
#pragma unroll
      for (int c0 = 0; c0 < NTOK; c0 += 16) {
        uint32_t v[16], u[16];
        ptx::tmem_ld16(taddr + c0, v);
        if (MODE == DEC_FC1) ptx::tmem_ld16(taddr + NTOK + c0, u);
        ptx::tmem_ld_wait();
        if (col < P.N_out) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = c0 + i;
            if (c < valid) {
              if (MODE == DEC_FC1) {
                const float a = silu(__uint_as_float(v[i])) * __uint_as_float(u[i]);
                static_cast<__nv_bfloat16*>(P.out)[(p0 + c) * P.N_out + col] = __float2bfloat16_rn(a);
              } else {
                const float w = __ldg(P.sorted_w + p0 + c);
                const long dst = (long)__ldg(P.reverse + p0 + c);
                static_cast<float*>(P.out)[dst * P.N_out + col] = __uint_as_float(v[i]) * w;
              }
            }
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
    ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  if (tid == 0 && abort_flag && P.status) atomicOr(P.status, MOE_STATUS_TIMEOUT);
}

template <int MODE, int NTOK>
int launch_dec(const CUtensorMap& w, const CUtensorMap& x, const DecParams& p, long S, cudaStream_t s,
               const char* name) {
  using C = DecCfg<MODE, NTOK>;
  if (int rc = ensure_smem_limit(ffn_decode_kernel<MODE, NTOK>, C::DSMEM, name)) return rc;
  const long max_tiles = ((S + NTOK - 1) / NTOK + p.E) * (long)p.NTW;
  const int grid = (int)(max_tiles < num_sms() ? max_tiles : num_sms());
  if (grid <= 0) return MOE_OK;
  ProfScope ps(name, s);
  const cudaError_t e = launch_pdl(ffn_decode_kernel<MODE, NTOK>, grid, DTHREADS, C::DSMEM, s, w, x, p);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", name, cudaGetErrorString(e));
  return check_launch(name);
}

template <int NTOK>
int run_decode(const FfnArgs& a, cudaStream_t s) {
  const long S = (long)a.T * a.k;
  CUtensorMap w1, x1, w2, x2;
  int rc;
  if ((rc = make_tmap(&w1, a.w13, (uint64_t)a.E * 2 * a.I, (uint64_t)a.H, DM))) return rc;
  if ((rc = make_tmap(&x1, a.hidden, (uint64_t)a.T, (uint64_t)a.H, 1))) return rc;
  if ((rc = make_tmap(&w2, a.w2, (uint64_t)a.E * a.H, (uint64_t)a.I, DM))) return rc;
  if ((rc = make_tmap(&x2, a.act, (uint64_t)S, (uint64_t)a.I, NTOK))) return rc;
  const bool local = a.logits && a.E <= kLocalExperts && a.T <= kLocalTokens;
  DecParams p1{a.counts, a.offsets, a.sorted_ids, a.sorted_w, a.reverse, a.E, a.H, a.I,
               (a.I + DM - 1) / DM, 2 * a.I, a.act, a.status, local ? a.logits : nullptr, a.norm, a.T, a.k,
               wait_limit_ns()};
  if ((rc = launch_dec<DEC_FC1, NTOK>(w1, x1, p1, S, s, "ffn_fc1_decode"))) return rc;
  DecParams p2{a.counts, a.offsets, a.sorted_ids, a.sorted_w, a.reverse, a.E, a.I, a.H,
               (a.H + DM - 1) / DM, a.H, a.staging, a.status, nullptr, 0, a.T, a.k, wait_limit_ns()};
  if ((rc = launch_dec<DEC_FC2, NTOK>(w2, x2, p2, S, s, "ffn_fc2_decode"))) return rc;
  return launch_combine(a.staging, 0, a.T, a.k, a.H, a.dtype, a.out, s);
}

}  // namespace

int launch_ffn_decode(const FfnArgs& a, cudaStream_t s) {
  if ((long)a.T * a.k == 0) return MOE_OK;
  if (ffn_gemv_applies(a.dtype, a.T, a.H, a.I, a.k)) return launch_ffn_gemv(a, s);
  if (a.T <= 16) return run_decode<16>(a, s);
  if (a.T <= 32) return run_decode<32>(a, s);
  return run_decode<64>(a, s);
}

}  // namespace moe
