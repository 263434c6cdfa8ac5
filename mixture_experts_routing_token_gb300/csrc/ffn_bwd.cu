// Backward of the grouped expert FFN and the weighted k-sum, bf16 on the
// tcgen05 tensor cores (2-SM clusters, cta_group::2, M = 256 x N = 256 x K = 16,
// f32 accumulation in TMEM).
//
// The forward is project_6 moe_expert_gemm.cpp, moe_prefill_experts (FC1 with
// w13[e], silu_and_mul, FC2 with w2[e], routing weight) and mlc-llm
// moe_misc.py, scatter_output / moe_sum. Its derivative, per routed slot p
// (token t, expert e, weight w_p; g, u the gate / up pre-activations, s =
// sigmoid(g), a = g s u rounded to bf16 as the forward rounds it):
//   d w_p = <dO[t], y_p> = <dO[t] W2, a_p>      dy_p = w_p dO[t]
//   dW2[e] = sum_p dy_p a_p^T                    da_p = w_p (dO[t] W2)
//   dg = da u s (1 + g (1 - s)),  du = da g s    dW13[e] = sum_p [dg du]_p^T x_t
//   dx_t = sum over the token's slots of [dg du]_p W13[e]
//
// Rows live in a padded expert-sorted order: expert e's rows start at poff[e],
// a multiple of 64, and its rows past counts[e] up to the next multiple of 64
// are zero. The weight gradients reduce over those rows in whole 64-row
// k-steps without masking.
//
// Launches, in stream order (each waits on its predecessor with a programmatic
// dependency, as in the forward):
//   bwd_pad         poff from counts;
//   bwd_gather      xs = hidden rows, dos = dO rows, dys = w_p dO rows (bf16);
// then, for H above kFusedMaxH:
//   RECOMPUTE       [g u] = xs W13^T -> gu (f32), act = bf16(silu(g) u);
//   DGRAD_A         G = dos W2 (B MN-major) -> dgu = bf16([dg du]) with
//                   da = w_p G, and per-tile partials of d w_p = <G, act>;
// or, for H up to kFusedMaxH, both in one kernel:
//   FUSED_A         per tile G and [g u] into TMEM, the same epilogue outputs
//                   without the f32 gu round trip through HBM;
//   zero_dropped    (staging rows of dropped slots);
//   DGRAD_X         dgu W13 (B MN-major) -> staging[reverse[p]] (f32);
//   combine         d_hidden[t] = sum_j staging[t k + j];
//   WGRAD dW2       dys^T act (A and B MN-major) over the expert's rows;
//   WGRAD dW13      dgu^T xs;
//   bwd_zero_empty  (weight gradients of experts without rows);
//   bwd_dw_reduce   d_weights[reverse[p]] = sum of the partials.
// The pair-kernel machinery (barriers, bounded waits, TMEM double buffer,
// cluster teardown) is the forward's (ffn_tc_pair.cu); an MN-major operand is
// two 64-column TMA boxes per SM, described by pair::sdesc_mn128.
#include <algorithm>

#include "common.cuh"
#include "pair_ptx.cuh"

namespace moe {
namespace {

using namespace pair;

constexpr int BM = 128;                 // rows of A per SM (256 per pair)
constexpr int BK = 64;
constexpr int BN = 256;                 // MMA N
constexpr int NSTAGE = 6;
constexpr int A_BYTES = BM * BK * 2;    // 16 KB
constexpr int B_BYTES = (BN / 2) * BK * 2;
constexpr int STAGE = A_BYTES + B_BYTES;
constexpr int DSMEM = NSTAGE * STAGE + 1024;
// Epilogue warps: 4 (one per TMEM lane quarter) or 8 (two per quarter, each
// draining every other 32-column chunk). The recompute / dA epilogues, which
// move several values per output element, measured faster with 8; the dX and
// weight-gradient ones with 4.
constexpr int MAX_THREADS = (2 + 8) * 32;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr int kRowPad = 64;
constexpr uint32_t kMnBlock = 64 * BK * 2;   // bytes between the two 64-column MN boxes
constexpr int kFusedMaxH = 3072;

enum { RECOMPUTE = 0, DGRAD_A = 1, DGRAD_X = 2, WGRAD = 3, FUSED_A = 4 };

template <int KIND>
constexpr int epi_warps() { return (KIND == RECOMPUTE || KIND == DGRAD_A || KIND == FUSED_A) ? 8 : 4; }
template <int KIND>
constexpr int kind_threads() { return (2 + epi_warps<KIND>()) * 32; }

template <int KIND>
struct Major {
  static constexpr int a_mn = KIND == WGRAD ? 1 : 0;
  static constexpr int b_mn = KIND == RECOMPUTE ? 0 : 1;
};

struct BwdParams {
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* poff;
  const float* sorted_w;
  const int32_t* reverse;
  int E, H, I;
  int K;            // reduction length of the row kinds (H or 2I)
  int NT;           // N tiles (per M tile of an expert; per expert for WGRAD)
  int MT;           // WGRAD: M tiles per expert
  int b_rows;       // per-expert row stride of the B tensor
  int M_dim, N_dim; // WGRAD output [E, M_dim, N_dim]
  float* gu;
  __nv_bfloat16* act;
  __nv_bfloat16* dgu;
  float* dwp;
  float* staging;
  __nv_bfloat16* dw;
  int dw_sector;    // WGRAD: dw is 32-byte aligned, so its rows take whole-sector stores
  int32_t* status;
};

struct BTile {
  int e, m_tile, n_tile, ksteps;
};

template <int KIND>
__device__ __forceinline__ int expert_tiles(int cnt, const BwdParams& P) {
  if (KIND == WGRAD) return cnt > 0 ? P.MT * P.NT : 0;
  return (cnt + 2 * BM - 1) / (2 * BM) * P.NT;
}

template <int KIND>
__device__ __forceinline__ BTile btile(int t, const int* tile_start, const BwdParams& P) {
  int lo = 0, hi = P.E;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int local = t - tile_start[lo];
  BTile d;
  d.e = lo;
  if (KIND == WGRAD) {
    // the operand with more columns is walked once (outer), the other one sweeps
    // past it (inner) and stays in L2 across the concurrently running tiles
    if (P.M_dim >= P.N_dim) {
      d.m_tile = local / P.NT;
      d.n_tile = local - d.m_tile * P.NT;
    } else {
      d.n_tile = local / P.MT;
      d.m_tile = local - d.n_tile * P.MT;
    }
    d.ksteps = (__ldg(P.poff + lo + 1) - __ldg(P.poff + lo)) / BK;
  } else {
    // as in the forward tile list: the operand with fewer tiles of this expert
    // stays in L2 (A and B tiles are both 256 rows x K)
    const int mt = (__ldg(P.counts + lo) + 2 * BM - 1) / (2 * BM);
    if (mt > P.NT) {
      d.m_tile = local / P.NT;
      d.n_tile = local - d.m_tile * P.NT;
    } else {
      d.n_tile = local / mt;
      d.m_tile = local - d.n_tile * mt;
    }
    d.ksteps = P.K / BK;
  }
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 32 values of one row: workspace rows (32-byte aligned) move in whole 32-byte
// sectors; store_bf16x32_16 is for caller buffers (16-byte aligned).
__device__ __forceinline__ void load_f32x32(const float* p, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t q[8];
    ld_v8(p + 8 * i, q);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[8 * i + j] = __uint_as_float(q[j]);
  }
}

__device__ __forceinline__ void store_f32x32(float* p, const float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = v[8 * i + j];
    st_v8(p + 8 * i, q);
  }
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* p, const float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = pack_bf16x2(v[16 * i + 2 * j], v[16 * i + 2 * j + 1]);
    st_v8(p + 16 * i, q);
  }
}

__device__ __forceinline__ void store_bf16x32_16(__nv_bfloat16* p, const float (&v)[32]) {
  uint4* d = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    d[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                      pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* p, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint32_t w[8];
    ld_v8(p + 16 * i, w);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[16 * i + 2 * j] = __uint_as_float(w[j] << 16);
      v[16 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  }
}

template <int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(MAX_THREADS, 1)
    bwd_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const BwdParams P) {
  constexpr int A_MN = Major<KIND>::a_mn, B_MN = Major<KIND>::b_mn;
  constexpr uint32_t IDESC = idesc_bf16_f32_major(2 * BM, BN, A_MN, B_MN);
  __shared__ __align__(8) uint64_t full_bar[NSTAGE], empty_bar[NSTAGE];
  __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int tile_start[MOE_MAX_EXPERTS + 1];
  extern __shared__ uint8_t dsmem_raw[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int cluster_id = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  const uint32_t dsmem = (ptx::smem_u32(dsmem_raw) + 1023u) & ~1023u;
  auto sA = [&](int s) { return dsmem + (uint32_t)(s * STAGE); };
  auto sB = [&](int s) { return dsmem + (uint32_t)(s * STAGE + A_BYTES); };
  volatile int* abort_p = &abort_flag;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&tfull_bar[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&tempty_bar[b]), 2 * epi_warps<KIND>());
    }
    ptx::mbar_init(ptx::smem_u32(&drain_bar), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     ptx::smem_u32(&tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  ptx::tc_fence_before();
  __syncthreads();
  cluster_sync();
  ptx::tc_fence_after();
  pdl_wait();          // poff and the operands written by the previous launches are read from here on
  pdl_trigger();
  if (warp == 2) {     // tile_start[e] = tiles of the experts before e
    const int per = (P.E + 31) / 32;
    const int e0 = min(P.E, lane * per), e1 = min(P.E, e0 + per);
    int run = 0;
    for (int e = e0; e < e1; ++e) run += expert_tiles<KIND>(__ldg(P.counts + e), P);
    int incl = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int acc = incl - run;
    for (int e = e0; e < e1; ++e) {
      tile_start[e] = acc;
      acc += expert_tiles<KIND>(__ldg(P.counts + e), P);
    }
    if (lane == 31) tile_start[P.E] = incl;
  }
  __syncthreads();
  const uint32_t tmem_base = tmem_slot;
  const int total = tile_start[P.E];

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      for (int t = cluster_id; t < total; t += nclusters) {
        const BTile ti = btile<KIND>(t, tile_start, P);
        const int pbase = __ldg(P.poff + ti.e);
        for (int kb = 0; kb < ti.ksteps; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&empty_bar[stage]), ph ^ 1u, abort_p, WAIT_NS)) goto producer_done;
          const uint32_t fb_local = ptx::smem_u32(&full_bar[stage]);
          if (leader) ptx::mbar_arrive_expect_tx(fb_local, 2 * STAGE);
          const uint32_t fb = map_to_rank(fb_local, 0);
          if (A_MN) {   // WGRAD: A = [rows][M_dim], this SM's 128 of the tile's 256 M columns
            const int x = ti.m_tile * (2 * BM) + (int)rank * BM, y = pbase + kb * BK;
            tma_load_2d_pair(sA(stage), &tmA, x, y, fb);
            tma_load_2d_pair(sA(stage) + kMnBlock, &tmA, x + 64, y, fb);
          } else {      // row kinds: A = this SM's 128 of the tile's 256 padded rows
            tma_load_2d_pair(sA(stage), &tmA, kb * BK, pbase + ti.m_tile * (2 * BM) + (int)rank * BM, fb);
          }
          if (KIND == RECOMPUTE) {   // gate rows on SM 0, the matching up rows on SM 1
            const int b_row = ti.e * P.b_rows + ti.n_tile * 128 + (leader ? 0 : P.I);
            tma_load_2d_pair(sB(stage), &tmB, kb * BK, b_row, fb);
          } else {                   // B MN-major: this SM's 128 of the tile's 256 N columns
            const int x = ti.n_tile * BN + (int)rank * 128;
            const int y = (KIND == WGRAD ? pbase : ti.e * P.b_rows) + kb * BK;
            tma_load_2d_pair(sB(stage), &tmB, x, y, fb);
            tma_load_2d_pair(sB(stage) + kMnBlock, &tmB, x + 64, y, fb);
          }
          if (++stage == NSTAGE) { stage = 0; ph ^= 1u; }
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader CTA)
    if (leader && lane == 0) {
      int stage = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      for (int t = cluster_id; t < total; t += nclusters) {
        const BTile ti = btile<KIND>(t, tile_start, P);
        if (!ptx::mbar_wait(ptx::smem_u32(&tempty_bar[acc]), aph ^ 1u, abort_p, WAIT_NS)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < ti.ksteps; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&full_bar[stage]), ph, abort_p, WAIT_NS)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = sA(stage), b0 = sB(stage);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = A_MN ? sdesc_mn128(a0 + kk * 2048, kMnBlock) : ptx::sdesc_k128(a0 + kk * 32);
            const uint64_t bd = B_MN ? sdesc_mn128(b0 + kk * 2048, kMnBlock) : ptx::sdesc_k128(b0 + kk * 32);
            mma_pair(d_tmem, ad, bd, IDESC, (kb | kk) != 0);
          }
          commit_pair(ptx::smem_u32(&empty_bar[stage]), 0x3);
          if (++stage == NSTAGE) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
        commit_pair(ptx::smem_u32(&tfull_bar[acc]), 0x3);
        if (++acc == 2) { acc = 0; aph ^= 1u; }
      }
      commit_pair(ptx::smem_u32(&drain_bar), 0x1);
      int dummy = 0;
      ptx::mbar_wait(ptx::smem_u32(&drain_bar), 0, &dummy, WAIT_NS);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    constexpr int NH = epi_warps<KIND>() / 4;   // warps per lane quarter
    const int half = (warp - 2) >> 2;           // which 32-column chunks it drains
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
    for (int t = cluster_id; t < total; t += nclusters) {
      const BTile ti = btile<KIND>(t, tile_start, P);
      if (!ptx::mbar_wait(ptx::smem_u32(&tfull_bar[acc]), aph, abort_p, WAIT_NS)) break;
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      if (KIND == WGRAD) {
        const int m = ti.m_tile * (2 * BM) + (int)rank * BM + row;
        __nv_bfloat16* dst = P.dw + ((long)ti.e * P.M_dim + m) * P.N_dim;
#pragma unroll 1
        for (int c = half; c < BN / 32; c += NH) {
          uint32_t y[32];
          ptx::tmem_ld32(taddr + c * 32, y);
          ptx::tmem_ld_wait();
          const int n0 = ti.n_tile * BN + c * 32;
          if (m < P.M_dim && n0 < P.N_dim) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(y[i]);
            if (P.dw_sector) store_bf16x32(dst + n0, v);
            else store_bf16x32_16(dst + n0, v);
          }
        }
      } else {
        const int cnt = __ldg(P.counts + ti.e);
        const int pcnt = __ldg(P.poff + ti.e + 1) - __ldg(P.poff + ti.e);
        const int r = ti.m_tile * (2 * BM) + (int)rank * BM + row;   // row within the expert
        const bool in_seg = r < pcnt;                                // a real or a zero pad row
        const bool real = r < cnt;
        const long pp = (long)__ldg(P.poff + ti.e) + r;              // padded row
        const int I = P.I, H = P.H;
        if (KIND == RECOMPUTE) {
#pragma unroll 1
          for (int c = half; c < 4; c += NH) {
            uint32_t g[32], u[32];
            ptx::tmem_ld32(taddr + c * 32, g);
            ptx::tmem_ld32(taddr + 128 + c * 32, u);
            ptx::tmem_ld_wait();
            const int col0 = ti.n_tile * 128 + c * 32;
            if (in_seg && col0 < I) {
              float gv[32], uv[32], av[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                gv[i] = __uint_as_float(g[i]);
                uv[i] = __uint_as_float(u[i]);
                av[i] = silu(gv[i]) * uv[i];
              }
              store_f32x32(P.gu + pp * 2 * I + col0, gv);
              store_f32x32(P.gu + pp * 2 * I + I + col0, uv);
              store_bf16x32(P.act + pp * I + col0, av);
            }
          }
        } else if (KIND == DGRAD_A) {
          const float wp = real ? __ldg(P.sorted_w + __ldg(P.offsets + ti.e) + r) : 0.0f;
          float dot = 0.0f;
#pragma unroll 1
          for (int c = half; c < BN / 32; c += NH) {
            uint32_t G[32];
            ptx::tmem_ld32(taddr + c * 32, G);
            ptx::tmem_ld_wait();
            const int i0 = ti.n_tile * BN + c * 32;
            if (in_seg && i0 < I) {
              float av[32];
              load_bf16x32(P.act + pp * I + i0, av);
#pragma unroll
              for (int i = 0; i < 32; ++i) dot = fmaf(__uint_as_float(G[i]), av[i], dot);
              float gv[32], uv[32];
              load_f32x32(P.gu + pp * 2 * I + i0, gv);
              load_f32x32(P.gu + pp * 2 * I + I + i0, uv);
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const float da = wp * __uint_as_float(G[i]);
                const float s = 1.0f / (1.0f + expf(-gv[i]));
                const float dg = da * uv[i] * s * (1.0f + gv[i] * (1.0f - s));
                const float du = da * gv[i] * s;
                gv[i] = dg;
                uv[i] = du;
              }
              store_bf16x32(P.dgu + pp * 2 * I + i0, gv);
              store_bf16x32(P.dgu + pp * 2 * I + I + i0, uv);
            }
          }
          if (in_seg) P.dwp[(pp * P.NT + ti.n_tile) * 2 + half] = dot;
        } else {   // DGRAD_X
          const long dst_row = real ? (long)__ldg(P.reverse + __ldg(P.offsets + ti.e) + r) : 0;
#pragma unroll 1
          for (int c = half; c < BN / 32; c += NH) {
            uint32_t y[32];
            ptx::tmem_ld32(taddr + c * 32, y);
            ptx::tmem_ld_wait();
            const int h0 = ti.n_tile * BN + c * 32;
            if (real && h0 < H) {
              float v[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(y[i]);
              store_f32x32(P.staging + dst_row * H + h0, v);
            }
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_remote(map_to_rank(ptx::smem_u32(&tempty_bar[acc]), 0));
      if (++acc == 2) { acc = 0; aph ^= 1u; }
    }
  }

  if (*abort_p) {   // after a timeout, let copies in flight land before the smem is released
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < 1000000ull) {
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
  if (tid == 0 && abort_flag && P.status) atomicOr(P.status, MOE_STATUS_TIMEOUT);
}

// ---- FC1 recomputed and dA, fused ----------------------------------------------
//
// One tile = 256 padded rows x 128 features of expert e. The leader issues two
// MMA phases per tile:
//   G phase:  G = dO rows . W2[e][:, features]      N = 128, W2 as an MN-major
//             B operand (each SM holds 64 of the 128 columns);
//   gu phase: [g | u] = x rows . [W1; W3][e]^T      N = 256, gate rows of the
//             128 features on SM 0, the matching up rows on SM 1 (as FC1).
// TMEM: [g | u] in columns 0..255 (one buffer), G in 256..383 and 384..511
// (two buffers), so the next tile's G phase runs while the epilogue drains the
// current tile. The epilogue forms s = sigmoid(g), a = bf16(g s u) (written:
// the dW2 operand), the partial <G, a> of d w_p, da = w_p G, and writes
// dg = da u s (1 + g (1 - s)), du = da g s as bf16.
constexpr int FA_FEAT = 128;
constexpr int FA_G_BYTES = (FA_FEAT / 2) * BK * 2;   // this SM's 64 columns of W2 per k-step

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(MAX_THREADS, 1)
    bwd_fused_a_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmW13, const __grid_constant__ CUtensorMap tmW2,
                       const BwdParams P) {
  constexpr uint32_t IDESC_G = idesc_bf16_f32_major(2 * BM, FA_FEAT, 0, 1);
  constexpr uint32_t IDESC_GU = idesc_bf16_f32_major(2 * BM, BN, 0, 0);
  __shared__ __align__(8) uint64_t full_bar[NSTAGE], empty_bar[NSTAGE];
  __shared__ __align__(8) uint64_t tfull_bar, gu_empty_bar, g_empty_bar[2], drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int tile_start[MOE_MAX_EXPERTS + 1];
  extern __shared__ uint8_t dsmem_raw[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int cluster_id = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  const uint32_t dsmem = (ptx::smem_u32(dsmem_raw) + 1023u) & ~1023u;
  auto sA = [&](int s) { return dsmem + (uint32_t)(s * STAGE); };
  auto sB = [&](int s) { return dsmem + (uint32_t)(s * STAGE + A_BYTES); };
  volatile int* abort_p = &abort_flag;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&tfull_bar), 1);
    ptx::mbar_init(ptx::smem_u32(&gu_empty_bar), 2 * epi_warps<FUSED_A>());
    ptx::mbar_init(ptx::smem_u32(&g_empty_bar[0]), 2 * epi_warps<FUSED_A>());
    ptx::mbar_init(ptx::smem_u32(&g_empty_bar[1]), 2 * epi_warps<FUSED_A>());
    ptx::mbar_init(ptx::smem_u32(&drain_bar), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmX);
    ptx::prefetch_tmap(&tmDO);
    ptx::prefetch_tmap(&tmW13);
    ptx::prefetch_tmap(&tmW2);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     ptx::smem_u32(&tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  ptx::tc_fence_before();
  __syncthreads();
  cluster_sync();
  ptx::tc_fence_after();
  pdl_wait();
  pdl_trigger();
  if (warp == 2) {     // tile_start[e] = tiles of the experts before e
    const int per = (P.E + 31) / 32;
    const int e0 = min(P.E, lane * per), e1 = min(P.E, e0 + per);
    int run = 0;
    for (int e = e0; e < e1; ++e) run += expert_tiles<DGRAD_X>(__ldg(P.counts + e), P);
    int incl = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int acc = incl - run;
    for (int e = e0; e < e1; ++e) {
      tile_start[e] = acc;
      acc += expert_tiles<DGRAD_X>(__ldg(P.counts + e), P);
    }
    if (lane == 31) tile_start[P.E] = incl;
  }
  __syncthreads();
  const uint32_t tmem_base = tmem_slot;
  const int total = tile_start[P.E];
  const int KB = P.K / BK;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      for (int t = cluster_id; t < total; t += nclusters) {
        const BTile ti = btile<DGRAD_X>(t, tile_start, P);
        const int a_row = __ldg(P.poff + ti.e) + ti.m_tile * (2 * BM) + (int)rank * BM;
        for (int step = 0; step < 2 * KB; ++step) {
          const bool gphase = step < KB;
          const int kb = gphase ? step : step - KB;
          if (!ptx::mbar_wait(ptx::smem_u32(&empty_bar[stage]), ph ^ 1u, abort_p, WAIT_NS)) goto producer_done;
          const uint32_t fb_local = ptx::smem_u32(&full_bar[stage]);
          if (leader) ptx::mbar_arrive_expect_tx(fb_local, gphase ? 2 * (A_BYTES + FA_G_BYTES) : 2 * STAGE);
          const uint32_t fb = map_to_rank(fb_local, 0);
          if (gphase) {
            tma_load_2d_pair(sA(stage), &tmDO, kb * BK, a_row, fb);
            tma_load_2d_pair(sB(stage), &tmW2, ti.n_tile * FA_FEAT + (int)rank * (FA_FEAT / 2), ti.e * P.H + kb * BK,
                             fb);
          } else {
            tma_load_2d_pair(sA(stage), &tmX, kb * BK, a_row, fb);
            tma_load_2d_pair(sB(stage), &tmW13, kb * BK,
                             ti.e * 2 * P.I + ti.n_tile * FA_FEAT + (leader ? 0 : P.I), fb);
          }
          if (++stage == NSTAGE) { stage = 0; ph ^= 1u; }
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader CTA)
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      uint32_t it = 0;
      bool ok = true;
      for (int t = cluster_id; t < total && ok; t += nclusters, ++it) {
        const uint32_t gb = it & 1u;
        for (int phase = 0; phase < 2 && ok; ++phase) {
          uint32_t d_tmem;
          if (phase == 0) {
            if (!ptx::mbar_wait(ptx::smem_u32(&g_empty_bar[gb]), ((it >> 1) & 1u) ^ 1u, abort_p, WAIT_NS)) {
              ok = false;
              break;
            }
            d_tmem = tmem_base + (uint32_t)(BN + gb * FA_FEAT);
          } else {
            if (!ptx::mbar_wait(ptx::smem_u32(&gu_empty_bar), (it & 1u) ^ 1u, abort_p, WAIT_NS)) {
              ok = false;
              break;
            }
            d_tmem = tmem_base;
          }
          ptx::tc_fence_after();
          for (int kb = 0; kb < KB; ++kb) {
            if (!ptx::mbar_wait(ptx::smem_u32(&full_bar[stage]), ph, abort_p, WAIT_NS)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t a0 = sA(stage), b0 = sB(stage);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              if (phase == 0)
                mma_pair(d_tmem, ptx::sdesc_k128(a0 + kk * 32), sdesc_mn128(b0 + kk * 2048, kMnBlock), IDESC_G,
                         (kb | kk) != 0);
              else
                mma_pair(d_tmem, ptx::sdesc_k128(a0 + kk * 32), ptx::sdesc_k128(b0 + kk * 32), IDESC_GU,
                         (kb | kk) != 0);
            }
            commit_pair(ptx::smem_u32(&empty_bar[stage]), 0x3);
            if (++stage == NSTAGE) { stage = 0; ph ^= 1u; }
          }
        }
        if (ok) commit_pair(ptx::smem_u32(&tfull_bar), 0x3);
      }
      commit_pair(ptx::smem_u32(&drain_bar), 0x1);
      int dummy = 0;
      ptx::mbar_wait(ptx::smem_u32(&drain_bar), 0, &dummy, WAIT_NS);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    const int half = (warp - 2) >> 2;    // which 32-column chunks it drains (every other one)
    const int row = q * 32 + lane;
    uint32_t it = 0;
    for (int t = cluster_id; t < total; t += nclusters, ++it) {
      const BTile ti = btile<DGRAD_X>(t, tile_start, P);
      if (!ptx::mbar_wait(ptx::smem_u32(&tfull_bar), it & 1u, abort_p, WAIT_NS)) break;
      ptx::tc_fence_after();
      const uint32_t gb = it & 1u;
      const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
      const int cnt = __ldg(P.counts + ti.e);
      const int pcnt = __ldg(P.poff + ti.e + 1) - __ldg(P.poff + ti.e);
      const int r = ti.m_tile * (2 * BM) + (int)rank * BM + row;
      const bool in_seg = r < pcnt;
      const bool real = r < cnt;
      const long pp = (long)__ldg(P.poff + ti.e) + r;
      const int I = P.I;
      const float wp = real ? __ldg(P.sorted_w + __ldg(P.offsets + ti.e) + r) : 0.0f;
      float dot = 0.0f;
#pragma unroll 1
      for (int c = half; c < FA_FEAT / 32; c += 2) {
        uint32_t G[32], g[32], u[32];
        ptx::tmem_ld32(lane_base + BN + gb * FA_FEAT + c * 32, G);
        ptx::tmem_ld32(lane_base + c * 32, g);
        ptx::tmem_ld32(lane_base + 128 + c * 32, u);
        ptx::tmem_ld_wait();
        const int i0 = ti.n_tile * FA_FEAT + c * 32;
        if (in_seg && i0 < I) {
          float av[32], dg[32], du[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float gv = __uint_as_float(g[i]), uv = __uint_as_float(u[i]), Gv = __uint_as_float(G[i]);
            const float s = 1.0f / (1.0f + expf(-gv));
            const float a = __bfloat162float(__float2bfloat16_rn(gv * s * uv));
            av[i] = a;
            dot = fmaf(Gv, a, dot);
            const float da = wp * Gv;
            dg[i] = da * uv * s * (1.0f + gv * (1.0f - s));
            du[i] = da * gv * s;
          }
          store_bf16x32(P.act + pp * I + i0, av);
          store_bf16x32(P.dgu + pp * 2 * I + i0, dg);
          store_bf16x32(P.dgu + pp * 2 * I + I + i0, du);
        }
      }
      if (in_seg) P.dwp[(pp * P.NT + ti.n_tile) * 2 + half] = dot;
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        arrive_remote(map_to_rank(ptx::smem_u32(&gu_empty_bar), 0));
        arrive_remote(map_to_rank(ptx::smem_u32(&g_empty_bar[gb]), 0));
      }
    }
  }

  if (*abort_p) {
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < 1000000ull) {
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                 : "memory");
  }
  if (tid == 0 && abort_flag && P.status) atomicOr(P.status, MOE_STATUS_TIMEOUT);
}

// ---- small kernels ------------------------------------------------------------

// poff[e] = sum over e' < e of counts[e'] rounded up to kRowPad; one CTA of 1024 threads.
__global__ void __launch_bounds__(1024) bwd_pad_kernel(const int32_t* __restrict__ counts, int E,
                                                       int32_t* __restrict__ poff) {
  __shared__ int wsum[32];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int v = tid < E ? (__ldg(counts + tid) + kRowPad - 1) / kRowPad * kRowPad : 0;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += o;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  const int excl = (warp ? wsum[warp - 1] : 0) + incl - v;
  if (tid < E) poff[tid] = excl;
  if (tid == E - 1) poff[E] = excl + v;
}

__device__ __forceinline__ int find_segment(const int* seg, int E, int q) {   // seg[e] <= q < seg[e + 1]
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (seg[mid] <= q) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Padded rows q: xs = hidden[t], dos = dO[t], dys = bf16(w_p * dO[t]) for the row's
// slot p; zeros on pad rows. 16-byte chunks (8 bf16).
__global__ void __launch_bounds__(256) bwd_gather_kernel(
    const uint4* __restrict__ hidden, const uint4* __restrict__ dout, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ poff, const int32_t* __restrict__ ids,
    const float* __restrict__ sw, int E, int H8, int sh, long Pmax, uint4* __restrict__ xs,
    uint4* __restrict__ dos, uint4* __restrict__ dys) {
  extern __shared__ int s_poff[];
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_poff[e] = __ldg(poff + e);
  __syncthreads();
  const long n = min(Pmax, (long)s_poff[E]) * H8;
  const long stride = (long)gridDim.x * blockDim.x;
  constexpr int U = 4;   // rows chunks per thread loaded before any store (more reads in flight)
  for (long i0 = (long)blockIdx.x * blockDim.x + threadIdx.x; i0 < n; i0 += U * stride) {
    uint4 x[U], d[U];
    float w[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      x[u] = make_uint4(0, 0, 0, 0);
      d[u] = x[u];
      w[u] = 0.0f;
      const long i = i0 + u * stride;
      if (i < n) {
        const int q = (int)div_idx(i, H8, sh);
        const int c = (int)(i - (long)q * H8);
        const int e = find_segment(s_poff, E, q);
        const int r = q - s_poff[e];
        if (r < __ldg(counts + e)) {
          const int p = __ldg(offsets + e) + r;
          const long t = __ldg(ids + p);
          w[u] = __ldg(sw + p);
          x[u] = __ldg(hidden + t * H8 + c);
          d[u] = __ldg(dout + t * H8 + c);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long i = i0 + u * stride;
      if (i < n) {
        const uint32_t dw[4] = {d[u].x, d[u].y, d[u].z, d[u].w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          o[j] = pack_bf16x2(w[u] * __uint_as_float(dw[j] << 16), w[u] * __uint_as_float(dw[j] & 0xffff0000u));
        xs[i] = x[u];
        dos[i] = d[u];
        dys[i] = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

// d_weights[reverse[p]] = sum over the row's partial dots (one per feature tile of dA).
__global__ void __launch_bounds__(256) bwd_dw_reduce_kernel(const int32_t* __restrict__ offsets,
                                                            const int32_t* __restrict__ poff,
                                                            const int32_t* __restrict__ reverse,
                                                            const float* __restrict__ dwp, int E, int NT,
                                                            float* __restrict__ d_weights) {
  extern __shared__ int s_off[];
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) s_off[e] = __ldg(offsets + e);
  __syncthreads();
  const int n = s_off[E];
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < n; p += gridDim.x * blockDim.x) {
    const int e = find_segment(s_off, E, p);
    const long pp = (long)__ldg(poff + e) + (p - s_off[e]);
    float s = 0.0f;
    for (int j = 0; j < NT; ++j) s += dwp[pp * NT + j];
    d_weights[__ldg(reverse + p)] = s;
  }
}

// Weight gradients of experts without rows are zero (no tile writes them).
__global__ void __launch_bounds__(256) bwd_zero_empty_kernel(const int32_t* __restrict__ counts, int E,
                                                             long per13, long per2, uint4* __restrict__ dw13,
                                                             uint4* __restrict__ dw2) {
  pdl_wait();
  pdl_trigger();
  for (int e = blockIdx.y; e < E; e += gridDim.y) {
    if (__ldg(counts + e) != 0) continue;
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < per13; i += (long)gridDim.x * blockDim.x)
      dw13[e * per13 + i] = z;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < per2; i += (long)gridDim.x * blockDim.x)
      dw2[e * per2 + i] = z;
  }
}

// ---- host -----------------------------------------------------------------------

template <int KIND>
int launch_bwd_pair(const CUtensorMap& a, const CUtensorMap& b, const BwdParams& p, long max_tiles,
                    cudaStream_t s, const char* name) {
  if (int rc = ensure_smem_limit(bwd_pair_kernel<KIND>, DSMEM, name)) return rc;
  const long pairs = num_sms() / 2;
  const int grid = 2 * (int)std::min(max_tiles, pairs);
  if (grid <= 0) return MOE_OK;
  ProfScope ps(name, s);
  const cudaError_t e = launch_pdl(bwd_pair_kernel<KIND>, grid, kind_threads<KIND>(), DSMEM, s, a, b, p);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", name, cudaGetErrorString(e));
  return check_launch(name);
}

int launch_fused_a(const CUtensorMap& x, const CUtensorMap& dO, const CUtensorMap& w13, const CUtensorMap& w2,
                   const BwdParams& p, long max_tiles, cudaStream_t s) {
  if (int rc = ensure_smem_limit(bwd_fused_a_kernel, DSMEM, "bwd_fc1_dact")) return rc;
  const int grid = 2 * (int)std::min(max_tiles, (long)(num_sms() / 2));
  if (grid <= 0) return MOE_OK;
  ProfScope ps("bwd_fc1_dact", s);
  const cudaError_t e = launch_pdl(bwd_fused_a_kernel, grid, kind_threads<FUSED_A>(), DSMEM, s, x, dO, w13, w2, p);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "bwd_fc1_dact: %s", cudaGetErrorString(e));
  return check_launch("bwd_fc1_dact");
}

template <typename... KArgs, typename... Args>
int launch_small(const char* name, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                 Args&&... args) {
  ProfScope ps(name, s);
  const cudaError_t e = launch_pdl(kernel, grid, block, smem, s, std::forward<Args>(args)...);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", name, cudaGetErrorString(e));
  return check_launch(name);
}

}  // namespace

long bwd_padded_rows(long S, int E) { return S + (long)kRowPad * E; }

// FC1 recompute and dA in one kernel for H up to this (measured: H = 2048 layers
// gain, where the separate dA epilogue's gu / act reads outweigh its MMAs; at
// H = 4096 the fused kernel's N = 128 G phase costs more than the round trip).
bool bwd_uses_fused(int H) { return H <= kFusedMaxH; }

int launch_ffn_backward(const FfnBwdArgs& a, cudaStream_t s) {
  const long S = (long)a.T * a.k;
  const int E = a.E, H = a.H, I = a.I;
  const long Pmax = bwd_padded_rows(S, E);
  int rc;
  if (a.d_weights) {
    const cudaError_t e = cudaMemsetAsync(a.d_weights, 0, (size_t)S * sizeof(float), s);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "d_weights memset: %s", cudaGetErrorString(e));
  }
  if ((rc = launch_small("bwd_pad", bwd_pad_kernel, 1, 1024, 0, s, a.counts, E, a.poff))) return rc;
  {
    const long units = Pmax * (H / 8);
    const int grid = (int)std::max(1L, std::min((long)num_sms() * 8, (units + 255) / 256));
    if ((rc = launch_small("bwd_gather", bwd_gather_kernel, grid, 256, (E + 1) * sizeof(int), s,
                           static_cast<const uint4*>(a.hidden), static_cast<const uint4*>(a.d_out), a.counts,
                           a.offsets, a.poff, a.sorted_ids, a.sorted_w, E, H / 8, pow2_shift(H / 8), Pmax,
                           static_cast<uint4*>(a.xs), static_cast<uint4*>(a.dos), static_cast<uint4*>(a.dys))))
      return rc;
  }
  const long row_tiles = (S + 2 * BM - 1) / (2 * BM) + E;
  CUtensorMap ta, tb;
  BwdParams p{};
  p.counts = a.counts;
  p.offsets = a.offsets;
  p.poff = a.poff;
  p.sorted_w = a.sorted_w;
  p.reverse = a.reverse;
  p.E = E;
  p.H = H;
  p.I = I;
  p.gu = a.gu;
  p.act = static_cast<__nv_bfloat16*>(a.act);
  p.dgu = static_cast<__nv_bfloat16*>(a.dgu);
  p.dwp = a.dwp;
  p.staging = a.staging;
  p.status = a.status;
  const bool fused = bwd_uses_fused(H);
  const int nt_a = fused ? (I + FA_FEAT - 1) / FA_FEAT : (I + BN - 1) / BN;

  if (fused) {   // FC1 recomputed and G = dO W2 in one kernel
    CUtensorMap tx, tdo, tw13, tw2;
    if ((rc = make_tmap(&tx, a.xs, (uint64_t)Pmax, (uint64_t)H, 128))) return rc;
    if ((rc = make_tmap(&tdo, a.dos, (uint64_t)Pmax, (uint64_t)H, 128))) return rc;
    if ((rc = make_tmap(&tw13, a.w13, (uint64_t)E * 2 * I, (uint64_t)H, 128))) return rc;
    if ((rc = make_tmap(&tw2, a.w2, (uint64_t)E * H, (uint64_t)I, 64))) return rc;
    p.K = H;
    p.NT = nt_a;
    if ((rc = launch_fused_a(tx, tdo, tw13, tw2, p, row_tiles * p.NT, s))) return rc;
  } else {
    // FC1 recomputed: gate / up pre-activations and the bf16 activation
    if ((rc = make_tmap(&ta, a.xs, (uint64_t)Pmax, (uint64_t)H, 128))) return rc;
    if ((rc = make_tmap(&tb, a.w13, (uint64_t)E * 2 * I, (uint64_t)H, 128))) return rc;
    p.K = H;
    p.NT = (I + 127) / 128;
    p.b_rows = 2 * I;
    if ((rc = launch_bwd_pair<RECOMPUTE>(ta, tb, p, row_tiles * p.NT, s, "bwd_fc1_recompute"))) return rc;

    // G = dO W2; dgu and the d w_p partials
    if ((rc = make_tmap(&ta, a.dos, (uint64_t)Pmax, (uint64_t)H, 128))) return rc;
    if ((rc = make_tmap(&tb, a.w2, (uint64_t)E * H, (uint64_t)I, 64))) return rc;
    p.K = H;
    p.NT = nt_a;
    p.b_rows = H;
    if ((rc = launch_bwd_pair<DGRAD_A>(ta, tb, p, row_tiles * p.NT, s, "bwd_dgrad_act"))) return rc;
  }

  // dx = dgu W13 into the slot rows, then the sum over k
  if ((rc = launch_zero_dropped(a.offsets, E, S, H, a.staging, 4, s))) return rc;
  if ((rc = make_tmap(&ta, a.dgu, (uint64_t)Pmax, (uint64_t)2 * I, 128))) return rc;
  if ((rc = make_tmap(&tb, a.w13, (uint64_t)E * 2 * I, (uint64_t)H, 64))) return rc;
  p.K = 2 * I;
  p.NT = (H + BN - 1) / BN;
  p.b_rows = 2 * I;
  if ((rc = launch_bwd_pair<DGRAD_X>(ta, tb, p, row_tiles * p.NT, s, "bwd_dgrad_x"))) return rc;
  if ((rc = launch_combine(a.staging, 0, a.T, a.k, H, MOE_BF16, a.d_hidden, s))) return rc;

  // dW2[e] = dys^T act, dW13[e] = dgu^T xs over the expert's padded rows
  if ((rc = make_tmap(&ta, a.dys, (uint64_t)Pmax, (uint64_t)H, 64))) return rc;
  if ((rc = make_tmap(&tb, a.act, (uint64_t)Pmax, (uint64_t)I, 64))) return rc;
  p.M_dim = H;
  p.N_dim = I;
  p.MT = (H + BN - 1) / BN;
  p.NT = (I + BN - 1) / BN;
  p.dw = static_cast<__nv_bfloat16*>(a.d_w2);
  p.dw_sector = (reinterpret_cast<uintptr_t>(p.dw) & 31) == 0;
  if ((rc = launch_bwd_pair<WGRAD>(ta, tb, p, (long)E * p.MT * p.NT, s, "bwd_wgrad_w2"))) return rc;
  if ((rc = make_tmap(&ta, a.dgu, (uint64_t)Pmax, (uint64_t)2 * I, 64))) return rc;
  if ((rc = make_tmap(&tb, a.xs, (uint64_t)Pmax, (uint64_t)H, 64))) return rc;
  p.M_dim = 2 * I;
  p.N_dim = H;
  p.MT = (2 * I + BN - 1) / BN;
  p.NT = (H + BN - 1) / BN;
  p.dw = static_cast<__nv_bfloat16*>(a.d_w13);
  p.dw_sector = (reinterpret_cast<uintptr_t>(p.dw) & 31) == 0;
  if ((rc = launch_bwd_pair<WGRAD>(ta, tb, p, (long)E * p.MT * p.NT, s, "bwd_wgrad_w13"))) return rc;
  if ((rc = launch_small("bwd_zero_empty", bwd_zero_empty_kernel, dim3(64, (unsigned)std::min(E, 1024)), 256, 0,
                         s, a.counts, E, (long)2 * I * H / 8, (long)H * I / 8, static_cast<uint4*>(a.d_w13),
                         static_cast<uint4*>(a.d_w2))))
    return rc;
  if (a.d_weights) {
    const int grid = (int)std::max(1L, std::min((long)num_sms() * 4, (S + 255) / 256));
    if ((rc = launch_small("bwd_dw_reduce", bwd_dw_reduce_kernel, grid, 256, (E + 1) * sizeof(int), s, a.offsets,
                           a.poff, a.reverse, a.dwp, E, 2 * nt_a, a.d_weights)))
      return rc;
  }
  return MOE_OK;
}

}  // namespace moe
