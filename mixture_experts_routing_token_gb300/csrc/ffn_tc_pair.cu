// Grouped expert FFN on SM pairs: tcgen05.mma.cta_group::2, M = 256 (128 rows
// per SM) x N = 256 x K = 16, accumulators in both SMs' TMEM.
//
// project_6 moe_expert_gemm.cpp moe_prefill_experts: FC1, silu_and_mul,
// FC2, routing weight; mlc-llm moe_misc.py scatter_output. Tiles are 256
// sorted rows of one expert (the tile list is built in every CTA from the
// align step's counts). Each SM of a 2-CTA cluster loads its own 128
// rows of A and ONE HALF of the 256 B rows:
//   FC1: CTA 0 the 128 gate rows n0.., CTA 1 the 128 matching up rows I+n0..;
//   FC2: CTA 0 rows n0..n0+127 of w2[e], CTA 1 rows n0+128..n0+255.
// The pair's MMA then leaves, in each SM's TMEM, its 128 rows x all 256
// columns (FC1: gate columns 0..127, up columns 128..255), so each SM's
// epilogue sees whole rows. Per SM and k-step this moves 32 KB instead of the
// 48 KB a one-SM 128 x 256 tile needs for the same tensor work, which is what lets a 6-stage ring hide the
// L2 -> shared-memory latency.
//
// Swapped remainder tiles (FC2). An expert's last tile of at most kSwapMax
// rows would waste most of a 256-row M tile, so FC2 runs it with the operands
// swapped: A = 256 rows of w2[e] (128 per SM: output features), B = the
// leftover act rows (N = 64 or 128, half of them per SM), D = features x
// tokens in TMEM; the epilogue writes staging columns. Measured 2-16% faster
// FC2 launches on ragged counts. FC1 keeps plain tiles: its swapped form
// needs two passes over K (gate, then up rows), so it issues as many k-steps
// per feature as the plain tile, and those k-steps, bounded by the ring's
// latency rather than by the MMA, measured no faster.
//
// Synchronisation:
//   full[s]   leader CTA only; the leader's producer posts the pair's bytes
//             (2 x 32 KB) and both CTAs' TMA loads complete on it
//             (.cta_group::2 form, barrier addressed in the leader's window);
//   empty[s]  in both CTAs; the leader's MMA commit multicasts to both;
//   tfull[b]  in both CTAs; multicast commit after a tile's last k-step;
//   tempty[b] leader only; one arrival per epilogue warp of both CTAs (8).
// Launched with a programmatic dependency on the previous kernel: the prologue
// (barriers, TMEM, tile list from the counts of the align step, which is
// complete by then) overlaps that kernel's tail; everything after waits for it.
// Every mbarrier wait is bounded (2 s of global time, then the abort path
// below); a cluster barrier brackets
// the kernel so neither CTA leaves while the other may still touch its
// shared memory.
#include "common.cuh"
#include "pair_ptx.cuh"

namespace moe {
namespace {

using namespace pair;

constexpr int PBM = 128;                // rows per CTA (256 per pair)
constexpr int PBK = 64;
constexpr int PBN = 256;                // MMA N
constexpr int PSTAGES = 6;
constexpr int PA_BYTES = PBM * PBK * 2;       // 16 KB
constexpr int PB_BYTES = (PBN / 2) * PBK * 2; // 16 KB: this CTA's half of B
constexpr int PSTAGE = PA_BYTES + PB_BYTES;
constexpr int PDSMEM = PSTAGES * PSTAGE + 1024;
constexpr int PTHREADS = 192;
constexpr uint32_t PTMEM_COLS = 2 * PBN;
constexpr uint64_t PWAIT_NS = 2000000000ull;   // the drain of issued MMAs
constexpr uint32_t PIDESC = ptx::idesc_bf16_f32(2 * PBM, PBN);
constexpr int kSwapMax = 128;           // FC2 remainders up to this many rows take a swapped tile
constexpr int kSwapBox = 32;            // token rows per TMA box of a swapped tile's B operand

enum { PAIR_FC1 = 0, PAIR_FC2 = 1 };

struct PairParams {
  const int32_t* counts;
  const int32_t* offsets;
  const float* sorted_w;
  const int32_t* reverse;
  int E;
  int K;          // H (FC1) or I (FC2)
  int N_out;      // I (FC1) or H (FC2)
  int NT;         // N tiles per expert
  int NTs;        // swapped tiles per expert remainder (256 output features each; 0: none)
  int b_rows;     // 2I (FC1) or H (FC2)
  void* out;
  int32_t* status;
  uint64_t wait_ns;   // limit of the waits on the other roles (moe_set_wait_limit_ns)
};

struct PTile {
  int e, m_tile, n_tile;
  int swap_n;     // 0: a 256-row tile; 64 or 128: a swapped tile with this many token columns
};

// Token columns of the swapped remainder tile of an expert with cnt rows, 0 when
// it has none (no swapped tiles at all when NTs == 0).
__host__ __device__ __forceinline__ int swap_cols(int cnt, int NTs) {
  const int rem = cnt % (2 * PBM);
  return (NTs == 0 || rem == 0 || rem > kSwapMax) ? 0 : (rem <= 64 ? 64 : 128);
}
// 256-row tiles of an expert with cnt rows (a remainder without a swapped tile gets one too).
__host__ __device__ __forceinline__ int full_mtiles(int cnt, int NTs) {
  return cnt / (2 * PBM) + (cnt % (2 * PBM) != 0 && swap_cols(cnt, NTs) == 0 ? 1 : 0);
}
__host__ __device__ __forceinline__ int expert_tiles(int cnt, int NT, int NTs) {
  return full_mtiles(cnt, NTs) * NT + (swap_cols(cnt, NTs) ? NTs : 0);
}

// Tile t of the list: the expert's 256-row tiles, then its swapped tiles. Pairs
// take consecutive tiles in the same round, so the order within an expert
// decides which operand they share in L2: with fewer M tiles than N tiles the
// expert's A rows (mt tiles) stay in L2 while N walks the weights once
// (N-tile-major); with more M tiles than N tiles its weight tiles (NT of them,
// at most a few tens of MB) stay in L2 while M walks the rows once
// (M-tile-major). A and B tiles have the same size (256 rows x K), so the
// smaller count is the smaller operand. (N-tile-major for an expert with 128
// M tiles and 12 N tiles streamed its 268 MB of rows past L2 once per N tile.)
__device__ __forceinline__ PTile ptile(int t, const int* tile_start, const int32_t* counts, int E, int NT,
                                       int NTs) {
  int lo = 0, hi = E;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int local = t - tile_start[lo];
  const int cnt = __ldg(counts + lo);
  const int mt = full_mtiles(cnt, NTs);
  PTile d;
  d.e = lo;
  if (local < mt * NT) {
    if (mt > NT) {
      d.m_tile = local / NT;
      d.n_tile = local - d.m_tile * NT;
    } else {
      d.n_tile = local / mt;
      d.m_tile = local - d.n_tile * mt;
    }
    d.swap_n = 0;
  } else {
    d.n_tile = local - mt * NT;
    d.m_tile = mt;
    d.swap_n = swap_cols(cnt, NTs);
  }
  return d;
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PTHREADS, 1)
    ffn_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmS, const PairParams P) {
  __shared__ __align__(8) uint64_t full_bar[PSTAGES], empty_bar[PSTAGES];
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
  auto sA = [&](int s) { return dsmem + (uint32_t)(s * PSTAGE); };
  auto sB = [&](int s) { return dsmem + (uint32_t)(s * PSTAGE + PA_BYTES); };
  volatile int* abort_p = &abort_flag;

  if (tid == 0) {
    for (int s = 0; s < PSTAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&tfull_bar[b]), 1);
      ptx::mbar_init(ptx::smem_u32(&tempty_bar[b]), 8);
    }
    ptx::mbar_init(ptx::smem_u32(&drain_bar), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    ptx::prefetch_tmap(&tmS);
  }
  if (warp == 1) {   // both CTAs of the pair allocate together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     ptx::smem_u32(&tmem_slot)),
                 "r"(PTMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  if (warp == 2) {   // tile_start[e] = sum over e' < e of the tiles of expert e'
    const int per = (P.E + 31) / 32;
    const int e0 = min(P.E, lane * per), e1 = min(P.E, e0 + per);
    int run = 0;
    for (int e = e0; e < e1; ++e) run += expert_tiles(__ldg(P.counts + e), P.NT, P.NTs);
    int incl = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int acc = incl - run;
    for (int e = e0; e < e1; ++e) {
      tile_start[e] = acc;
      acc += expert_tiles(__ldg(P.counts + e), P.NT, P.NTs);
    }
    if (lane == 31) tile_start[P.E] = incl;
  }
  ptx::tc_fence_before();
  __syncthreads();
  cluster_sync();      // barriers of both CTAs initialised before any cross-CTA signal
  ptx::tc_fence_after();
  pdl_wait();          // the previous kernel's output (x_sorted / act) is read from here on
  pdl_trigger();
  const uint32_t tmem_base = tmem_slot;
  const int total = tile_start[P.E];
  const int KB = P.K / PBK;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      for (int t = cluster_id; t < total; t += nclusters) {
        const PTile ti = ptile(t, tile_start, P.counts, P.E, P.NT, P.NTs);
        if (MODE == PAIR_FC2 && ti.swap_n) {
          // A: 128 rows of w2[e] per SM; B: this SM's half of the act rows, in boxes of kSwapBox rows
          const int half = ti.swap_n / 2;
          const int tok_row = __ldg(P.offsets + ti.e) + ti.m_tile * (2 * PBM) + (int)rank * half;
          const int w_row = ti.e * P.b_rows + ti.n_tile * (2 * PBM) + (int)rank * PBM;
          for (int kb = 0; kb < KB; ++kb) {
            if (!ptx::mbar_wait(ptx::smem_u32(&empty_bar[stage]), ph ^ 1u, abort_p, P.wait_ns)) goto producer_done;
            const uint32_t fb_local = ptx::smem_u32(&full_bar[stage]);
            if (leader) ptx::mbar_arrive_expect_tx(fb_local, 2 * (PA_BYTES + half * PBK * 2));
            const uint32_t fb = map_to_rank(fb_local, 0);
            tma_load_2d_pair(sA(stage), &tmB, kb * PBK, w_row, fb);
            for (int b = 0; b < half; b += kSwapBox)
              tma_load_2d_pair(sB(stage) + (uint32_t)(b * PBK * 2), &tmS, kb * PBK, tok_row + b, fb);
            if (++stage == PSTAGES) { stage = 0; ph ^= 1u; }
          }
          continue;
        }
        const int a_row = __ldg(P.offsets + ti.e) + ti.m_tile * (2 * PBM) + (int)rank * PBM;
        int b_row;
        if (MODE == PAIR_FC1) b_row = ti.e * P.b_rows + ti.n_tile * 128 + (leader ? 0 : P.N_out);
        else b_row = ti.e * P.b_rows + ti.n_tile * PBN + (int)rank * 128;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&empty_bar[stage]), ph ^ 1u, abort_p, P.wait_ns)) goto producer_done;
          const uint32_t fb_local = ptx::smem_u32(&full_bar[stage]);
          if (leader) ptx::mbar_arrive_expect_tx(fb_local, 2 * PSTAGE);
          const uint32_t fb = map_to_rank(fb_local, 0);
          tma_load_2d_pair(sA(stage), &tmA, kb * PBK, a_row, fb);
          tma_load_2d_pair(sB(stage), &tmB, kb * PBK, b_row, fb);
          if (++stage == PSTAGES) { stage = 0; ph ^= 1u; }
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
        const PTile ti = ptile(t, tile_start, P.counts, P.E, P.NT, P.NTs);
        const uint32_t idesc = ti.swap_n ? ptx::idesc_bf16_f32(2 * PBM, ti.swap_n) : PIDESC;
        if (!ptx::mbar_wait(ptx::smem_u32(&tempty_bar[acc]), aph ^ 1u, abort_p, P.wait_ns)) break;
        ptx::tc_fence_after();
        bool ok = true;
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * PBN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_u32(&full_bar[stage]), ph, abort_p, P.wait_ns)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = sA(stage), b0 = sB(stage);
#pragma unroll
          for (int kk = 0; kk < PBK / 16; ++kk)
            mma_pair(d_tmem, ptx::sdesc_k128(a0 + kk * 32), ptx::sdesc_k128(b0 + kk * 32), idesc,
                     (kb | kk) != 0);
          commit_pair(ptx::smem_u32(&empty_bar[stage]), 0x3);
          if (++stage == PSTAGES) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
        commit_pair(ptx::smem_u32(&tfull_bar[acc]), 0x3);
        if (++acc == 2) { acc = 0; aph ^= 1u; }
      }
      commit_pair(ptx::smem_u32(&drain_bar), 0x1);
      int dummy = 0;
      ptx::mbar_wait(ptx::smem_u32(&drain_bar), 0, &dummy, PWAIT_NS);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
    for (int t = cluster_id; t < total; t += nclusters) {
      // the tile's row data first: these loads do not wait for the accumulator
      const PTile ti = ptile(t, tile_start, P.counts, P.E, P.NT, P.NTs);
      const int cnt = __ldg(P.counts + ti.e);
      const long pe = (long)__ldg(P.offsets + ti.e);
      const int r = ti.m_tile * (2 * PBM) + (int)rank * PBM + row;
      const bool valid = r < cnt;
      float wt = 0.0f;
      long dst_row = 0;
      if (MODE == PAIR_FC2 && !ti.swap_n && valid) {
        wt = __ldg(P.sorted_w + pe + r);
        dst_row = (long)__ldg(P.reverse + pe + r);
      }
      if (!ptx::mbar_wait(ptx::smem_u32(&tfull_bar[acc]), aph, abort_p, P.wait_ns)) break;
      ptx::tc_fence_after();
      if (MODE == PAIR_FC2 && ti.swap_n) {
        // lane = output feature f of this SM's 128; TMEM column j = act row r0 + j
        const int r0 = ti.m_tile * (2 * PBM);
        const long p0 = pe + r0;
        const int f = ti.n_tile * (2 * PBM) + (int)rank * PBM + row;
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * PBN);
        const int H = P.N_out;
        __nv_bfloat16* staging = static_cast<__nv_bfloat16*>(P.out);
#pragma unroll 1
        for (int c = 0; c < ti.swap_n / 32; ++c) {
          uint32_t y[32];
          ptx::tmem_ld32(taddr + c * 32, y);
          ptx::tmem_ld_wait();
          const bool vl = r0 + c * 32 + lane < cnt;   // lane l fetches row c*32 + l's weight and slot
          const float wl = vl ? __ldg(P.sorted_w + p0 + c * 32 + lane) : 0.0f;
          const int sl = vl ? __ldg(P.reverse + p0 + c * 32 + lane) : 0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float wj = __shfl_sync(0xffffffffu, wl, j);
            const int sj = __shfl_sync(0xffffffffu, sl, j);
            if (r0 + c * 32 + j < cnt && f < H) staging[(long)sj * H + f] = __float2bfloat16_rn(__uint_as_float(y[j]) * wj);
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_remote(map_to_rank(ptx::smem_u32(&tempty_bar[acc]), 0));
        if (++acc == 2) { acc = 0; aph ^= 1u; }
        continue;
      }
      const long p = pe + r;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * PBN);
      if (MODE == PAIR_FC1) {
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
              pk[i] = pack2(a0, a1);
            }
            uint32_t lo8[8], hi8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) { lo8[i] = pk[i]; hi8[i] = pk[8 + i]; }
            st_v8(act + p * I + col0, lo8);        // two whole 32-byte sectors
            st_v8(act + p * I + col0 + 16, hi8);
          }
        }
      } else {
        const int H = P.N_out;
        __nv_bfloat16* staging = static_cast<__nv_bfloat16*>(P.out);
#pragma unroll 1
        for (int c = 0; c < PBN / 32; c += 2) {   // two 32-column chunks per TMEM wait
          uint32_t y[2][32];
          ptx::tmem_ld32(taddr + c * 32, y[0]);
          ptx::tmem_ld32(taddr + c * 32 + 32, y[1]);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col0 = ti.n_tile * PBN + (c + h) * 32;
            if (valid && col0 < H) {   // 32 bf16 = two whole 32-byte sectors
              uint32_t lo8[8], hi8[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                lo8[i] = pack2(__uint_as_float(y[h][2 * i]) * wt, __uint_as_float(y[h][2 * i + 1]) * wt);
                hi8[i] = pack2(__uint_as_float(y[h][16 + 2 * i]) * wt, __uint_as_float(y[h][17 + 2 * i]) * wt);
              }
              st_v8(staging + dst_row * H + col0, lo8);
              st_v8(staging + dst_row * H + col0 + 16, hi8);
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

  // Teardown. After a timeout, give copies that may still be in flight time
  // to land before the shared memory is released.
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
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(PTMEM_COLS)
                 : "memory");
  }
  if (tid == 0 && abort_flag && P.status) atomicOr(P.status, MOE_STATUS_TIMEOUT);
}

template <int MODE>
int launch_pair(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sw, const PairParams& p, long S,
                cudaStream_t s, const char* name) {
  if (int rc = ensure_smem_limit(ffn_tc_pair_kernel<MODE>, PDSMEM, name)) return rc;
  const long max_tiles = ((S + 2 * PBM - 1) / (2 * PBM) + p.E) * (long)p.NT;
  const long pairs = num_sms() / 2;
  const int grid = 2 * (int)(max_tiles < pairs ? max_tiles : pairs);
  if (grid <= 0) return MOE_OK;
  ProfScope ps(name, s);
  const cudaError_t e = launch_pdl(ffn_tc_pair_kernel<MODE>, grid, PTHREADS, PDSMEM, s, a, b, sw, p);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", name, cudaGetErrorString(e));
  return check_launch(name);
}

}  // namespace

int launch_ffn_pair_gemms(const FfnArgs& a, const CUtensorMap& tA1, const CUtensorMap& tB1,
                          const CUtensorMap& tA2, const CUtensorMap& tB2, const CUtensorMap& tS2,
                          cudaStream_t s) {
  const long S = (long)a.T * a.k;
  PairParams p1{a.counts, a.offsets, a.sorted_w, a.reverse, a.E, a.H, a.I, (a.I + 127) / 128, 0,
                2 * a.I, a.act, a.status, wait_limit_ns()};
  int rc = launch_pair<PAIR_FC1>(tA1, tB1, tA1, p1, S, s, "ffn_fc1_tc");   // (no swapped tiles: tmS unused)
  if (rc) return rc;
  PairParams p2{a.counts, a.offsets, a.sorted_w, a.reverse, a.E, a.I, a.H, (a.H + PBN - 1) / PBN,
                (a.H + 2 * PBM - 1) / (2 * PBM), a.H, a.staging, a.status, wait_limit_ns()};
  return launch_pair<PAIR_FC2>(tA2, tB2, tS2, p2, S, s, "ffn_fc2_tc");
}

}  // namespace moe
