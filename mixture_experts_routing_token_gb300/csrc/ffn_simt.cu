// Grouped expert FFN on the CUDA cores (float32, and bf16 shapes the tensor
// path does not take). Same semantics as the tensor-core path:
// project_6 moe_expert_gemm.cpp moe_prefill_experts (FC1, silu_and_mul, FC2,
// weight), mlc-llm moe_misc.py scatter_output (row p -> slot reverse[p]).
//
// Each CTA computes a 32 x 32 output tile of one expert; the tile list (32
// sorted rows of one expert per x-block) is rebuilt in every CTA from the
// expert counts, so no host synchronisation is needed. Accumulation is fp32.
#include "common.cuh"

namespace moe {
namespace {

constexpr int TM = 32, TN = 32, TK = 32;

// tstart[e] = number of TM-row tiles of experts < e; tstart[E] = total.
__device__ void build_row_tiles(const int32_t* __restrict__ counts, int E, int* tstart) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int run = 0;
    for (int e = e0; e < e1; ++e) run += (__ldg(counts + e) + TM - 1) / TM;
    int incl = run;
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int acc = incl - run;
    for (int e = e0; e < e1; ++e) {
      tstart[e] = acc;
      acc += (__ldg(counts + e) + TM - 1) / TM;
    }
    if (lane == 31) tstart[E] = incl;
  }
}

__device__ __forceinline__ int find_expert(const int* tstart, int E, int t) {
  int lo = 0, hi = E;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tstart[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// MODE 0: act[p, n] = silu(x_t . w13[e, n]) * (x_t . w13[e, I + n])
// MODE 1: staging[reverse[p], n] = sorted_w[p] * (act[p] . w2[e, n])
template <int MODE, class T>
__global__ void __launch_bounds__(256) ffn_simt_kernel(
    const T* __restrict__ xsrc, const T* __restrict__ w, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ ids,
    const float* __restrict__ sorted_w, const int32_t* __restrict__ reverse, int E, int K, int N,
    T* __restrict__ act_out, float* __restrict__ staging) {
  __shared__ int tstart[MOE_MAX_EXPERTS + 1];
  __shared__ float Xs[TM][TK + 1], W0[TN][TK + 1], W1[TN][TK + 1];
  build_row_tiles(counts, E, tstart);
  __syncthreads();
  const int mt = blockIdx.x;
  if (mt >= tstart[E]) return;
  const int e = find_expert(tstart, E, mt);
  const int cnt = __ldg(counts + e);
  const int row0 = (mt - tstart[e]) * TM;
  const long p0 = (long)__ldg(offsets + e) + row0;
  const int n0 = blockIdx.y * TN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  // weight rows of this tile: FC1 gate rows n, up rows I + n of w13[e] ([2I, K]); FC2 rows n of w2[e]
  const long wrows = MODE == 0 ? 2L * N : (long)N;
  const T* we = w + (long)e * wrows * K;

  float a0[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, a1[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  for (int k0 = 0; k0 < K; k0 += TK) {
    for (int i = threadIdx.x; i < TM * TK; i += 256) {
      const int r = i / TK, c = i % TK;
      const bool kin = k0 + c < K;
      float xv = 0.f;
      if (row0 + r < cnt && kin) {
        const long src = MODE == 0 ? (long)__ldg(ids + p0 + r) : p0 + r;
        xv = to_float(xsrc[src * K + k0 + c]);
      }
      Xs[r][c] = xv;
      const bool nin = n0 + r < N && kin;
      W0[r][c] = nin ? to_float(we[(long)(n0 + r) * K + k0 + c]) : 0.f;
      if (MODE == 0) W1[r][c] = nin ? to_float(we[(long)(N + n0 + r) * K + k0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < TK; ++kk) {
      const float x0 = Xs[ty * 2][kk], x1 = Xs[ty * 2 + 1][kk];
      const float g0 = W0[tx * 2][kk], g1 = W0[tx * 2 + 1][kk];
      a0[0][0] = fmaf(x0, g0, a0[0][0]);
      a0[0][1] = fmaf(x0, g1, a0[0][1]);
      a0[1][0] = fmaf(x1, g0, a0[1][0]);
      a0[1][1] = fmaf(x1, g1, a0[1][1]);
      if (MODE == 0) {
        const float u0 = W1[tx * 2][kk], u1 = W1[tx * 2 + 1][kk];
        a1[0][0] = fmaf(x0, u0, a1[0][0]);
        a1[0][1] = fmaf(x0, u1, a1[0][1]);
        a1[1][0] = fmaf(x1, u0, a1[1][0]);
        a1[1][1] = fmaf(x1, u1, a1[1][1]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 2; ++a) {
    const int r = row0 + ty * 2 + a;
    if (r >= cnt) continue;
    const long p = p0 + ty * 2 + a;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int n = n0 + tx * 2 + b;
      if (n >= N) continue;
      if (MODE == 0) {
        act_out[p * N + n] = from_float<T>(silu(a0[a][b]) * a1[a][b]);
      } else {
        staging[(long)__ldg(reverse + p) * N + n] = a0[a][b] * __ldg(sorted_w + p);
      }
    }
  }
}

template <class T>
int launch_simt_t(const FfnArgs& a, cudaStream_t s) {
  const long S = (long)a.T * a.k;
  const unsigned gx = (unsigned)((S + TM - 1) / TM + a.E);
  {
    ProfScope ps("ffn_fc1_simt", s);
    dim3 grid(gx, (a.I + TN - 1) / TN);
    ffn_simt_kernel<0, T><<<grid, 256, 0, s>>>(
        static_cast<const T*>(a.hidden), static_cast<const T*>(a.w13), a.counts, a.offsets,
        a.sorted_ids, a.sorted_w, a.reverse, a.E, a.H, a.I, static_cast<T*>(a.act), nullptr);
    int rc = check_launch("ffn_fc1_simt");
    if (rc) return rc;
  }
  {
    ProfScope ps("ffn_fc2_simt", s);
    dim3 grid(gx, (a.H + TN - 1) / TN);
    ffn_simt_kernel<1, T><<<grid, 256, 0, s>>>(
        static_cast<const T*>(a.act), static_cast<const T*>(a.w2), a.counts, a.offsets,
        a.sorted_ids, a.sorted_w, a.reverse, a.E, a.I, a.H, nullptr, static_cast<float*>(a.staging));
    int rc = check_launch("ffn_fc2_simt");
    if (rc) return rc;
  }
  return launch_combine(a.staging, 0, a.T, a.k, a.H, a.dtype, a.out, s);
}

}  // namespace

int launch_ffn_simt(const FfnArgs& a, cudaStream_t s) {
  if ((long)a.T * a.k == 0) return MOE_OK;
  return a.dtype == MOE_F32 ? launch_simt_t<float>(a, s) : launch_simt_t<__nv_bfloat16>(a, s);
}

}  // namespace moe
