// Routing kernels: gating softmax-top-k, indices -> multihot, multihot -> indices.
//
// gating: mlc-llm moe_misc.py, gating_topk / gating_softmax_topk.
// multihot: Megatron-LM fused_indices_converter.py, _indices_to_multihot_kernel
//           and _multihot_to_indices_kernel.
//
// Gating dispatch by E: up to 8 experts one thread per token (row in
// registers); up to 128 one thread per token over a block's rows staged in
// shared memory (by TMA when k <= 8 and a row is a whole number of 128-byte
// boxes, else by cp.async); wider rows a group of L lanes per token, lane g
// holding the V = 64 contiguous experts g*V .. g*V + V - 1 (vector loads of its
// run). Group-limited top-k: one lane per expert group (groups of 32 with
// coalesced row reads), or a thread / warp per token for larger groups.
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "gating_device.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

using gate::better;
using gate::group_mask;
using gate::kNone;

constexpr int kBlock = 256;
template <int L, int V, typename In>
__global__ void __launch_bounds__(kBlock) gating_kernel(const In* __restrict__ logits, int T,
                                                        int E, int k, int norm,
                                                        float* __restrict__ w_out,
                                                        int32_t* __restrict__ idx_out) {
  const long t = (long)blockIdx.x * (kBlock / L) + threadIdx.x / L;
  if (t >= T) return;   // whole groups leave together
  gate::gate_one_token<L, V, In>(logits, t, E, k, norm, w_out, idx_out);
}

// Gating for E <= 8, K = k: a thread per token over a grid-stride loop, the next
// token's row loaded before the current one is ranked (one row in flight while
// the thread computes). FULL: E == 8, so no expert is masked (the selection is
// bound by the integer / compare pipe, and the masks cost a sixth of it).
template <int K, typename In, bool FULL>
__global__ void __launch_bounds__(kBlock, 6) gating_rows8_kernel(const In* __restrict__ logits, int T, int E_rt,
                                                                 int norm, float* __restrict__ w_out,
                                                                 int32_t* __restrict__ idx_out) {
  const int E = FULL ? 8 : E_rt;
  const long stride = (long)gridDim.x * kBlock;
  long t = (long)blockIdx.x * kBlock + threadIdx.x;
  if (t >= T) return;
  float v[8];
  gate::load_row_part<8>(logits + t * (long)E, 0, E, v);
  for (;;) {
    const long tn = t + stride;
    float nv[8];
    if (tn < T) gate::load_row_part<8>(logits + tn * (long)E, 0, E, nv);
    gate::gate_row_regs<8, K>(v, E, norm, t, w_out, idx_out);
    if (tn >= T) break;
    t = tn;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = nv[i];
  }
}

// Gating for E <= 128, one thread per token: each CTA stages its 128 rows in
// shared memory and runs gate::topk_staged_row on them (gating_device.cuh).
constexpr int kSmemGateThreads = gate::kStageRows;

// Staged as 16-bit patterns: bf16 logits with at least 64 experts.
template <int EP, typename In>
using StageT = typename std::conditional<!std::is_same<In, float>::value && EP >= 64, uint16_t, float>::type;
// Group maxima in registers (gate::topk_staged_row): float32 rows of 64-128 experts
// (measured faster there; the 16-bit stages keep them in shared memory).
template <int EP, typename In>
constexpr bool kRegMax = std::is_same<StageT<EP, In>, float>::value && EP >= 64;

// The parked results of the block's rows (gate::topk_staged_row<TO_COL>: weights
// as words 0..k-1, indices as words 8..8+k-1 of each row's first chunks) written
// out contiguously.
template <typename St, typename Lay = gate::StagePadded>
__device__ __forceinline__ void copy_out_parked(const St* col, long t0, int nt, int k, float* __restrict__ w_out,
                                                int32_t* __restrict__ idx_out, int tid, int nthr) {
  if (k == 8 || k == 4) {   // whole 16-byte chunks
    const uint4* c4 = reinterpret_cast<const uint4*>(col);
    const int hs = k >> 3;   // chunks per row's weights, minus one
    for (int f = tid; f < (nt << hs); f += nthr) {
      const int r = f >> hs, h = f & hs;
      reinterpret_cast<uint4*>(w_out + (t0 + r) * k)[h] = c4[Lay::chunk(h, r)];
      reinterpret_cast<uint4*>(idx_out + (t0 + r) * k)[h] = c4[Lay::chunk(2 + h, r)];
    }
    return;
  }
  auto get32 = [&](int slot, int r) -> uint32_t {   // word `slot` of the row's parking chunks
    return reinterpret_cast<const uint32_t*>(col)[Lay::chunk(slot >> 2, r) * 4 + (slot & 3)];
  };
  const int n = nt * k;
  const int kshift = (k & (k - 1)) == 0 ? __ffs(k) - 1 : -1;   // row of output f: f >> kshift, or f / k
  for (int f = tid; f < n; f += nthr) {
    const int r = kshift >= 0 ? f >> kshift : (int)((uint32_t)f / (uint32_t)k), j = f - r * k;
    w_out[t0 * k + f] = __uint_as_float(get32(j, r));
    idx_out[t0 * k + f] = (int32_t)get32(gate::kRegSel + j, r);
  }
}

template <int EP, typename In, int U = 8>
__global__ void __launch_bounds__(kSmemGateThreads) gating_smem_kernel(
    const In* __restrict__ logits, int T, int E, int k, int norm, float* __restrict__ w_out,
    int32_t* __restrict__ idx_out) {
  using St = StageT<EP, In>;
  constexpr bool RM = kRegMax<EP, In>;
  extern __shared__ __align__(16) uint8_t stage_raw[];   // gate::stage_bytes<EP, St, RM>()
  St* col = reinterpret_cast<St*>(stage_raw);
  const int tid = threadIdx.x;
  const long t0 = (long)blockIdx.x * kSmemGateThreads;
  const int nt = (int)min((long)kSmemGateThreads, (long)T - t0);
  gate::stage_rows<EP, In, U, St>(logits, t0, nt, E, col, tid, kSmemGateThreads);
  __syncthreads();
  if (k > gate::kRegSel) {
    if (tid < nt) gate::topk_staged_row<EP, false, St, RM>(col, tid, t0 + tid, E, k, norm, w_out, idx_out);
    return;
  }
  // Each thread touches only its own row's column, so it parks its k weights and
  // indices there; after the barrier the block writes its rows' outputs out
  // contiguously.
  if (tid < nt) gate::topk_staged_row<EP, true, St, RM>(col, tid, tid, E, k, norm, nullptr, nullptr);
  __syncthreads();
  copy_out_parked(col, t0, nt, k, w_out, idx_out, tid, kSmemGateThreads);
}

// The same with the block's rows brought in by TMA (k <= kRegSel, rows a whole
// number of 128-byte boxes): one thread issues E * sizeof(In) / 128 tensor-map
// copies of 128 rows x 128 bytes each (128-byte swizzle, gate::StageSwz128) on
// one mbarrier, so the 128 threads spend no instructions on staging (measured
// without the selection, the cp.async staging alone ran at 0.58-0.64 of the
// copy peak), and every 16-byte read of the selection is conflict-free. The wait
// is bounded (kGateWaitNs); a block whose rows never arrive writes nothing.
constexpr uint64_t kGateWaitNs = 2000000000ull;

template <int EP, typename In>
__global__ void __launch_bounds__(kSmemGateThreads) gating_tma_kernel(
    const __grid_constant__ CUtensorMap tm, int T, int E, int k, int norm, float* __restrict__ w_out,
    int32_t* __restrict__ idx_out) {
  using St = StageT<EP, In>;
  using Lay = gate::StageSwz128;
  constexpr bool RM = kRegMax<EP, In>;
  extern __shared__ __align__(16) uint8_t stage_raw[];   // gate::stage_bytes<EP, St, RM, Lay>() + 1024
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  St* col = reinterpret_cast<St*>(stage_raw + ((1024u - (ptx::smem_u32(stage_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x;
  const long t0 = (long)blockIdx.x * kSmemGateThreads;
  const int nt = (int)min((long)kSmemGateThreads, (long)T - t0);
  const uint32_t b = ptx::smem_u32(&bar);
  if (tid == 0) {
    abort_flag = 0;
    ptx::mbar_init(b, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const int nbox = E * (int)sizeof(In) / 128;
  if (tid == 0) {
    ptx::mbar_arrive_expect_tx(b, (uint32_t)nbox * kSmemGateThreads * 128u);
    for (int i = 0; i < nbox; ++i)
      ptx::tma_load_2d(ptx::smem_u32(col) + (uint32_t)i * kSmemGateThreads * 128u, &tm, i * (128 / (int)sizeof(In)),
                       (int)t0, b);
  }
  ptx::mbar_wait(b, 0, &abort_flag, kGateWaitNs);
  for (int e = E; e < EP; ++e) gate::st_neg_inf(col + gate::sofs<St, Lay>(e, tid));   // experts past E: -inf
  __syncthreads();
  if (abort_flag) return;
  if (tid < nt) gate::topk_staged_row<EP, true, St, RM, Lay>(col, tid, tid, E, k, norm, nullptr, nullptr);
  __syncthreads();
  copy_out_parked<St, Lay>(col, t0, nt, k, w_out, idx_out, tid, kSmemGateThreads);
}

template <int EP, typename In>
int launch_gating_tma(const In* logits, int T, int E, int k, int norm, float* w, int32_t* idx, cudaStream_t s) {
  using St = StageT<EP, In>;
  CUtensorMap tm;
  if (int rc = make_tmap_rows128(&tm, logits, (uint64_t)T, (uint64_t)E, (int)sizeof(In), kSmemGateThreads)) return rc;
  const size_t smem = (size_t)gate::stage_bytes<EP, St, kRegMax<EP, In>, gate::StageSwz128>() + 1024;
  if (int rc = ensure_smem_limit(gating_tma_kernel<EP, In>, smem, "gating_softmax_topk")) return rc;
  const unsigned grid = (unsigned)((T + kSmemGateThreads - 1) / kSmemGateThreads);
  gating_tma_kernel<EP, In><<<grid, kSmemGateThreads, smem, s>>>(tm, T, E, k, norm, w, idx);
  return check_launch("gating_softmax_topk");
}

template <int EP, typename In>
int launch_gating_smem(const In* logits, int T, int E, int k, int norm, float* w, int32_t* idx,
                       cudaStream_t s) {
  if constexpr (EP >= 64 && sizeof(StageT<EP, In>) == sizeof(In))
    if (k <= gate::kRegSel && (E * (int)sizeof(In)) % 128 == 0)
      return launch_gating_tma<EP, In>(logits, T, E, k, norm, w, idx, s);
  const unsigned grid = (unsigned)((T + kSmemGateThreads - 1) / kSmemGateThreads);
  const size_t smem = (size_t)gate::stage_bytes<EP, StageT<EP, In>, kRegMax<EP, In>>();
  if (int rc = ensure_smem_limit(gating_smem_kernel<EP, In>, smem, "gating_softmax_topk")) return rc;
  gating_smem_kernel<EP, In><<<grid, kSmemGateThreads, smem, s>>>(logits, T, E, k, norm, w, idx);
  return check_launch("gating_softmax_topk");
}

template <int K, typename In>
int launch_rows8(const In* logits, int T, int E, int norm, float* w, int32_t* idx, cudaStream_t s) {
  const long blocks = ((long)T + kBlock - 1) / kBlock, cap = (long)num_sms() * 6;
  const unsigned grid = (unsigned)(blocks < cap ? blocks : cap);
  if (E == 8) gating_rows8_kernel<K, In, true><<<grid, kBlock, 0, s>>>(logits, T, E, norm, w, idx);
  else gating_rows8_kernel<K, In, false><<<grid, kBlock, 0, s>>>(logits, T, E, norm, w, idx);
  return check_launch("gating_softmax_topk");
}

template <typename In>
int launch_gating_rows8(const In* logits, int T, int E, int k, int norm, float* w, int32_t* idx,
                        cudaStream_t s) {
  switch (k) {
    case 1: return launch_rows8<1, In>(logits, T, E, norm, w, idx, s);
    case 2: return launch_rows8<2, In>(logits, T, E, norm, w, idx, s);
    case 3: return launch_rows8<3, In>(logits, T, E, norm, w, idx, s);
    case 4: return launch_rows8<4, In>(logits, T, E, norm, w, idx, s);
    case 5: return launch_rows8<5, In>(logits, T, E, norm, w, idx, s);
    case 6: return launch_rows8<6, In>(logits, T, E, norm, w, idx, s);
    case 7: return launch_rows8<7, In>(logits, T, E, norm, w, idx, s);
    default: return launch_rows8<8, In>(logits, T, E, norm, w, idx, s);
  }
}

template <int L, int V, typename In>
int launch_gating_t(const In* logits, int T, int E, int k, int norm, float* w, int32_t* idx,
                    cudaStream_t s) {
  const int tpb = kBlock / L;
  const int grid = (T + tpb - 1) / tpb;
  gating_kernel<L, V, In><<<grid, kBlock, 0, s>>>(logits, T, E, k, norm, w, idx);
  return check_launch("gating_softmax_topk");
}

// ---------------------------------------------------------------------------
// indices -> multihot: one thread writes 8 consecutive experts of one row when
// E % 8 == 0 (whole 32-byte sectors, indices_to_multihot8_kernel), else 4 (three
// 16/4-byte vector stores); it reads the row's k indices and probs as vectors
// when k is 1, 2, 4 or 8 (the row's threads share them in L1).

template <int K>
__device__ __forceinline__ void load_row(const int32_t* __restrict__ idx, const float* __restrict__ probs,
                                         long t, int (&e)[K], float (&p)[K]) {
  if constexpr (K == 8) {
    const int4 a = __ldg(reinterpret_cast<const int4*>(idx + t * 8));
    const int4 b = __ldg(reinterpret_cast<const int4*>(idx + t * 8) + 1);
    const float4 c = __ldg(reinterpret_cast<const float4*>(probs + t * 8));
    const float4 d = __ldg(reinterpret_cast<const float4*>(probs + t * 8) + 1);
    e[0] = a.x; e[1] = a.y; e[2] = a.z; e[3] = a.w; e[4] = b.x; e[5] = b.y; e[6] = b.z; e[7] = b.w;
    p[0] = c.x; p[1] = c.y; p[2] = c.z; p[3] = c.w; p[4] = d.x; p[5] = d.y; p[6] = d.z; p[7] = d.w;
  } else if constexpr (K == 4) {
    const int4 a = __ldg(reinterpret_cast<const int4*>(idx + t * 4));
    const float4 c = __ldg(reinterpret_cast<const float4*>(probs + t * 4));
    e[0] = a.x; e[1] = a.y; e[2] = a.z; e[3] = a.w;
    p[0] = c.x; p[1] = c.y; p[2] = c.z; p[3] = c.w;
  } else if constexpr (K == 2) {
    const int2 a = __ldg(reinterpret_cast<const int2*>(idx + t * 2));
    const float2 c = __ldg(reinterpret_cast<const float2*>(probs + t * 2));
    e[0] = a.x; e[1] = a.y;
    p[0] = c.x; p[1] = c.y;
  } else {
#pragma unroll
    for (int j = 0; j < K; ++j) {
      e[j] = __ldg(idx + t * K + j);
      p[j] = __ldg(probs + t * K + j);
    }
  }
}

// K > 0: k == K known at compile time; K == 0: any k (scalar loads).
template <int K>
__global__ void __launch_bounds__(kBlock) indices_to_multihot_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ probs, int T, int k, int E,
    uint8_t* __restrict__ mh, float* __restrict__ pm, int32_t* __restrict__ pos, int e4_shift) {
  const int E4 = (E + 3) >> 2;
  const long n = (long)T * E4;
  for (long tid = (long)blockIdx.x * blockDim.x + threadIdx.x; tid < n; tid += (long)gridDim.x * blockDim.x) {
    const long t = div_idx(tid, E4, e4_shift);
    const int e0 = (int)(tid - t * E4) * 4;
    unsigned m[4] = {0, 0, 0, 0};
    float p[4] = {0.f, 0.f, 0.f, 0.f};
    int q[4] = {-1, -1, -1, -1};
    if constexpr (K > 0) {
      int re[K];
      float rp[K];
      load_row<K>(idx, probs, t, re, rp);
#pragma unroll
      for (int j = K - 1; j >= 0; --j) {   // descending, so the lowest j is kept on a repeat
        const int d = re[j] - e0;
        if (re[j] >= 0 && re[j] < E && d >= 0 && d < 4) {
          m[d] = 1;
          p[d] = rp[j];
          q[d] = j;
        }
      }
    } else {
      for (int j = k - 1; j >= 0; --j) {
        const int e = __ldg(idx + t * k + j);
        const int d = e - e0;
        if (e >= 0 && e < E && d >= 0 && d < 4) {
          m[d] = 1;
          p[d] = __ldg(probs + t * k + j);
          q[d] = j;
        }
      }
    }
    const long base = t * (long)E + e0;
    if ((E & 3) == 0) {
      __stcs(reinterpret_cast<unsigned*>(mh + base), m[0] | (m[1] << 8) | (m[2] << 16) | (m[3] << 24));
      __stcs(reinterpret_cast<float4*>(pm + base), make_float4(p[0], p[1], p[2], p[3]));
      __stcs(reinterpret_cast<int4*>(pos + base), make_int4(q[0], q[1], q[2], q[3]));
    } else {
      for (int d = 0; d < 4 && e0 + d < E; ++d) {
        mh[base + d] = (uint8_t)m[d];
        pm[base + d] = p[d];
        pos[base + d] = q[d];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// multihot -> indices. Vector form (E % 4 == 0): G lanes per row, each reading
// NV aligned 16-byte vectors of the position map and of the probs; a lane
// writes the slots its experts fill, the group ORs the filled-slot masks and
// lane j % G writes any slot j that no expert fills. Every output slot is
// written once. Scalar form for other E.

template <int G, int NV>
__global__ void __launch_bounds__(kBlock) multihot_to_indices_vec_kernel(
    const float* __restrict__ pm, const int32_t* __restrict__ pos, int T, int E, int k,
    float* __restrict__ probs, int32_t* __restrict__ idx_out) {
  const int g = threadIdx.x & (G - 1);
  const unsigned gm = group_mask<G>();
  const long rows_per_grid = (long)gridDim.x * (kBlock / G);
  for (long t = (long)blockIdx.x * (kBlock / G) + threadIdx.x / G; t < T; t += rows_per_grid) {
    unsigned filled = 0;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int e0 = (v * G + g) * 4;
      const int4 q = __ldcs(reinterpret_cast<const int4*>(pos + t * E + e0));
      const float4 w = __ldcs(reinterpret_cast<const float4*>(pm + t * E + e0));
      const int qa[4] = {q.x, q.y, q.z, q.w};
      const float wa[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int d = 0; d < 4; ++d) {
        const int p = qa[d];
        if (p >= 0 && p < k) {
          probs[t * k + p] = wa[d];
          if (idx_out) idx_out[t * k + p] = e0 + d;
          filled |= 1u << p;
        }
      }
    }
#pragma unroll
    for (int off = G / 2; off >= 1; off >>= 1) filled |= __shfl_xor_sync(gm, filled, off, G);
    for (int j = g; j < k; j += G) {
      if (!((filled >> j) & 1u)) {
        probs[t * k + j] = 0.0f;
        if (idx_out) idx_out[t * k + j] = -1;
      }
    }
  }
}

template <int L, int V>
__global__ void __launch_bounds__(kBlock) multihot_to_indices_kernel(
    const float* __restrict__ pm, const int32_t* __restrict__ pos, int T, int E, int k,
    float* __restrict__ probs, int32_t* __restrict__ idx_out) {
  const int g = threadIdx.x & (L - 1);
  const long t = (long)blockIdx.x * (kBlock / L) + threadIdx.x / L;
  if (t >= T) return;
  const unsigned gm = group_mask<L>();
  unsigned filled = 0;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = g + i * L;
    if (e < E) {
      const int p = __ldg(pos + t * E + e);
      if (p >= 0 && p < k) {
        probs[t * k + p] = __ldg(pm + t * E + e);
        if (idx_out) idx_out[t * k + p] = e;
        filled |= 1u << p;
      }
    }
  }
#pragma unroll
  for (int off = L / 2; off >= 1; off >>= 1) filled |= __shfl_xor_sync(gm, filled, off, L);
  for (int j = g; j < k; j += L) {
    if (!((filled >> j) & 1u)) {
      probs[t * k + j] = 0.0f;
      if (idx_out) idx_out[t * k + j] = -1;
    }
  }
}

template <int L, int V>
int launch_m2i_t(const float* pm, const int32_t* pos, int T, int E, int k, float* probs,
                 int32_t* idx, cudaStream_t s) {
  const int tpb = kBlock / L;
  multihot_to_indices_kernel<L, V><<<(T + tpb - 1) / tpb, kBlock, 0, s>>>(pm, pos, T, E, k, probs, idx);
  return check_launch("multihot_to_indices");
}

template <int G, int NV>
int launch_m2i_vec(const float* pm, const int32_t* pos, int T, int E, int k, float* probs, int32_t* idx,
                   cudaStream_t s) {
  const int rows_per_block = kBlock / G;
  long blocks = ((long)T + rows_per_block - 1) / rows_per_block;
  const long cap = (long)num_sms() * 16;
  multihot_to_indices_vec_kernel<G, NV><<<(unsigned)(blocks < cap ? blocks : cap), kBlock, 0, s>>>(
      pm, pos, T, E, k, probs, idx);
  return check_launch("multihot_to_indices");
}

// E % 8 == 0: one thread per 8 experts of a row, so each of its pm / pos pieces is
// a whole 32-byte sector, written with one 256-bit store (V8, outputs 32-byte
// aligned) or two 128-bit ones. Measured on GB300: a thread that writes only
// half a sector per store (the 4-expert form) sends ~4x the bytes from L1 to L2
// even when the warp's stores are contiguous, and ran at 35% of the copy peak
// against 85-95% here.
template <int K, bool V8>
__global__ void __launch_bounds__(kBlock) indices_to_multihot8_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ probs, int T, int k, int E,
    uint8_t* __restrict__ mh, float* __restrict__ pm, int32_t* __restrict__ pos, int e8_shift) {
  const int E8 = E >> 3;
  const long n = (long)T * E8;
  for (long tid = (long)blockIdx.x * blockDim.x + threadIdx.x; tid < n; tid += (long)gridDim.x * blockDim.x) {
    const long t = div_idx(tid, E8, e8_shift);
    const int e0 = (int)(tid - t * E8) * 8;
    uint32_t mlo = 0, mhi = 0;
    float p[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int q[8] = {-1, -1, -1, -1, -1, -1, -1, -1};
    if constexpr (K > 0) {
      int re[K];
      float rp[K];
      load_row<K>(idx, probs, t, re, rp);
#pragma unroll
      for (int j = K - 1; j >= 0; --j) {   // descending, so the lowest j is kept on a repeat
        const int d = re[j] - e0;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          if (re[j] >= 0 && re[j] < E && d == c) { p[c] = rp[j]; q[c] = j; }
      }
    } else {
      for (int j = k - 1; j >= 0; --j) {
        const int e = __ldg(idx + t * k + j);
        const int d = e - e0;
        if (e >= 0 && e < E && d >= 0 && d < 8) {
          const float pj = __ldg(probs + t * k + j);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            if (d == c) { p[c] = pj; q[c] = j; }
        }
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      mlo |= (q[c] >= 0 ? 1u : 0u) << (8 * c);
      mhi |= (q[c + 4] >= 0 ? 1u : 0u) << (8 * c);
    }
    const long base = t * (long)E + e0;
    *reinterpret_cast<uint2*>(mh + base) = make_uint2(mlo, mhi);
    if constexpr (V8) {
      asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(pm + base), "f"(p[0]),
                   "f"(p[1]), "f"(p[2]), "f"(p[3]), "f"(p[4]), "f"(p[5]), "f"(p[6]), "f"(p[7])
                   : "memory");
      asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(pos + base), "r"(q[0]),
                   "r"(q[1]), "r"(q[2]), "r"(q[3]), "r"(q[4]), "r"(q[5]), "r"(q[6]), "r"(q[7])
                   : "memory");
    } else {
      *reinterpret_cast<float4*>(pm + base) = make_float4(p[0], p[1], p[2], p[3]);
      *reinterpret_cast<float4*>(pm + base + 4) = make_float4(p[4], p[5], p[6], p[7]);
      *reinterpret_cast<int4*>(pos + base) = make_int4(q[0], q[1], q[2], q[3]);
      *reinterpret_cast<int4*>(pos + base + 4) = make_int4(q[4], q[5], q[6], q[7]);
    }
  }
}

template <int K>
int launch_i2m(const int32_t* idx, const float* probs, int T, int k, int E, uint8_t* mh, float* pm,
               int32_t* pos, cudaStream_t s) {
  if (E % 8 == 0) {
    const long n8 = (long)T * (E / 8);
    const long blocks8 = (n8 + kBlock - 1) / kBlock;
    const long cap8 = (long)num_sms() * 16;
    const unsigned g = (unsigned)(blocks8 < cap8 ? blocks8 : cap8);
    const bool v8 = ((reinterpret_cast<uintptr_t>(pm) | reinterpret_cast<uintptr_t>(pos)) & 31) == 0;
    if (v8)
      indices_to_multihot8_kernel<K, true><<<g, kBlock, 0, s>>>(idx, probs, T, k, E, mh, pm, pos, pow2_shift(E / 8));
    else
      indices_to_multihot8_kernel<K, false><<<g, kBlock, 0, s>>>(idx, probs, T, k, E, mh, pm, pos, pow2_shift(E / 8));
    return check_launch("indices_to_multihot");
  }
  const long n = (long)T * ((E + 3) / 4);
  long blocks = (n + kBlock - 1) / kBlock;
  const long cap = (long)num_sms() * 16;
  indices_to_multihot_kernel<K><<<(unsigned)(blocks < cap ? blocks : cap), kBlock, 0, s>>>(
      idx, probs, T, k, E, mh, pm, pos, pow2_shift((E + 3) / 4));
  return check_launch("indices_to_multihot");
}

// ---------------------------------------------------------------------------
// Group-limited top-k: mlc-llm moe_misc.py, group_limited_greedy_topk.
// One warp per token; the choice scores (scores, + bias for noaux_tc) are kept
// in registers (lane l holds experts l, l+32, ...) and in a per-warp shared row
// from which lane g < n_group scores group g (its max, or the sum of its two
// largest for noaux_tc, both as float32 like the page). topk_group rounds of
// warp arg-max pick the groups, then k rounds pick experts inside them; the
// tie rule is the page's (larger value first, lower index on equality).

constexpr int kGroupWarps = 8;

template <int V>
__global__ void __launch_bounds__(kGroupWarps * 32) group_topk_kernel(
    const float* __restrict__ scores, const float* __restrict__ bias, int T, int E, int k, int n_group,
    int topk_group, int noaux, float* __restrict__ w_out, int32_t* __restrict__ idx_out) {
  extern __shared__ float rows[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const long t = (long)blockIdx.x * kGroupWarps + wid;
  if (t >= T) return;                          // whole warps leave together
  float* row = rows + wid * E;
  const int gs = E / n_group;
  float sv[V], cv[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    sv[i] = e < E ? __ldg(scores + t * E + e) : 0.0f;
    cv[i] = (e < E && noaux) ? sv[i] + __ldg(bias + e) : sv[i];
    if (e < E) row[e] = cv[i];
  }
  __syncwarp();
  // group scores (lanes g < n_group); each lane starts its scan at a different
  // column so the lanes hit different shared-memory banks (max and top-2 do not
  // depend on the scan order)
  unsigned gkey = 0;
  if (lane < n_group) {
    const float* g = row + lane * gs;
    float b1 = -FLT_MAX, b2 = -FLT_MAX;
    int c = lane % gs;
    for (int n = 0; n < gs; ++n) {
      const float x = g[c];
      if (x > b1) { b2 = b1; b1 = x; }
      else if (x > b2) b2 = x;
      if (++c == gs) c = 0;
    }
    gkey = gate::okey(noaux ? b1 + b2 : b1);
  }
  unsigned gsel = 0;
  {
    unsigned gk[1] = {gkey};
    unsigned gtaken = lane < n_group ? 0u : 1u;
    for (int j = 0; j < topk_group; ++j) {
      unsigned m;
      const int bi = gate::warp_argmax_round<1>(gk, gtaken, lane, &m);
      gsel |= 1u << bi;
      if (bi == lane) gtaken = 1u;
    }
  }
  // experts of the kept groups
  unsigned taken = 0;
  unsigned key[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    key[i] = gate::okey(cv[i]);
    if (e >= E || !((gsel >> (e / gs)) & 1u)) taken |= 1u << i;
  }
  float my_w = 0.0f;
  int my_i = -1;
  for (int j = 0; j < k; ++j) {
    unsigned m;
    const int bi = gate::warp_argmax_round<V>(key, taken, lane, &m);
    float s_owner = 0.0f;
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (lane + 32 * i == bi) s_owner = sv[i];
    const float bs = __shfl_sync(0xffffffffu, s_owner, bi & 31);
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) { my_w = noaux ? bs : gate::okey_value(m); my_i = bi; }
  }
  if (lane < k) {
    w_out[t * k + lane] = my_w;
    idx_out[t * k + lane] = my_i;
  }
}

// Groups of at most 32 experts, L >= n_group lanes per token (one per group). Lane g
// parks its group's choice scores in its own shared-memory row (32 + 1 floats:
// conflict-free) and keeps the maxima of the group's sub-groups of 8 in
// registers. The group score (max, or the sum of the two largest, computed with
// min/max only) and the topk_group best groups come first; then each of the k
// rounds takes every lane's best remaining (value, expert) from its sub-group
// maxima, merges the token's lanes with a butterfly on (value desc, expert asc),
// and only the lane owning the winner marks it taken (-inf) and rescans that
// sub-group. 8 lanes per token share the token's 1 KB of scores, so many warps
// fit per SM.
constexpr int kLaneSmemLd = 33;

template <int L>
__global__ void __launch_bounds__(kBlock) group_topk_lane_smem_kernel(
    const float* __restrict__ scores, const float* __restrict__ bias, int T, int E, int k, int n_group,
    int topk_group, int noaux, float* __restrict__ w_out, int32_t* __restrict__ idx_out) {
  __shared__ float park[kBlock * kLaneSmemLd];
  const int g = threadIdx.x & (L - 1);
  const unsigned gm = group_mask<L>();
  float* my = park + threadIdx.x * kLaneSmemLd;
  const int gs = E / n_group;
  const bool has = g < n_group;
  const int base = g * gs;
  const int nsub = (gs + 7) / 8;
  const long step = (long)gridDim.x * (kBlock / L);
  for (long t = (long)blockIdx.x * (kBlock / L) + threadIdx.x / L; t < T; t += step) {
    const float* row = scores + t * (long)E + base;
    float b1 = -FLT_MAX, b2 = -FLT_MAX;
    if (has && (gs & 3) == 0) {
      // all of the group's vectors (gs <= 32: at most 8) are requested before the
      // first is used: one memory round trip per token instead of one per vector
      float4 xq[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < gs / 4) xq[q] = __ldg(reinterpret_cast<const float4*>(row) + q);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (q >= gs / 4) break;
        float4 x = xq[q];
        if (noaux) {
          const float4 b = __ldg(reinterpret_cast<const float4*>(bias + base) + q);
          x.x += b.x; x.y += b.y; x.z += b.z; x.w += b.w;
        }
        const float v[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          my[4 * q + i] = v[i];
          const float lo = fminf(b1, v[i]);
          b1 = fmaxf(b1, v[i]);
          b2 = fmaxf(b2, lo);
        }
      }
    } else if (has) {
      for (int i = 0; i < gs; ++i) {
        const float v = noaux ? __ldg(row + i) + __ldg(bias + base + i) : __ldg(row + i);
        my[i] = v;
        const float lo = fminf(b1, v);
        b1 = fmaxf(b1, v);
        b2 = fmaxf(b2, lo);
      }
    }
    if (has)
      for (int i = gs; i < 8 * nsub; ++i) my[i] = -INFINITY;
    const float gscore = noaux ? b1 + b2 : b1;
    unsigned gsel = 0;
    for (int j = 0; j < topk_group; ++j) {
      float bv = gscore;
      int bi = (has && !((gsel >> g) & 1u)) ? g : kNone;
#pragma unroll
      for (int off = L / 2; off >= 1; off >>= 1) {
        const float ov = __shfl_xor_sync(gm, bv, off, L);
        const int oi = __shfl_xor_sync(gm, bi, off, L);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      gsel |= 1u << bi;
    }
    const bool live = has && ((gsel >> g) & 1u);
    // sub-group maxima (value, first expert holding it)
    float sv[4];
    int si[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float v = -INFINITY;
      int i0 = kNone;
      if (live && q < nsub) {
        v = my[8 * q];
        i0 = base + 8 * q;
#pragma unroll
        for (int c = 1; c < 8; ++c) {
          const float x = my[8 * q + c];
          i0 = x > v ? base + 8 * q + c : i0;
          v = fmaxf(v, x);
        }
      }
      sv[q] = v;
      si[q] = i0;
    }
    for (int j = 0; j < k; ++j) {
      float bv = sv[0];
      int bi = si[0];
#pragma unroll
      for (int q = 1; q < 4; ++q) {   // sub-groups in ascending expert order: strict > keeps the lower
        const bool b = sv[q] > bv;
        bv = b ? sv[q] : bv;
        bi = b ? si[q] : bi;
      }
      if (bi != kNone && bv == -INFINITY) bi = kNone;   // a dead or exhausted lane offers nothing
#pragma unroll
      for (int off = L / 2; off >= 1; off >>= 1) {
        const float ov = __shfl_xor_sync(gm, bv, off, L);
        const int oi = __shfl_xor_sync(gm, bi, off, L);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if (bi >= base && bi < base + gs) {   // this lane owns the winner: take it, rescan its sub-group
        const int q = (bi - base) >> 3;
        my[bi - base] = -INFINITY;
        float v = my[8 * q];
        int i0 = base + 8 * q;
#pragma unroll
        for (int c = 1; c < 8; ++c) {
          const float x = my[8 * q + c];
          i0 = x > v ? base + 8 * q + c : i0;
          v = fmaxf(v, x);
        }
#pragma unroll
        for (int qq = 0; qq < 4; ++qq)
          if (qq == q) { sv[qq] = v; si[qq] = i0; }
      }
      if ((j & (L - 1)) == g) {
        // noaux_tc reports the un-biased score of the chosen expert (a cached re-read)
        w_out[t * k + j] = noaux ? __ldg(scores + t * (long)E + bi) : bv;
        idx_out[t * k + j] = bi;
      }
    }
  }
}

// Groups of exactly 32 experts (DeepSeek-V3: 8 groups of 32), L >= n_group lanes
// per token, lane g owning group g. The token's lanes read its row as
// consecutive 16-byte vectors (a warp instruction covers whole 128-byte lines),
// add the bias from a padded shared-memory copy and drop each vector into the
// parked row of the lane owning its group (36-float rows: every 16-byte access
// pattern below is conflict-free per quarter warp). Each lane then reads its
// group back as 16-byte vectors, forms the group score and the maxima of its
// four sub-groups of 8. The topk_group groups are those of rank < topk_group
// among the token's group scores (score desc, group asc); each of the k rounds
// takes the token's largest offered value (a max butterfly), then the lowest
// expert offering it (a min butterfly), and the owning lane rescans one
// sub-group, as in group_topk_lane_smem_kernel.
constexpr int kG32Ld = 36;

template <int L>
__global__ void __launch_bounds__(kBlock) group_topk_g32_kernel(
    const float* __restrict__ scores, const float* __restrict__ bias, int T, int E, int k, int n_group,
    int topk_group, int noaux, float* __restrict__ w_out, int32_t* __restrict__ idx_out) {
  __shared__ __align__(16) float park[kBlock * kG32Ld];
  __shared__ __align__(16) float sbias[32 * kG32Ld];
  const int g = threadIdx.x & (L - 1);
  const unsigned gm = group_mask<L>();
  const bool has = g < n_group;
  const int nv = E >> 2;   // 16-byte vectors per row, 8 per group
  for (int f = threadIdx.x; f < n_group * 32; f += kBlock)
    sbias[(f >> 5) * kG32Ld + (f & 31)] = noaux ? __ldg(bias + f) : 0.0f;
  __syncthreads();
  float* my = park + threadIdx.x * kG32Ld;
  float* tp = park + (threadIdx.x & ~(L - 1)) * kG32Ld;   // the token's first parked row
  const long step = (long)gridDim.x * (kBlock / L);
  for (long t = (long)blockIdx.x * (kBlock / L) + threadIdx.x / L; t < T; t += step) {
    const float4* row4 = reinterpret_cast<const float4*>(scores + t * (long)E);
    float4 xq[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (g + L * i < nv) xq[i] = __ldg(row4 + g + L * i);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = g + L * i;
      if (v < nv) {
        const int at = (v >> 3) * kG32Ld + (v & 7) * 4;
        float4 x = xq[i];
        if (noaux) {
          const float4 b = *reinterpret_cast<const float4*>(sbias + at);
          x.x += b.x; x.y += b.y; x.z += b.z; x.w += b.w;
        }
        *reinterpret_cast<float4*>(tp + at) = x;
      }
    }
    __syncwarp(gm);
    // sub-group maxima (value, first expert holding it) from the parked group
    float sv[4];
    int si[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      sv[q] = -INFINITY;
      si[q] = kNone;
    }
    if (has) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 a = *reinterpret_cast<const float4*>(my + 8 * q);
        const float4 c = *reinterpret_cast<const float4*>(my + 8 * q + 4);
        const float x[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
        float v = x[0];
        int i0 = 0;
#pragma unroll
        for (int j = 1; j < 8; ++j) {
          i0 = x[j] > v ? j : i0;
          v = fmaxf(v, x[j]);
        }
        sv[q] = v;
        si[q] = 32 * g + 8 * q + i0;
      }
    }
    // group score: its largest value, or (noaux_tc) the float32 sum of its two
    // largest: the largest of the other sub-groups' maxima and of the first
    // holding sub-group without its arg-max
    const float b1 = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
    float gscore = has ? b1 : -INFINITY;
    if (noaux && has) {
      int qs = 3;
#pragma unroll
      for (int q = 2; q >= 0; --q) qs = sv[q] == b1 ? q : qs;
      float b2 = -INFINITY;
      int ia = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        b2 = fmaxf(b2, q == qs ? -INFINITY : sv[q]);
        ia = q == qs ? si[q] & 7 : ia;
      }
      const float4 a = *reinterpret_cast<const float4*>(my + 8 * qs);
      const float4 c = *reinterpret_cast<const float4*>(my + 8 * qs + 4);
      const float x[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) b2 = fmaxf(b2, j == ia ? -INFINITY : x[j]);
      gscore = b1 + b2;
    }
    // the topk_group best groups (score desc, group asc): a group's rank among the token's lanes
    int rank = 0;
#pragma unroll
    for (int gg = 0; gg < L; ++gg) {
      const float o = __shfl_sync(gm, gscore, gg, L);
      rank += (o > gscore || (o == gscore && gg < g)) ? 1 : 0;
    }
    if (!(has && rank < topk_group)) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        sv[q] = -INFINITY;
        si[q] = kNone;
      }
    }
    for (int j = 0; j < k; ++j) {
      float bv = sv[0];
      int bi = si[0];
#pragma unroll
      for (int q = 1; q < 4; ++q) {   // sub-groups in ascending expert order: strict > keeps the lower
        const bool b = sv[q] > bv;
        bv = b ? sv[q] : bv;
        bi = b ? si[q] : bi;
      }
      // the token's largest offer, then the lowest expert offering it
      float mx = bv;
#pragma unroll
      for (int off = L / 2; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(gm, mx, off, L));
      int ci = bv == mx ? bi : kNone;
#pragma unroll
      for (int off = L / 2; off >= 1; off >>= 1) ci = min(ci, __shfl_xor_sync(gm, ci, off, L));
      bv = mx;
      bi = ci;
      if ((bi >> 5) == g) {   // this lane owns the winner: take it, rescan its sub-group
        const int q = (bi >> 3) & 3;
        my[bi & 31] = -INFINITY;
        const float4 a = *reinterpret_cast<const float4*>(my + 8 * q);
        const float4 c = *reinterpret_cast<const float4*>(my + 8 * q + 4);
        const float x[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
        float v = x[0];
        int i0 = 0;
#pragma unroll
        for (int cc = 1; cc < 8; ++cc) {
          i0 = x[cc] > v ? cc : i0;
          v = fmaxf(v, x[cc]);
        }
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          sv[qq] = qq == q ? v : sv[qq];
          si[qq] = qq == q ? 32 * g + 8 * q + i0 : si[qq];
        }
      }
      if ((j & (L - 1)) == g) {
        // noaux_tc reports the un-biased score of the chosen expert (a cached re-read)
        w_out[t * k + j] = noaux ? __ldg(scores + t * (long)E + bi) : bv;
        idx_out[t * k + j] = bi;
      }
    }
    __syncwarp(gm);   // the parked rows are rewritten by the next token's vectors
  }
}

template <int L>
int launch_group_g32(const float* scores, const float* bias, int T, int E, int k, int n_group, int topk_group,
                     int noaux, float* w, int32_t* idx, cudaStream_t s) {
  const int tpb = kBlock / L;
  const long blocks = ((long)T + tpb - 1) / tpb;
  const long cap = (long)num_sms() * 8;
  group_topk_g32_kernel<L><<<(unsigned)(blocks < cap ? blocks : cap), kBlock, 0, s>>>(
      scores, bias, T, E, k, n_group, topk_group, noaux, w, idx);
  return check_launch("group_limited_topk");
}

// Thread-per-token form for E <= 256: the choice row and the group scores live in
// shared memory (column-major, conflict free); groups are picked by scanning
// the group scores, experts of the other groups are set to -inf, then k rounds
// over register maxima of 8-expert blocks as in gating_smem_kernel.
constexpr int kSmemGroupThreads = 64;

template <int EP>
__global__ void __launch_bounds__(kSmemGroupThreads) group_topk_smem_kernel(
    const float* __restrict__ scores, const float* __restrict__ bias, int T, int E, int k, int n_group,
    int topk_group, int noaux, float* __restrict__ w_out, int32_t* __restrict__ idx_out) {
  constexpr int B = EP / 8;
  constexpr int LD = kSmemGroupThreads + 1;        // padded column stride
  extern __shared__ float sm[];                    // [EP][LD] choice | [32][LD] group score
  const int tid = threadIdx.x;
  const long t0 = (long)blockIdx.x * kSmemGroupThreads;
  const int nt = (int)min((long)kSmemGroupThreads, (long)T - t0);
  const float* blk = scores + t0 * (long)E;
  if ((E & 3) == 0) {   // U loads in flight per thread, then their stores
    constexpr int U = 8;
    const int n4 = nt * E / 4;
    const float4* src = reinterpret_cast<const float4*>(blk);
    for (int f0 = tid; f0 < n4; f0 += U * kSmemGroupThreads) {
      float4 q[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (f0 + u * kSmemGroupThreads < n4) q[u] = __ldg(src + f0 + u * kSmemGroupThreads);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int f = f0 + u * kSmemGroupThreads;
        if (f < n4) {
          const int tl = (int)((uint32_t)(4 * f) / (uint32_t)E), e0 = 4 * f - tl * E;
          if (noaux) {
            const float4 b = __ldg(reinterpret_cast<const float4*>(bias + e0));
            q[u].x += b.x; q[u].y += b.y; q[u].z += b.z; q[u].w += b.w;
          }
          sm[e0 * LD + tl] = q[u].x;
          sm[(e0 + 1) * LD + tl] = q[u].y;
          sm[(e0 + 2) * LD + tl] = q[u].z;
          sm[(e0 + 3) * LD + tl] = q[u].w;
        }
      }
    }
  } else {
    for (int f = tid; f < nt * E; f += kSmemGroupThreads) {
      const int tl = f / E, e = f - tl * E;
      sm[e * LD + tl] = noaux ? __ldg(blk + f) + __ldg(bias + e) : __ldg(blk + f);
    }
  }
  for (int e = E; e < EP; ++e) sm[e * LD + tid] = -INFINITY;
  __syncthreads();
  if (tid >= nt) return;
  const long t = t0 + tid;
  auto at = [&](int i) -> float& { return sm[i * LD + tid]; };
  auto gsc = [&](int g) -> float& { return sm[(EP + g) * LD + tid]; };
  const float* row = scores + t * (long)E;
  const int gs = E / n_group;
  // group scores: max, or the float32 sum of the two largest
  for (int g = 0; g < n_group; ++g) {
    float b1 = -FLT_MAX, b2 = -FLT_MAX;
    for (int c = 0; c < gs; ++c) {
      const float x = at(g * gs + c);
      if (x > b1) { b2 = b1; b1 = x; }
      else if (x > b2) b2 = x;
    }
    gsc(g) = noaux ? b1 + b2 : b1;
  }
  unsigned gsel = 0;
  for (int j = 0; j < topk_group; ++j) {
    int bg = -1;
    float bv = 0.0f;
    for (int g = 0; g < n_group; ++g)
      if (!((gsel >> g) & 1u) && (bg < 0 || gsc(g) > bv)) { bv = gsc(g); bg = g; }
    gsel |= 1u << bg;
  }
  for (int g = 0; g < n_group; ++g)
    if (!((gsel >> g) & 1u))
      for (int c = 0; c < gs; ++c) at(g * gs + c) = -INFINITY;
  float bvv[B];
  int bii[B];
#pragma unroll
  for (int b = 0; b < B; ++b) {
    float v = at(8 * b);
    int i = 8 * b;
#pragma unroll
    for (int c = 1; c < 8; ++c) {
      const float x = at(8 * b + c);
      if (x > v) { v = x; i = 8 * b + c; }
    }
    bvv[b] = v;
    bii[b] = i;
  }
  for (int j = 0; j < k; ++j) {
    float bv = bvv[0];
    int bi = bii[0], bb = 0;
#pragma unroll
    for (int b = 1; b < B; ++b)
      if (bvv[b] > bv) { bv = bvv[b]; bi = bii[b]; bb = b; }
    at(bi) = -INFINITY;
    float nv = at(8 * bb);
    int ni = 8 * bb;
#pragma unroll
    for (int c = 1; c < 8; ++c) {
      const float x = at(8 * bb + c);
      if (x > nv) { nv = x; ni = 8 * bb + c; }
    }
#pragma unroll
    for (int b = 0; b < B; ++b)
      if (b == bb) { bvv[b] = nv; bii[b] = ni; }
    w_out[t * k + j] = noaux ? __ldg(row + bi) : bv;
    idx_out[t * k + j] = bi;
  }
}

template <int EP>
int launch_group_smem(const float* scores, const float* bias, int T, int E, int k, int n_group, int topk_group,
                      int noaux, float* w, int32_t* idx, cudaStream_t s) {
  const size_t smem = (size_t)(EP + 32) * (kSmemGroupThreads + 1) * sizeof(float);
  if (int rc = ensure_smem_limit(group_topk_smem_kernel<EP>, smem, "group_limited_topk")) return rc;
  group_topk_smem_kernel<EP><<<(T + kSmemGroupThreads - 1) / kSmemGroupThreads, kSmemGroupThreads, smem, s>>>(
      scores, bias, T, E, k, n_group, topk_group, noaux, w, idx);
  return check_launch("group_limited_topk");
}

template <int L>
int launch_group_lane_smem(const float* scores, const float* bias, int T, int E, int k, int n_group, int topk_group,
                           int noaux, float* w, int32_t* idx, cudaStream_t s) {
  const int tpb = kBlock / L;
  const long blocks = ((long)T + tpb - 1) / tpb;
  const long cap = (long)num_sms() * 16;
  group_topk_lane_smem_kernel<L><<<(unsigned)(blocks < cap ? blocks : cap), kBlock, 0, s>>>(
      scores, bias, T, E, k, n_group, topk_group, noaux, w, idx);
  return check_launch("group_limited_topk");
}

template <int V>
int launch_group_t(const float* scores, const float* bias, int T, int E, int k, int n_group,
                   int topk_group, int noaux, float* w, int32_t* idx, cudaStream_t s) {
  const size_t smem = (size_t)kGroupWarps * E * sizeof(float);
  if (int rc = ensure_smem_limit(group_topk_kernel<V>, (size_t)kGroupWarps * MOE_MAX_EXPERTS * sizeof(float),
                                 "group_limited_topk"))
    return rc;
  group_topk_kernel<V><<<(T + kGroupWarps - 1) / kGroupWarps, kGroupWarps * 32, smem, s>>>(
      scores, bias, T, E, k, n_group, topk_group, noaux, w, idx);
  return check_launch("group_limited_topk");
}

// E <= 8: a thread per token, row in registers (k <= E <= 8); E <= 128: the staged thread-per-token
// kernel; wider rows: L lanes of 64 experts per token.
template <typename In>
int launch_gating_any(const In* logits, int T, int E, int k, int norm, float* w, int32_t* idx,
                      cudaStream_t s, const char* name) {
  if (T == 0) return MOE_OK;
  ProfScope ps(name, s);
  if (E <= 8) return launch_gating_rows8<In>(logits, T, E, k, norm, w, idx, s);
  if (E <= 16) return launch_gating_smem<16, In>(logits, T, E, k, norm, w, idx, s);
  if (E <= 32) return launch_gating_smem<32, In>(logits, T, E, k, norm, w, idx, s);
  if (E <= 64) return launch_gating_smem<64, In>(logits, T, E, k, norm, w, idx, s);
  if (E <= 128) return launch_gating_smem<128, In>(logits, T, E, k, norm, w, idx, s);
  if (E <= 256) return launch_gating_t<4, 64, In>(logits, T, E, k, norm, w, idx, s);
  if (E <= 512) return launch_gating_t<8, 64, In>(logits, T, E, k, norm, w, idx, s);
  return launch_gating_t<16, 64, In>(logits, T, E, k, norm, w, idx, s);
}

}  // namespace

int launch_gating(const float* logits, int T, int E, int k, int norm, float* w, int32_t* idx,
                  cudaStream_t s) {
  return launch_gating_any(logits, T, E, k, norm, w, idx, s, "gating_softmax_topk");
}

int launch_gating_bf16(const void* logits, int T, int E, int k, int norm, float* w, int32_t* idx,
                       cudaStream_t s) {
  return launch_gating_any(static_cast<const __nv_bfloat16*>(logits), T, E, k, norm, w, idx, s,
                           "gating_softmax_topk_bf16");
}

int launch_indices_to_multihot(const int32_t* idx, const float* probs, int T, int k, int E,
                               uint8_t* mh, float* pm, int32_t* pos, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  ProfScope ps("indices_to_multihot", s);
  switch (k) {
    case 1: return launch_i2m<1>(idx, probs, T, k, E, mh, pm, pos, s);
    case 2: return launch_i2m<2>(idx, probs, T, k, E, mh, pm, pos, s);
    case 4: return launch_i2m<4>(idx, probs, T, k, E, mh, pm, pos, s);
    case 8: return launch_i2m<8>(idx, probs, T, k, E, mh, pm, pos, s);
    default: return launch_i2m<0>(idx, probs, T, k, E, mh, pm, pos, s);
  }
}

int launch_multihot_to_indices(const float* pm, const int32_t* pos, int T, int E, int k,
                               float* probs, int32_t* idx, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  ProfScope ps("multihot_to_indices", s);
  switch (E) {
    case 4: return launch_m2i_vec<1, 1>(pm, pos, T, E, k, probs, idx, s);
    case 8: return launch_m2i_vec<2, 1>(pm, pos, T, E, k, probs, idx, s);
    case 16: return launch_m2i_vec<4, 1>(pm, pos, T, E, k, probs, idx, s);
    case 32: return launch_m2i_vec<8, 1>(pm, pos, T, E, k, probs, idx, s);
    case 64: return launch_m2i_vec<16, 1>(pm, pos, T, E, k, probs, idx, s);
    case 128: return launch_m2i_vec<32, 1>(pm, pos, T, E, k, probs, idx, s);
    case 256: return launch_m2i_vec<32, 2>(pm, pos, T, E, k, probs, idx, s);
    case 512: return launch_m2i_vec<32, 4>(pm, pos, T, E, k, probs, idx, s);
    case 1024: return launch_m2i_vec<32, 8>(pm, pos, T, E, k, probs, idx, s);
    default: break;
  }
  MOE_DISPATCH_LV(E, launch_m2i_t, pm, pos, T, E, k, probs, idx, s);
}

int launch_group_limited_topk(const float* scores, const float* bias, int T, int E, int k, int n_group,
                              int topk_group, int noaux, float* w, int32_t* idx, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  ProfScope ps("group_limited_topk", s);
  const int gs = E / n_group;
  if (gs == 32) {   // groups of 32: coalesced row reads, one lane per group
    if (n_group <= 4) return launch_group_g32<4>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
    if (n_group <= 8) return launch_group_g32<8>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
    if (n_group <= 16) return launch_group_g32<16>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
    return launch_group_g32<32>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
  }
  if (gs <= 32) {   // one lane per group (measured 1.7x faster than a thread per token at E = 256)
    if (n_group <= 4) return launch_group_lane_smem<4>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
    if (n_group <= 8) return launch_group_lane_smem<8>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
    if (n_group <= 16) return launch_group_lane_smem<16>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
    return launch_group_lane_smem<32>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
  }
  if (E <= 64) return launch_group_smem<64>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
  if (E <= 128) return launch_group_smem<128>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
  if (E <= 256) return launch_group_smem<256>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
  if (E <= 32) return launch_group_t<1>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
  if (E <= 64) return launch_group_t<2>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
  if (E <= 128) return launch_group_t<4>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
  if (E <= 256) return launch_group_t<8>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
  if (E <= 512) return launch_group_t<16>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
  return launch_group_t<32>(scores, bias, T, E, k, n_group, topk_group, noaux, w, idx, s);
}

}  // namespace moe
