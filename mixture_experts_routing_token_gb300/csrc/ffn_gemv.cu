// Expert FFN of one or two tokens as matrix-vector products on the CUDA cores.
//
// project_6 moe_expert_gemm.cpp, moe_decode_experts: for each expert a token is
// routed to, FC1 (x @ w13[e]^T), silu_and_mul, FC2 (act @ w2[e]^T), scaled by
// the routing weight and summed over the token's k experts.
//
// With one or two tokens every weight element meets at most two activation
// values: the step is the routed experts' weight bytes, each read once from
// HBM, and no contraction for the tensor cores (tiles of 128 weight rows give a
// few dozen tiles per call and leave many of the 152 SMs idle). Here the work
// is cut into units of whole weight rows spread evenly over all SMs:
//   FC1  unit (active expert a, activation column i): gate row i and up row
//        I + i of w13[e], each lane streaming 16-byte pieces (eight of each row
//        in flight) against the token rows held in shared memory as float32;
//        act[p][i] = silu(x_t . gate) * (x_t . up) for each sorted slot p of e,
//        token t = sorted_ids[p];
//   FC2  unit (output column c, token t), the combine folded in:
//        out[t][c] = sum over j of w[t, j] * (w2[e_tj][c] . act[p_tj]), summed in
//        float32 and rounded once. A warp asks for all k rows of a unit at once
//        with asynchronous copies into its own shared-memory buffer (no registers
//        held while they are on their way) and reduces the unit from there. Units
//        of one column are adjacent, so a row both tokens use is read once from HBM.
//
// Every kernel pays a fixed cost before its loads reach full rate and after
// they drain (measured: a read-only kernel over 46 MB takes 16 us where the copy
// bandwidth asks 7). Inside the layer call the whole FFN is therefore one
// kernel (decode_pipe_kernel): every CTA routes the batch itself; its FC1 warps
// stream FC1 units (after a first unit each, in order from a counter that all
// CTAs share, so faster SMs take more) and count each finished unit on its
// expert's counter; its FC2 warps run behind them, one expert at a time as its
// counter completes, on the CTA's own output columns: the expert's w2 rows for
// those columns come into shared memory by bulk copies two of the warp's turns
// ahead and meet the expert's activation rows on the tensor cores (mma.sync),
// so FC2 streams with FC1 and only the last expert's FC2 and the combine follow
// it. The counters are a workspace region that the routing kernel launched just
// before zeroes, every wait on them is bounded, and the grid leaves one SM to
// that routing kernel, so that every CTA is resident. Elsewhere (routing given
// by the caller, or E > 64) FC1 and FC2 are two kernels, FC2 on the CUDA cores.
#include "common.cuh"
#include "gating_device.cuh"
#include "sm100_ptx.cuh"   // smem_u32, globaltimer

namespace moe {
namespace {

constexpr int kGemvThreads = 256;                        // FC1 kernel: two CTAs per SM
constexpr int kPieces = 8;                               // FC1: 16-byte pieces per lane per row in flight
constexpr int kMaxSlots = kGemvMaxTokens * MOE_MAX_TOPK;
constexpr int kRouteExperts = 64;                        // in-CTA routing (gate::route_block): E <= 64
constexpr int kFc2Buffers = 8;                           // FC2 warps with a row buffer each, at most
constexpr int kFc2Threads = kFc2Buffers * 32;            // FC2 kernel
constexpr size_t kFc2SmemMax = 200 * 1024;               // FC2 kernel: buffers + activation rows

struct GemvParams {
  const uint4* hidden;   // [T, H] bf16
  const uint4* w13;      // [E, 2I, H] bf16
  const uint4* w2;       // [E, H, I] bf16
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* sorted_ids;
  const float* sorted_w;
  const int32_t* reverse;
  __nv_bfloat16* act;    // [S, I], sorted slot order
  __nv_bfloat16* out;    // [T, H]
  const float* logits;   // route the batch inside every CTA (E <= 64), or null
  int32_t* sync;         // one-kernel FFN: kDecodeSyncWords counters, zero at launch
  int32_t* status;
  uint64_t wait_ns;      // limit of the waits on those counters and copies (moe_set_wait_limit_ns)
  int T, H, I, E, k;
};

// Shared memory of FC2: one buffer (the k weight rows of one unit) per FC2 warp,
// the batch's activation rows (bf16), then (layer kernel) the token rows (float32).
struct Fc2Layout {
  int buffers;
  size_t slot, ring, act, x, total;
};

__host__ __device__ inline Fc2Layout fc2_layout(int T, int k, int H, int I) {
  Fc2Layout L;
  const size_t row = (size_t)I * 2;
  L.slot = ((size_t)k * row + 127) & ~(size_t)127;
  L.act = ((size_t)T * k * row + 127) & ~(size_t)127;
  L.x = 0;
  const size_t cap = kFc2SmemMax;
  const size_t room = cap > L.act + L.x ? cap - L.act - L.x : 0;
  const size_t fit = room / L.slot;
  L.buffers = (int)(fit < (size_t)kFc2Buffers ? fit : (size_t)kFc2Buffers);
  L.ring = L.slot * L.buffers;
  L.total = L.ring + L.act + L.x + 128;   // + alignment of the base to 128 bytes
  return L;
}

// L2 policy for data used once: evicted before other lines.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Weight rows are read once: not kept in L1, first out of L2.
__device__ __forceinline__ uint4 ld_stream(const uint4* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

// 16 bytes global -> shared without a register (L1 bypassed).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ptx::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// bf16 halves of a 32-bit word as float32 (exact).
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// acc + the dot product of eight bf16 pairs, float32 FMAs in element order.
__device__ __forceinline__ float dot8(const uint4& w, const uint4& x, float acc) {
  acc = fmaf(bf_lo(w.x), bf_lo(x.x), acc);
  acc = fmaf(bf_hi(w.x), bf_hi(x.x), acc);
  acc = fmaf(bf_lo(w.y), bf_lo(x.y), acc);
  acc = fmaf(bf_hi(w.y), bf_hi(x.y), acc);
  acc = fmaf(bf_lo(w.z), bf_lo(x.z), acc);
  acc = fmaf(bf_hi(w.z), bf_hi(x.z), acc);
  acc = fmaf(bf_lo(w.w), bf_lo(x.w), acc);
  acc = fmaf(bf_hi(w.w), bf_hi(x.w), acc);
  return acc;
}

// acc + the dot product of eight bf16 weights with eight float32 values (x0: the
// first four), float32 FMAs in element order.
__device__ __forceinline__ float dot8f(const uint4& w, const float4& x0, const float4& x1, float acc) {
  acc = fmaf(bf_lo(w.x), x0.x, acc);
  acc = fmaf(bf_hi(w.x), x0.y, acc);
  acc = fmaf(bf_lo(w.y), x0.z, acc);
  acc = fmaf(bf_hi(w.y), x0.w, acc);
  acc = fmaf(bf_lo(w.z), x1.x, acc);
  acc = fmaf(bf_hi(w.z), x1.y, acc);
  acc = fmaf(bf_lo(w.w), x1.z, acc);
  acc = fmaf(bf_hi(w.w), x1.w, acc);
  return acc;
}

// The bf16 values of p[0, n) (n a multiple of 8) as float32 in dst, by the whole block.
__device__ __forceinline__ void stage_f32(const uint4* __restrict__ p, long n, float4* dst) {
  for (long c = threadIdx.x; c < n / 8; c += blockDim.x) {
    const uint4 v = p[c];
    dst[2 * c] = make_float4(bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y));
    dst[2 * c + 1] = make_float4(bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w));
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// The experts with tokens, ascending, into a_e[0, *a_n) (warp 0 of the block).
__device__ __forceinline__ void active_experts(const int32_t* counts, int E, int32_t* a_e, int* a_n) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  int n = 0;
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int e = e0 + lane;
    const bool on = e < E && counts[e] > 0;
    const unsigned m = __ballot_sync(0xffffffffu, on);
    const int at = n + __popc(m & ((1u << lane) - 1u));
    if (on && at < kMaxSlots) a_e[at] = e;
    n += __popc(m);
  }
  if (lane == 0) *a_n = min(n, kMaxSlots);
}

// FC1 unit (expert e, column i) by the calling warp: gate row i and up row I + i
// of w13[e] against the expert's token rows (xs, float32), silu_and_mul, act
// written by lane 0 (slot rows offsets[e] ..).
// TT: most tokens an expert can have (the batch size bound).
template <int TT, int PIECES = kPieces>
__device__ __forceinline__ void fc1_unit(const GemvParams& P, const float4* xs, int e, const int32_t* counts,
                                         const int32_t* offsets, const int32_t* sorted_ids, int i, uint64_t pol) {
  const int lane = threadIdx.x & 31;
  const int nch = P.H >> 3;
  const int cnt = min(counts[e], TT);
  const int p0 = offsets[e];
  int tok[TT];
#pragma unroll
  for (int r = 0; r < TT; ++r) tok[r] = r < cnt ? sorted_ids[p0 + r] : 0;
  const uint4* g = P.w13 + ((long)e * 2 * P.I + i) * nch;
  const uint4* up = g + (long)P.I * nch;
  float ag[TT], au[TT];
#pragma unroll
  for (int r = 0; r < TT; ++r) ag[r] = au[r] = 0.0f;
  for (int c0 = 0; c0 < nch; c0 += 32 * PIECES) {
    uint4 wg[PIECES], wu[PIECES];
#pragma unroll
    for (int b = 0; b < PIECES; ++b) {
      const int c = c0 + b * 32 + lane;
      if (c < nch) {
        wg[b] = ld_stream(g + c, pol);
        wu[b] = ld_stream(up + c, pol);
      }
    }
#pragma unroll
    for (int b = 0; b < PIECES; ++b) {
      const int c = c0 + b * 32 + lane;
      if (c < nch) {
#pragma unroll
        for (int r = 0; r < TT; ++r)
          if (r < cnt) {
            const float4 x0 = xs[(tok[r] * nch + c) * 2], x1 = xs[(tok[r] * nch + c) * 2 + 1];
            ag[r] = dot8f(wg[b], x0, x1, ag[r]);
            au[r] = dot8f(wu[b], x0, x1, au[r]);
          }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < TT; ++r) {
    ag[r] = warp_sum(ag[r]);
    au[r] = warp_sum(au[r]);
  }
  if (lane == 0)
#pragma unroll
    for (int r = 0; r < TT; ++r)
      if (r < cnt) P.act[(long)(p0 + r) * P.I + i] = __float2bfloat16_rn(silu(ag[r]) * au[r]);
}

// FC1 units u0, u0 + ustride, ... < u1 (unit u = a * I + i), taken in turn by the
// block's warps.
template <int TT, int PIECES = kPieces>
__device__ __forceinline__ void fc1_units(const GemvParams& P, const float4* xs, const int32_t* a_e,
                                          const int32_t* counts, const int32_t* offsets,
                                          const int32_t* sorted_ids, long u0, long u1, long ustride = 1) {
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const uint64_t pol = evict_first_policy();
  for (long u = u0 + warp * ustride; u < u1; u += nwarps * ustride) {
    const int a = (int)(u / P.I), i = (int)(u - (long)a * P.I);
    fc1_unit<TT, PIECES>(P, xs, a_e[a], counts, offsets, sorted_ids, i, pol);
  }
}

// FC1 pair (expert e, columns i and i + 1, i even) by the calling warp: gate rows
// i, i + 1 and up rows I + i, I + i + 1 of w13[e] (two contiguous row pairs, all
// four rows' pieces in flight together) against the expert's token rows,
// silu_and_mul, both activations written by lane 0 as one 4-byte store.
template <int TT>
__device__ __forceinline__ void fc1_pair(const GemvParams& P, const float4* xs, int e, const int32_t* counts,
                                         const int32_t* offsets, const int32_t* sorted_ids, int i, uint64_t pol) {
  const int lane = threadIdx.x & 31;
  const int nch = P.H >> 3;
  const int cnt = min(counts[e], TT);
  const int p0 = offsets[e];
  int tok[TT];
#pragma unroll
  for (int r = 0; r < TT; ++r) tok[r] = r < cnt ? sorted_ids[p0 + r] : 0;
  const uint4* g = P.w13 + ((long)e * 2 * P.I + i) * nch;   // gate rows i, i + 1
  const uint4* up = g + (long)P.I * nch;                     // up rows I + i, I + i + 1
  float acc[4][TT];
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int r = 0; r < TT; ++r) acc[q][r] = 0.0f;
  for (int c0 = 0; c0 < nch; c0 += 32 * kPieces) {
    uint4 wv[4][kPieces];
#pragma unroll
    for (int b = 0; b < kPieces; ++b) {
      const int c = c0 + b * 32 + lane;
      if (c < nch) {
        wv[0][b] = ld_stream(g + c, pol);
        wv[1][b] = ld_stream(g + nch + c, pol);
        wv[2][b] = ld_stream(up + c, pol);
        wv[3][b] = ld_stream(up + nch + c, pol);
      }
    }
#pragma unroll
    for (int b = 0; b < kPieces; ++b) {
      const int c = c0 + b * 32 + lane;
      if (c < nch) {
#pragma unroll
        for (int r = 0; r < TT; ++r)
          if (r < cnt) {
            const float4 x0 = xs[(tok[r] * nch + c) * 2], x1 = xs[(tok[r] * nch + c) * 2 + 1];
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q][r] = dot8f(wv[q][b], x0, x1, acc[q][r]);
          }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int r = 0; r < TT; ++r) acc[q][r] = warp_sum(acc[q][r]);
  if (lane == 0)
#pragma unroll
    for (int r = 0; r < TT; ++r)
      if (r < cnt)
        *reinterpret_cast<__nv_bfloat162*>(P.act + (long)(p0 + r) * P.I + i) =
            __floats2bfloat162_rn(silu(acc[0][r]) * acc[2][r], silu(acc[1][r]) * acc[3][r]);
}

// FC2 unit u = c * T + t: the weight rows of the token's valid slots (s_e[q] >= 0)
// into buf [k][I / 8], asynchronously, by the calling warp.
__device__ __forceinline__ void fc2_fetch(const GemvParams& P, const int32_t* s_e, long u, uint4* buf,
                                          int ld = 0, int j0 = 0, int jstep = 1) {
  const int lane = threadIdx.x & 31, nch = P.I >> 3;
  if (ld == 0) ld = nch;   // row stride of buf in 16-byte pieces; rows j0, j0 + jstep, ...
  const int c = (int)(u / P.T), t = (int)(u - (long)c * P.T);
  for (int j = j0; j < P.k; j += jstep) {
    const int e = s_e[t * P.k + j];
    if (e < 0) continue;
    const uint4* src = P.w2 + ((long)e * P.H + c) * nch;
    for (int pc = lane; pc < nch; pc += 32) cp_async16(buf + j * ld + pc, src + pc);
  }
  cp_async_commit();
}

// FC2 units u0 + i, i = w, w + nbuf, ... < nloc of FC2 warp w (its buffer holding
// the rows of its first unit already requested): out[t][c] as above.
__device__ __forceinline__ void fc2_units(const GemvParams& P, const int32_t* s_pos, const int32_t* s_e,
                                          const float* s_w, const uint4* act_s, uint4* buf, long u0, int nloc,
                                          int nbuf) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nch = P.I >> 3;
  for (int i = warp; i < nloc; i += nbuf) {
    cp_async_wait_all();
    __syncwarp();
    const long u = u0 + i;
    const int c = (int)(u / P.T), t = (int)(u - (long)c * P.T);
    float acc = 0.0f;
    for (int j = 0; j < P.k; ++j) {
      const int q = t * P.k + j;
      if (s_e[q] < 0) continue;
      const uint4* wr = buf + j * nch;
      const uint4* ar = act_s + s_pos[q] * nch;
      float sj = 0.0f;
      for (int pc = lane; pc < nch; pc += 32) sj = dot8(wr[pc], ar[pc], sj);
      acc = fmaf(s_w[q], sj, acc);
    }
    __syncwarp();   // every lane is done with the buffer
    if (i + nbuf < nloc) fc2_fetch(P, s_e, u0 + i + nbuf, buf);
    acc = warp_sum(acc);
    if (lane == 0) P.out[(long)t * P.H + c] = __float2bfloat16_rn(acc);
  }
}

// ---- tensor-core FC2 of the layer kernel ------------------------------------
// Eight 8x8 bf16 matrices' worth of rows: ldmatrix with one row address per lane.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
// D (16x8, f32) += A (16x16, bf16, row-major) * B (16x8, bf16, column-major).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Rows [0, n) of the activations (bf16, written by other CTAs or the previous
// kernel) into shared memory, read through L2.
__device__ __forceinline__ void stage_act(const GemvParams& P, int n, uint4* act_s, int ld = 0) {
  const uint4* act = reinterpret_cast<const uint4*>(P.act);
  const int nch = P.I >> 3;
  if (ld == 0 || ld == nch) {
    const long m = (long)n * nch;
    for (long x = threadIdx.x; x < m; x += blockDim.x) act_s[x] = __ldcg(act + x);
  } else {   // rows ld pieces apart
    for (long x = threadIdx.x; x < (long)n * nch; x += blockDim.x) {
      const long r = x / nch;
      act_s[r * ld + (x - r * nch)] = __ldcg(act + x);
    }
  }
}

template <int TT>
__global__ void __launch_bounds__(kGemvThreads, 2) fc1_gemv_kernel(const GemvParams P) {
  extern __shared__ float4 xs[];   // [T][H / 4]: the batch's token rows as float32
  __shared__ int32_t l_idx[kMaxSlots], l_ids[kMaxSlots];
  __shared__ int32_t l_cnt[kRouteExperts], l_off[kRouteExperts + 1], l_run[kRouteExperts];
  __shared__ int32_t a_e[kMaxSlots];
  __shared__ int a_n;
  const bool local = P.logits != nullptr;
  stage_f32(P.hidden, (long)P.T * P.H, xs);
  const int32_t* counts = P.counts;
  const int32_t* offsets = P.offsets;
  const int32_t* sorted_ids = P.sorted_ids;
  if (local) {
    gate::route_block(P.logits, P.T, P.E, P.k, l_idx, l_cnt, l_off, l_ids, l_run);
    counts = l_cnt;
    offsets = l_off;
    sorted_ids = l_ids;
  } else {
    pdl_wait();      // the routing comes from the previous kernel
    pdl_trigger();
  }
  active_experts(counts, P.E, a_e, &a_n);
  __syncthreads();
  const long U = (long)a_n * P.I;   // a contiguous range of units per CTA
  fc1_units<TT>(P, xs, a_e, counts, offsets, sorted_ids, U * blockIdx.x / gridDim.x,
                U * (blockIdx.x + 1) / gridDim.x);
  // FC2 reads the routing kernel's outputs: release it only once they exist. One
  // warp waits, after its units, so that no warp stalls on the routing kernel.
  if (local && threadIdx.x < 32) {
    pdl_wait();
    pdl_trigger();
  }
}

// FC2 with the combine, one CTA per SM over a contiguous range of units.
__global__ void __launch_bounds__(kFc2Threads, 1) fc2_gemv_kernel(const GemvParams P) {
  extern __shared__ uint8_t fc2_raw[];
  __shared__ int32_t s_pos[kMaxSlots], s_e[kMaxSlots];
  __shared__ float s_w[kMaxSlots];
  __shared__ int32_t s_off[MOE_MAX_EXPERTS + 1];
  const int tid = threadIdx.x, warp = tid >> 5;
  const int S = P.T * P.k;
  const Fc2Layout L = fc2_layout(P.T, P.k, P.H, P.I);
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(fc2_raw) + 127) & ~uintptr_t(127));
  uint4* act_s = reinterpret_cast<uint4*>(base + L.ring);               // [n][I / 8]
  uint4* buf = reinterpret_cast<uint4*>(base + (size_t)warp * L.slot);   // this warp's rows [k][I / 8]
  // The routing outputs were written two launches back: complete once FC1 has
  // released this kernel. Slot q = t * k + j sits at sorted row s_pos[q] (-1:
  // dropped), in the range of expert s_e[q], with routing weight s_w[q]. The
  // workspace holds S entries of reverse and sorted_w; those past offsets[E] are
  // read but not used.
  int rv = -1;
  float wv = 0.0f;
  if (tid < S) {
    rv = __ldg(P.reverse + tid);
    wv = __ldg(P.sorted_w + tid);
  }
  for (int e = tid; e <= P.E; e += kFc2Threads) s_off[e] = __ldg(P.offsets + e);
  for (int q = tid; q < S; q += kFc2Threads) s_pos[q] = s_e[q] = -1;
  __syncthreads();
  const int n = min(s_off[P.E], S);
  if (tid < n && rv >= 0 && rv < S) {
    int lo = 0, hi = P.E - 1;   // the expert whose range [offsets[e], offsets[e + 1]) holds row tid
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_off[mid] <= tid) lo = mid; else hi = mid - 1;
    }
    s_pos[rv] = tid;
    s_e[rv] = lo;
    s_w[rv] = wv;
  }
  __syncthreads();
  const long U = (long)P.H * P.T;   // unit u = c * T + t
  const long u0 = U * blockIdx.x / gridDim.x, u1 = U * (blockIdx.x + 1) / gridDim.x;
  const int nloc = (int)(u1 - u0);
  if (warp < L.buffers && warp < nloc) fc2_fetch(P, s_e, u0 + warp, buf);   // before FC1 ends
  pdl_wait();        // FC1's activations
  pdl_trigger();
  stage_act(P, n, act_s);
  __syncthreads();
  if (warp < L.buffers) fc2_units(P, s_pos, s_e, s_w, act_s, buf, u0, nloc, L.buffers);
}

// ---- the pipelined one-kernel decode FFN ------------------------------------
// FC1 warps (the first kPipeFc1Warps) stream FC1 column pairs (units of two
// columns: both gate rows and both up rows in flight together) over the flat
// range [0, a_n * I / 2), each warp's first pair fixed and the rest taken in
// order from a counter all CTAs share (every CTA finishes expert a's pairs at
// about the same time, experts in order), and count each finished pair on its
// expert's counter (done[a] += 2, zeroed by the routing kernel launched just
// before; the activations are stored first, the add releases them). FC1 is bound
// by the bytes each SM keeps in flight, which registers hold: 10 warps of 168
// registers with 16 KB each. The other warps run FC2 behind them:
// the CTA owns output columns [c0, c1); for each active expert in turn they wait
// (bounded) until its I units are counted, stage its activation rows, and take
// the dot products of their columns' w2 rows (asked of L2 at the start) with
// them into shared memory, so FC2 of expert a overlaps FC1 of the later experts
// and only the last expert's FC2 and the combine follow the FC1 stream. One
// warp keeps pace: its products are mma.sync tiles (16 w2 rows x the expert's
// activation rows) over rows that bulk copies (one per row, one expert ahead)
// bring into shared memory. The combine: out[t][c] = sum
// over j of w_j * (row c of w2[e_j] . act_j), float32 in j order, rounded once.
constexpr int kPipeThreads = 384;   // 12 warps of up to 168 registers: FC1 warps keep 16 KB in flight
constexpr int kPipeFc2Warps = 2;    // each takes every other expert
constexpr int kPipeFc1Warps = kPipeThreads / 32 - kPipeFc2Warps;
constexpr int kPipeFc2Threads = kPipeFc2Warps * 32;
constexpr int kPipeCols = 32;   // most output columns per CTA
static_assert(kMaxSlots + 1 <= kDecodeSyncWords, "one counter per active expert, one of FC1 units taken");

// bytes (a multiple of 16) global -> shared by the TMA engine, completing on bar.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Shared memory of decode_pipe_kernel: token rows [T][H] (float32), then per FC2
// warp its activation rows [TT][I + 8] and nb buffers of the CTA's w2 rows of one
// expert [ceil(H / G)][I + 8] (bf16, rows padded by 16 bytes). nb = 1: the rows of
// the warp's next expert are requested once the current one is multiplied (two
// buffers, the next two experts' rows in flight, measured 0.5% slower at T = 1:
// their opening requests compete with FC1's first column pairs).
constexpr size_t kPipeSmemMax = 216 * 1024;   // + the kernel's ~10 KB of static shared memory <= 227 KB
__host__ __device__ inline size_t pipe_smem_nb(int T, int TT, int H, int I, int G, int nb) {
  return (size_t)T * H * 4 + (size_t)kPipeFc2Warps * ((size_t)TT + (size_t)nb * ((H + G - 1) / G)) * (I + 8) * 2;
}
__host__ __device__ inline int pipe_buffers(int, int, int, int, int) { return 1; }
__host__ __device__ inline size_t pipe_smem(int T, int TT, int H, int I, int G) {
  return pipe_smem_nb(T, TT, H, I, G, pipe_buffers(T, TT, H, I, G));
}

template <int TT>
__global__ void __launch_bounds__(kPipeThreads, 1) decode_pipe_kernel(const GemvParams P) {
  extern __shared__ float4 pipe_raw[];
  __shared__ int32_t l_idx[kMaxSlots], l_ids[kMaxSlots];
  __shared__ int32_t l_cnt[kRouteExperts], l_off[kRouteExperts + 1], l_run[kRouteExperts];
  __shared__ int32_t a_e[kMaxSlots];
  __shared__ int32_t s_pos[kMaxSlots];
  __shared__ float s_w[kMaxSlots];
  __shared__ float part[kMaxSlots * kPipeCols];   // [sorted slot][column - c0]
  __shared__ int a_n, abort_flag;
  __shared__ __align__(8) uint64_t wbar[kPipeFc2Warps * 2];   // each row buffer's copies
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float4* xs = pipe_raw;                                                   // [T][H / 4]
  uint4* acts = reinterpret_cast<uint4*>(pipe_raw + (long)P.T * P.H / 4);  // [W][TT][I / 8 + 1]
  uint4* wbuf = acts + (long)kPipeFc2Warps * TT * ((P.I >> 3) + 1);         // [W][nb][ceil(H / G)][I / 8 + 1]
  // the token rows by the warps that do not route (their loads overlap the logits')
  for (long c = tid - 64; c >= 0 && c < (long)P.T * P.H / 8; c += kPipeThreads - 64) {
    const uint4 v = P.hidden[c];
    xs[2 * c] = make_float4(bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y));
    xs[2 * c + 1] = make_float4(bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w));
  }
  gate::route_block(P.logits, P.T, P.E, P.k, l_idx, l_cnt, l_off, l_ids, l_run, s_pos, a_e, &a_n);
  if (P.T != 1) active_experts(l_cnt, P.E, a_e, &a_n);   // one token: listed by route_block
  if (tid == 0) abort_flag = 0;
  __syncthreads();
  const int G = gridDim.x, b = blockIdx.x;
  const int I = P.I, nch = I >> 3;
  int32_t* done = P.sync;   // [kMaxSlots]: FC1 units finished per active expert
  if (warp < kPipeFc1Warps) {
    // every warp's first unit is b + G * warp; later units are taken in order from a
    // counter shared by all CTAs (the next one requested while the current one
    // streams), so CTAs that run faster take more of them and the experts still
    // complete in order
    const uint64_t pol = evict_first_policy();
    const int Ih = I >> 1;   // column pairs per expert (I is even here)
    const long U1 = (long)a_n * Ih, nfirst = (long)kPipeFc1Warps * G;
    int32_t* work = P.sync + kMaxSlots;
    long u = b + (long)G * warp;
    int next = 0;
    for (bool first = true; u < U1; first = false) {
      if (!first && lane == 0) next = atomicAdd(work, 1);
      const int a = (int)(u / Ih), i = 2 * (int)(u - (long)a * Ih);
      fc1_pair<TT>(P, xs, a_e[a], l_cnt, l_off, l_ids, i, pol);
      if (first) {   // the routing kernel (complete from here on) zeroed the counters
        pdl_wait();
        if (lane == 0) next = atomicAdd(work, 1);
      }
      if (lane == 0)   // the activations (this lane's store) before their count
        asm volatile("red.release.gpu.global.add.s32 [%0], 2;" ::"l"(done + a) : "memory");
      u = nfirst + __shfl_sync(0xffffffffu, next, 0);
    }
    return;   // no barrier of the whole CTA follows
  }
  // ---- the FC2 warps: warp f takes the active experts a = f, f + kPipeFc2Warps, ...
  // with its own activation rows and nb row buffers
  const int f = warp - kPipeFc1Warps, ftid = tid - kPipeFc1Warps * 32;
  const int S = P.T * P.k;
  const int c0 = (int)((long)P.H * b / G), c1 = (int)((long)P.H * (b + 1) / G), nc = c1 - c0;
  const int ld = nch + 1;   // row stride in shared memory, 16-byte pieces (ldmatrix: distinct banks)
  const long wstride = (long)((P.H + G - 1) / G) * ld;   // one buffer of rows
  const int nb = pipe_buffers(P.T, TT, P.H, P.I, G);     // row buffers per FC2 warp
  uint4* my_acts = acts + (long)f * TT * ld;
  uint4* my_buf = wbuf + (long)f * nb * wstride;
  uint64_t* my_bar = wbar + f * 2;
  if (lane == 0) {
    for (int z = 0; z < nb; ++z) ptx::mbar_init(ptx::smem_u32(&my_bar[z]), 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  // this CTA's w2 rows of expert a (rows c0 .. c1 - 1) into buffer (a / W) % nb: one bulk
  // copy per row by lane 0 (rows padded in shared memory), completing on its mbarrier;
  // the n-th use of a buffer completes phase n % 2
  constexpr int W = kPipeFc2Warps;
  auto slot = [&](int a) { return (a / W) % nb; };
  auto phase = [&](int a) { return (uint32_t)((a / W / nb) & 1); };
  int fetched = f;   // this warp's experts whose rows were requested: f, f + W, ... < fetched
  auto fetch = [&](int a) {
    if (a >= a_n) return;
    fetched = a + W;
    if (lane == 0) {
      const uint32_t bar = ptx::smem_u32(&my_bar[slot(a)]);
      ptx::mbar_arrive_expect_tx(bar, (uint32_t)nc * I * 2);
      const char* src = reinterpret_cast<const char*>(P.w2 + ((long)a_e[a] * P.H + c0) * nch);
      const uint32_t dst = ptx::smem_u32(my_buf + slot(a) * wstride);
      for (int r = 0; r < nc; ++r) bulk_load(dst + (uint32_t)(r * ld * 16), src + (long)r * I * 2, I * 2, bar);
    }
  };
  for (int z = 0; z < nb; ++z) fetch(f + z * W);
  pdl_wait();   // the routing kernel's weights
  for (int q = ftid; q < S; q += kPipeFc2Threads) s_w[q] = __ldg(P.sorted_w + s_pos[q]);
  const uint4* act4 = reinterpret_cast<const uint4*>(P.act);
  const int ksteps = I >> 4;   // 16 bf16 per mma step
  bool aborted = false;
  int a = f;
  for (; a < a_n; a += W) {
    const int e = a_e[a], cnt = min(l_cnt[e], TT), p0 = l_off[e];
    bool ready = true;
    if (lane == 0) {
      const uint64_t t0 = ptx::globaltimer();
      while (ld_acquire(done + a) < I) {
        if (ptx::globaltimer() - t0 > P.wait_ns || abort_flag) {
          ready = false;
          break;
        }
        __nanosleep(32);
      }
    }
    if (!__shfl_sync(0xffffffffu, ready, 0)) {
      aborted = true;
      break;
    }
    for (int r = 0; r < cnt; ++r)   // the expert's activation rows (bf16)
      for (int pc = lane; pc < nch; pc += 32) my_acts[r * ld + pc] = __ldcg(act4 + (long)(p0 + r) * nch + pc);
    const bool rows = ptx::mbar_wait(ptx::smem_u32(&my_bar[slot(a)]), phase(a), &abort_flag, P.wait_ns);
    if (!__all_sync(0xffffffffu, rows)) {   // the rows (every lane leaves together)
      aborted = true;
      break;
    }
    __syncwarp();
    // D (16 columns x 8 slots) = A (16 w2 rows x I) * B (I x the expert's activation rows), on the
    // tensor cores; rows past nc / cnt repeat a valid row and their products are not kept
    const uint32_t wb = ptx::smem_u32(my_buf + slot(a) * wstride), ab = ptx::smem_u32(my_acts);
    const uint32_t brow = ab + (uint32_t)(min(lane & 7, cnt - 1) * ld * 16) + (uint32_t)(((lane >> 3) & 1) * 16);
    for (int m0 = 0; m0 < nc; m0 += 16) {
      const uint32_t arow = wb + (uint32_t)(min(m0 + (lane & 15), nc - 1) * ld * 16) + (uint32_t)((lane >> 4) * 16);
      // four accumulators (steps st mod 4), the four steps' fragments loaded before their mma
      float d[4][4];
#pragma unroll
      for (int z = 0; z < 4; ++z) d[z][0] = d[z][1] = d[z][2] = d[z][3] = 0.0f;
      int st = 0;
      for (; st + 4 <= ksteps; st += 4) {
        uint32_t fa[4][4], fb[4][2];
#pragma unroll
        for (int z = 0; z < 4; ++z) {
          ldsm_x4(arow + (st + z) * 32, fa[z]);
          ldsm_x2(brow + (st + z) * 32, fb[z][0], fb[z][1]);
        }
#pragma unroll
        for (int z = 0; z < 4; ++z) mma_16816(d[z], fa[z], fb[z][0], fb[z][1]);
      }
#pragma unroll
      for (int z = 0; z < 3; ++z)   // the last ksteps % 4 steps
        if (st + z < ksteps) {
          uint32_t fa[4], b0, b1;
          ldsm_x4(arow + (st + z) * 32, fa);
          ldsm_x2(brow + (st + z) * 32, b0, b1);
          mma_16816(d[z], fa, b0, b1);
        }
      // lane l holds D[l / 4 (+ 8)][2 (l % 4) + (0, 1)]
      const int m = m0 + (lane >> 2), n = 2 * (lane & 3);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (m + 8 * h < nc && n + q < cnt)
            part[(p0 + n + q) * kPipeCols + m + 8 * h] =
                (d[0][2 * h + q] + d[1][2 * h + q]) + (d[2][2 * h + q] + d[3][2 * h + q]);
    }
    __syncwarp();   // this warp's activation rows and buffer are free again
    if (a + nb * W < a_n) {   // a copy will rewrite the buffer: order the reads above before it
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      fetch(a + nb * W);
    }
  }
  if (aborted) {
    if (lane == 0) {   // no copy in flight when the CTA leaves: experts a, a + W, .. < fetched
      abort_flag = 1;
      if (P.status) atomicOr(P.status, MOE_STATUS_TIMEOUT);
      const uint64_t t0 = ptx::globaltimer();
      for (int x = a; x < fetched; x += W)
        while (!ptx::mbar_test_wait(ptx::smem_u32(&my_bar[slot(x)]), phase(x)) && ptx::globaltimer() - t0 < P.wait_ns) {
        }
    }
    __syncwarp();
  }
  ptx::named_bar_sync(1, kPipeFc2Threads);   // every FC2 warp's products (and abort_flag) are in
  if (!abort_flag) {
    for (int x = ftid; x < P.T * nc; x += kPipeFc2Threads) {
      const int t = x / nc, cc = x - t * nc;
      float acc = 0.0f;
      for (int j = 0; j < P.k; ++j) {
        const int q = t * P.k + j;
        acc = fmaf(s_w[q], part[s_pos[q] * kPipeCols + cc], acc);
      }
      P.out[(long)t * P.H + c0 + cc] = __float2bfloat16_rn(acc);
    }
  }
  pdl_trigger();   // only now may the next kernel (which zeroes the counters again) start
}

template <typename K>
int launch_one(K kernel, int grid, int threads, size_t smem, cudaStream_t s, const GemvParams& p,
               const char* name) {
  if (int rc = ensure_smem_limit(kernel, smem, name)) return rc;
  ProfScope ps(name, s);
  const cudaError_t e = launch_pdl(kernel, grid, threads, smem, s, p);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", name, cudaGetErrorString(e));
  return check_launch(name);
}

template <int TT>
int run_gemv(const FfnArgs& a, cudaStream_t s) {
  const bool local = a.logits && a.E <= kRouteExperts;
  const GemvParams p{static_cast<const uint4*>(a.hidden), static_cast<const uint4*>(a.w13),
                     static_cast<const uint4*>(a.w2), a.counts, a.offsets, a.sorted_ids, a.sorted_w, a.reverse,
                     static_cast<__nv_bfloat16*>(a.act), static_cast<__nv_bfloat16*>(a.out),
                     local ? a.logits : nullptr, a.sync, a.status, wait_limit_ns(), a.T, a.H, a.I, a.E, a.k};
  const int G = num_sms() - 1;
  if (local && a.sync && G >= 1 && (a.H + G - 1) / G <= kPipeCols && (a.H * 2) % 128 == 0 && (a.I * 2) % 128 == 0 &&
      pipe_smem(a.T, TT, a.H, a.I, G) <= kPipeSmemMax)
    return launch_one(decode_pipe_kernel<TT>, G, kPipeThreads, pipe_smem(a.T, TT, a.H, a.I, G), s, p,
                      "ffn_decode_layer");
  const int rc = launch_one(fc1_gemv_kernel<TT>, 2 * num_sms(), kGemvThreads, (size_t)a.T * a.H * 4, s, p,
                            "ffn_fc1_gemv");
  if (rc) return rc;
  return launch_one(fc2_gemv_kernel, num_sms(), kFc2Threads, fc2_layout(a.T, a.k, a.H, a.I).total, s, p,
                    "ffn_fc2_gemv");
}

}  // namespace

bool ffn_gemv_applies(int dtype, int T, int H, int I, int k) {
  return ffn_uses_tensor_cores(dtype, H, I) && T >= 1 && T <= kGemvMaxTokens &&
         (size_t)T * H * 4 <= kGemvSmemMax && fc2_layout(T, k, H, I).buffers >= 2;
}

int launch_ffn_gemv(const FfnArgs& a, cudaStream_t s) {
  if (a.T == 1) return run_gemv<1>(a, s);
  return run_gemv<2>(a, s);
}

}  // namespace moe
