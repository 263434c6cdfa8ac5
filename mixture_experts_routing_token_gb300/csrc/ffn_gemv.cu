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
// kernel (decode_layer_kernel): every CTA routes the batch itself; before its
// FC1 units it requests the weight rows of its FC2 units (they do not depend on
// FC1: the first eight units into the buffers of eight warps, the rest into L2),
// so that DRAM streams FC2's weights together with FC1's; it then meets the other
// CTAs at a grid barrier (a counter that the routing kernel just before it
// zeroed, polled with a time limit) and runs FC2 on the tensor cores (mma.sync
// on pairs of units, the later units copied into the buffers as the first ones
// are done). Its grid leaves one SM to the routing kernel it overlaps, so that
// every CTA of the barrier is resident. Elsewhere (routing given by the caller,
// or E > 64) FC1 and FC2 are two kernels, FC2 on the CUDA cores.
#include "common.cuh"
#include "gating_device.cuh"
#include "sm100_ptx.cuh"   // smem_u32, globaltimer

namespace moe {
namespace {

constexpr int kGemvThreads = 256;                        // FC1 kernel: two CTAs per SM
constexpr int kLayerThreads = 512;                       // layer kernel: one CTA per SM
constexpr int kPieces = 8;                               // FC1: 16-byte pieces per lane per row in flight
constexpr int kMaxSlots = kGemvMaxTokens * MOE_MAX_TOPK;
constexpr int kRouteExperts = 64;                        // in-CTA routing (gate::route_block): E <= 64
constexpr int kFc2Buffers = 8;                           // FC2 warps with a row buffer each, at most
constexpr int kFc2Threads = kFc2Buffers * 32;            // FC2 kernel
constexpr size_t kFc2SmemMax = 200 * 1024;               // FC2 kernel: buffers + activation rows
constexpr size_t kLayerSmemMax = 216 * 1024;             // layer kernel: buffers + activations + token rows
constexpr int kMaxPairs = 4;                             // layer kernel: FC2 unit pairs per round (four warps each)

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
  int32_t* sync;         // layer kernel: grid barrier counter, zero at launch
  int32_t* status;
  uint64_t wait_ns;      // limit of the grid barrier wait (moe_set_wait_limit_ns)
  int T, H, I, E, k;
};

// Shared memory of FC2: one buffer (the k weight rows of one unit) per FC2 warp,
// the batch's activation rows (bf16), then (layer kernel) the token rows (float32).
struct Fc2Layout {
  int buffers;
  size_t slot, ring, act, x, total;
};

__host__ __device__ inline Fc2Layout fc2_layout(int T, int k, int H, int I, bool with_x) {
  Fc2Layout L;
  // the layer kernel's rows are one 16-byte piece longer: a row of I bf16 is a
  // multiple of 128 bytes, so without it the eight rows an ldmatrix reads would
  // all start on the same banks
  const size_t row = (size_t)I * 2 + (with_x ? 16 : 0);
  L.slot = ((size_t)k * row + 127) & ~(size_t)127;
  L.act = ((size_t)T * k * row + 127) & ~(size_t)127;
  L.x = with_x ? (size_t)T * H * 4 : 0;
  const size_t cap = with_x ? kLayerSmemMax : kFc2SmemMax;
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

// FC1 units u0, u0 + ustride, ... < u1 (unit u = a * I + i), taken in turn by the
// block's warps.
// TT: most tokens an expert can have (the batch size bound).
template <int TT, int PIECES = kPieces>
__device__ __forceinline__ void fc1_units(const GemvParams& P, const float4* xs, const int32_t* a_e,
                                          const int32_t* counts, const int32_t* offsets,
                                          const int32_t* sorted_ids, long u0, long u1, long ustride = 1) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int nch = P.H >> 3;
  const uint64_t pol = evict_first_policy();
  for (long u = u0 + warp * ustride; u < u1; u += nwarps * ustride) {
    const int a = (int)(u / P.I), i = (int)(u - (long)a * P.I);
    const int e = a_e[a];
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
}

// Row j of FC2 unit u = c * T + t: row c of w2[s_e[t * k + j]] (a valid slot).
__device__ __forceinline__ const uint4* fc2_row(const GemvParams& P, const int32_t* s_e, long u, int j) {
  const int c = (int)(u / P.T), t = (int)(u - (long)c * P.T);
  return P.w2 + ((long)s_e[t * P.k + j] * P.H + c) * (P.I >> 3);
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

// Steps [s0, s1) of K of the FC2 products of units ua and ub = ua + T (the same
// token t), whose k weight rows sit in the shared buffers at sa and sb (rows ld
// pieces apart; the activation rows in act likewise), for experts jb .. jb + 7,
// by one warp on the tensor cores: A = rows j of unit ua then of unit ub (16 x K),
// B = the token's activation rows of the same eight experts (K x 8); the products
// wanted are D's diagonal, D[8h + j][j] = row j of unit h . act row of expert j.
// Lane 4j + j/2 returns them: [0] for unit ua, [1] for unit ub (expert jb + j).
__device__ __forceinline__ float2 fc2_pair_mma(const GemvParams& P, const int32_t* s_pos, uint32_t sa,
                                               uint32_t sb, uint32_t act, int ld, int t, int jb, int s0,
                                               int s1) {
  const int lane = threadIdx.x & 31;
  // A: lane l gives row (l & 15) (rows 8..15 from unit ub) at k half (l >> 4)
  const int ja = min(jb + (lane & 7), P.k - 1);   // rows past k: any valid row, unused
  const uint32_t arow = ((lane & 8) ? sb : sa) + (uint32_t)(ja * ld * 16) + (uint32_t)((lane >> 4) * 16);
  // B: lane l (0..15) gives the activation row of expert jb + (l & 7) at k half (l >> 3) & 1
  const uint32_t brow = act + (uint32_t)(s_pos[t * P.k + ja] * ld * 16) + (uint32_t)(((lane >> 3) & 1) * 16);
  float d0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, d1[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // even / odd steps
  for (int st = s0; st < s1; st += 2) {
    uint32_t a[4], b0, b1;
    ldsm_x4(arow + st * 32, a);
    ldsm_x2(brow + st * 32, b0, b1);
    mma_16816(d0, a, b0, b1);
    if (st + 1 < s1) {
      ldsm_x4(arow + (st + 1) * 32, a);
      ldsm_x2(brow + (st + 1) * 32, b0, b1);
      mma_16816(d1, a, b0, b1);
    }
  }
  // D[8h + j][j] sits in lane 4j + j/2, register 2h + (j & 1); in the other lanes: unused
  const bool odd = (lane >> 2) & 1;   // j & 1 for the lane holding expert j = lane / 4
  return make_float2(odd ? d0[1] + d1[1] : d0[0] + d1[0], odd ? d0[3] + d1[3] : d0[2] + d1[2]);
}

// Ask L2 for the 128-byte line holding p.
__device__ __forceinline__ void prefetch_line_l2(const void* p) {
  asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p) : "memory");
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
  const Fc2Layout L = fc2_layout(P.T, P.k, P.H, P.I, false);
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

// Bounded grid barrier (thread 0 of each CTA, between __syncthreads): count this
// CTA in and wait until all `nblocks` have arrived. False when the limit ran out.
__device__ __forceinline__ bool grid_barrier(int32_t* ctr, int nblocks, uint64_t limit_ns) {
  __threadfence();   // this CTA's activations before its arrival
  atomicAdd(ctr, 1);
  const uint64_t t0 = ptx::globaltimer();
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= nblocks) return true;
    if (ptx::globaltimer() - t0 > limit_ns) return false;
    __nanosleep(64);
  }
}

// The whole FFN of a batch of at most TT tokens inside the layer call (logits
// given, E <= 64), one CTA on every SM but one. See the file comment.
template <int TT>
__global__ void __launch_bounds__(kLayerThreads, 1) decode_layer_kernel(const GemvParams P) {
  extern __shared__ uint8_t lay_raw[];
  __shared__ int32_t l_idx[kMaxSlots], l_ids[kMaxSlots];
  __shared__ int32_t l_cnt[kRouteExperts], l_off[kRouteExperts + 1], l_run[kRouteExperts];
  __shared__ int32_t a_e[kMaxSlots];
  __shared__ int32_t s_pos[kMaxSlots];
  __shared__ float s_w[kMaxSlots];
  __shared__ float part[kMaxPairs * 4 * 16];
  __shared__ int a_n, go;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = P.T * P.k;
  const Fc2Layout L = fc2_layout(P.T, P.k, P.H, P.I, true);
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(lay_raw) + 127) & ~uintptr_t(127));
  uint4* act_s = reinterpret_cast<uint4*>(base + L.ring);
  float4* xs = reinterpret_cast<float4*>(base + L.ring + L.act);
  uint4* buf = reinterpret_cast<uint4*>(base + (size_t)warp * L.slot);
  // the token rows by the warps that do not route (their loads overlap the logits')
  for (long c = tid - 64; c >= 0 && c < (long)P.T * P.H / 8; c += kLayerThreads - 64) {
    const uint4 v = P.hidden[c];
    xs[2 * c] = make_float4(bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y));
    xs[2 * c + 1] = make_float4(bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w));
  }
  gate::route_block(P.logits, P.T, P.E, P.k, l_idx, l_cnt, l_off, l_ids, l_run, s_pos);
  active_experts(l_cnt, P.E, a_e, &a_n);
  __syncthreads();
  const int G = gridDim.x;
  const long U2 = (long)P.H * P.T;
  const long u0 = U2 * blockIdx.x / G, u1 = U2 * (blockIdx.x + 1) / G;
  const int nloc = (int)(u1 - u0);
  // ---- FC2 weight rows (they do not depend on FC1), requested now so that DRAM
  // streams them together with FC1's: the first unit of each FC2 warp into its
  // buffer, the rows of the CTA's later units into L2
  const int ld = (P.I >> 3) + 1;   // row stride of the buffers and activation rows, 16-byte pieces
  if (warp < L.buffers && warp < nloc) fc2_fetch(P, l_idx, u0 + warp, buf, ld);
  {
    const int lpr = P.I / 64;   // 128-byte lines per row
    const long nl = (long)max(nloc - L.buffers, 0) * P.k * lpr;
    for (long x = tid; x < nl; x += kLayerThreads) {
      const long r = x / lpr;
      const int i = L.buffers + (int)(r / P.k), j = (int)(r - (long)(r / P.k) * P.k);
      prefetch_line_l2(reinterpret_cast<const char*>(fc2_row(P, l_idx, u0 + i, j)) + (x - r * lpr) * 128);
    }
  }
  // ---- FC1
  const long U1 = (long)a_n * P.I;
  fc1_units<TT>(P, xs, a_e, l_cnt, l_off, l_ids, blockIdx.x, U1, G);   // units b, b + G, ... of CTA b
  // ---- the routing kernel is complete (barrier counter zeroed, routing weights
  // written); then every CTA's activations
  pdl_wait();
  pdl_trigger();
  if (tid < S) s_w[tid] = __ldg(P.sorted_w + s_pos[tid]);
  cp_async_wait_all();   // this warp's buffered rows land before the CTA may leave
  __syncthreads();
  if (tid == 0) {
    go = grid_barrier(P.sync, G, P.wait_ns);
    if (!go && P.status) atomicOr(P.status, MOE_STATUS_TIMEOUT);
  }
  __syncthreads();
  if (!go) return;
  stage_act(P, S, act_s, ld);
  __syncthreads();
  // ---- FC2 on the tensor cores, in rounds of L.buffers units (unit r0 + b in
  // buffer b): the pairs of units (b, b + T) of one token, each pair by four warps
  // (a quarter of K each), which own the pair's two buffers: after a round they
  // refill them with the pair's units of the next round (rows asked of L2 at the
  // start) while the other pairs compute.
  const int B = L.buffers, T2 = 2 * P.T;
  const int npairs = (B + T2 - 1) / T2 * P.T;
  const int pr = warp >> 2, qw = warp & 3;       // pair of this warp, its quarter
  const int ksteps = (P.I >> 3) >> 1;            // 16 bf16 per step
  if (pr < npairs && pr < kMaxPairs) {
    const int b0 = pr / P.T * T2 + pr % P.T, b1 = b0 + P.T;
    uint4* buf0 = reinterpret_cast<uint4*>(base + (size_t)b0 * L.slot);
    uint4* buf1 = reinterpret_cast<uint4*>(base + (size_t)b1 * L.slot);
    const int s0 = ksteps * qw / 4, s1 = ksteps * (qw + 1) / 4;
    float* dg = part + pr * 4 * 16;              // [quarter][h * 8 + j]
    for (int r0 = 0; r0 < nloc && b0 < B; r0 += B) {
      const int nr = min(B, nloc - r0);
      if (b0 >= nr) break;
      const bool two = b1 < nr;
      const long ua = u0 + r0 + b0;
      const int t = (int)(ua % P.T);
      if (r0 > 0) {   // rows qw, qw + 4, ... of both units
        fc2_fetch(P, l_idx, ua, buf0, ld, qw, 4);
        if (two) fc2_fetch(P, l_idx, ua + P.T, buf1, ld, qw, 4);
        cp_async_wait_all();
        ptx::named_bar_sync(1 + pr, 128);
      }
      float acc0 = 0.0f, acc1 = 0.0f;
      for (int jb = 0; jb < P.k; jb += 8) {
        const float2 d = fc2_pair_mma(P, s_pos, ptx::smem_u32(buf0), ptx::smem_u32(two ? buf1 : buf0),
                                      ptx::smem_u32(act_s), ld, t, jb, s0, s1);
        const int j = lane >> 2;
        if ((lane & 3) == (j >> 1)) {   // lane 4j + j/2 holds expert j's products
          dg[qw * 16 + j] = d.x;
          dg[qw * 16 + 8 + j] = d.y;
        }
        ptx::named_bar_sync(1 + pr, 128);
        if (qw == 0 && lane == 0)
          for (int jj = 0; jj < 8 && jb + jj < P.k; ++jj) {
            const float w = s_w[t * P.k + jb + jj];
            acc0 = fmaf(w, (dg[jj] + dg[16 + jj]) + (dg[32 + jj] + dg[48 + jj]), acc0);
            acc1 = fmaf(w, (dg[8 + jj] + dg[24 + jj]) + (dg[40 + jj] + dg[56 + jj]), acc1);
          }
        ptx::named_bar_sync(1 + pr, 128);   // dg and the buffers are free again
      }
      if (qw == 0 && lane == 0) {
        const int ca = (int)(ua / P.T);
        P.out[(long)t * P.H + ca] = __float2bfloat16_rn(acc0);
        if (two) P.out[(long)t * P.H + ca + 1] = __float2bfloat16_rn(acc1);
      }
    }
  }
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
  const Fc2Layout LL = fc2_layout(a.T, a.k, a.H, a.I, true);
  const int G = num_sms() - 1;
  if (local && a.sync && LL.buffers >= 2 && G >= 1)
    return launch_one(decode_layer_kernel<TT>, G, kLayerThreads, LL.total, s, p, "ffn_decode_layer");
  const int rc = launch_one(fc1_gemv_kernel<TT>, 2 * num_sms(), kGemvThreads, (size_t)a.T * a.H * 4, s, p,
                            "ffn_fc1_gemv");
  if (rc) return rc;
  return launch_one(fc2_gemv_kernel, num_sms(), kFc2Threads, fc2_layout(a.T, a.k, a.H, a.I, false).total, s, p,
                    "ffn_fc2_gemv");
}

}  // namespace

bool ffn_gemv_applies(int dtype, int T, int H, int I, int k) {
  return ffn_uses_tensor_cores(dtype, H, I) && T >= 1 && T <= kGemvMaxTokens &&
         (size_t)T * H * 4 <= kGemvSmemMax && fc2_layout(T, k, H, I, false).buffers >= 2;
}

int launch_ffn_gemv(const FfnArgs& a, cudaStream_t s) {
  if (a.T == 1) return run_gemv<1>(a, s);
  return run_gemv<2>(a, s);
}

}  // namespace moe
