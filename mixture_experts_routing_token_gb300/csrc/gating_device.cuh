// Device-side gating pieces shared by the gating kernel (routing.cu) and the
// fused small-batch routing kernel (align.cu).
// mlc-llm moe_misc.py, gating_topk / gating_softmax_topk.
#pragma once

#include <float.h>

#include <type_traits>

#include "common.cuh"

namespace moe {
namespace gate {

constexpr int kNone = 0x7fffffff;   // "no candidate" index
constexpr int kRegSel = 8;          // up to this k, one thread per token keeps the selected logits in registers

// Logits are float32 or bf16; bf16 values are widened to float32 exactly, so
// everything after the load is the float32 computation on the widened row.
__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float load_logit(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_logit(const __nv_bfloat16* p) {
  return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p)) << 16);
}
// 8 consecutive bf16 logits from a 16-byte aligned address
__device__ __forceinline__ void load8_bf16(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
  x[0] = lo_bf16(q.x); x[1] = hi_bf16(q.x); x[2] = lo_bf16(q.y); x[3] = hi_bf16(q.y);
  x[4] = lo_bf16(q.z); x[5] = hi_bf16(q.z); x[6] = lo_bf16(q.w); x[7] = hi_bf16(q.w);
}

// (value, index) order of the page's top-k: larger value first; equal values
// keep the lower expert index first. kNone loses to everything.
__device__ __forceinline__ bool better(float av, int ai, float bv, int bi) {
  if (ai == kNone) return false;
  if (bi == kNone) return true;
  return av > bv || (av == bv && ai < bi);
}

// Lanes of this thread's group of L (L a power of two, groups aligned in the warp).
template <int L>
__device__ __forceinline__ unsigned group_mask() {
  if constexpr (L == 32) {
    return 0xffffffffu;
  } else {
    const unsigned lane = threadIdx.x & 31;
    return ((1u << L) - 1u) << (lane & ~(unsigned)(L - 1));
  }
}

// exp(a - b) with the rounding error of the float subtraction folded back in
// (a - b = s + err exactly, exp(s + err) ~= exp(s) * (1 + err)).
__device__ __forceinline__ float exp_diff(float a, float b) {
  const float s = a - b;
  const float bb = s - a;
  const float err = (a - (s - bb)) + (-b - bb);
  const float e = expf(s);
  return fmaf(e, err, e);
}

// Order-preserving map of a finite float to an unsigned key (larger float ->
// larger key; -0 and +0 share a key; 0 is below every finite float's key).
__device__ __forceinline__ unsigned okey(float x) {
  const unsigned u = __float_as_uint(x + 0.0f);   // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float okey_value(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// (hi, lo) += x with the rounding error of the add kept in lo (TwoSum).
__device__ __forceinline__ void two_sum_add(float& hi, float& lo, float x) {
  const float s = hi + x;
  const float bb = s - hi;
  lo += (hi - (s - bb)) + (x - bb);
  hi = s;
}

// One arg-max round over the 32 lanes of a warp, each holding V candidates
// (expert g + 32 i, key 0 = none): largest key, then lowest expert among equal
// keys. Returns the winning expert (every lane gets it) and its key in *kout.
template <int V>
__device__ __forceinline__ int warp_argmax_round(const unsigned (&key)[V], unsigned taken, int g,
                                                 unsigned* kout) {
  unsigned best = 0;
#pragma unroll
  for (int i = 0; i < V; ++i)
    if (!((taken >> i) & 1u)) best = max(best, key[i]);
  const unsigned m = __reduce_max_sync(0xffffffffu, best);
  unsigned cand = 0xffffffffu;
#pragma unroll
  for (int i = V - 1; i >= 0; --i)
    if (!((taken >> i) & 1u) && key[i] == m) cand = (unsigned)(g + 32 * i);
  *kout = m;
  return (int)__reduce_min_sync(0xffffffffu, cand);
}

// Experts [base, base + V) of one logits row as float32 (0 past E); 16-byte vector
// loads when E allows them.
template <int V, typename In>
__device__ __forceinline__ void load_row_part(const In* __restrict__ row, int base, int E, float (&v)[V]) {
  if constexpr (!std::is_same<In, float>::value) {
    if ((V % 8) == 0 && (E & 7) == 0) {
#pragma unroll
      for (int q = 0; q < V / 8; ++q) {
        const int e0 = base + 8 * q;
        float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (e0 < E) load8_bf16(row + e0, x);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[8 * q + i] = x[i];
      }
    } else {
#pragma unroll
      for (int i = 0; i < V; ++i) v[i] = base + i < E ? load_logit(row + base + i) : 0.0f;
    }
  } else if ((V % 4) == 0 && (E & 3) == 0) {
#pragma unroll
    for (int q = 0; q < V / 4; ++q) {
      const int e0 = base + 4 * q;
      const float4 x = e0 < E ? __ldg(reinterpret_cast<const float4*>(row + e0)) : make_float4(0.f, 0.f, 0.f, 0.f);
      v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) v[i] = base + i < E ? __ldg(row + base + i) : 0.0f;
  }
}

// One thread's token (row v[0, V), experts past E ignored), K = k: each round an
// arg-max tree over the row (a right node wins only when strictly larger: the
// lower expert among equal values), the winner then set to -inf; the selected
// numerators are kept (the first, exp(m - m), is exactly 1). Weights as in
// gate_one_token.
template <int V, int K>
__device__ __forceinline__ void gate_row_regs(const float (&v)[V], int E, int norm, long t,
                                              float* __restrict__ w_out, int32_t* __restrict__ idx_out) {
  float w[V];
#pragma unroll
  for (int i = 0; i < V; ++i) w[i] = i < E ? v[i] : -INFINITY;
  float ex[K], m = 0.0f, hi = 0.0f, lo = 0.0f;
  int sid[K];
  if constexpr (K == 2 && V >= 2) {
    // the two largest by pairwise merges: every node keeps its range's best and
    // second (value, expert); a node's left range holds the lower experts, so the
    // right side wins only when strictly larger, for the best and for the second
    float bv[V / 2], sv[V / 2];
    int bi[V / 2], si[V / 2];
#pragma unroll
    for (int q = 0; q < V / 2; ++q) {
      const bool r = w[2 * q + 1] > w[2 * q];
      bv[q] = r ? w[2 * q + 1] : w[2 * q];
      bi[q] = r ? 2 * q + 1 : 2 * q;
      sv[q] = r ? w[2 * q] : w[2 * q + 1];
      si[q] = r ? 2 * q : 2 * q + 1;
    }
#pragma unroll
    for (int n = V / 2; n > 1; n /= 2)
#pragma unroll
      for (int q = 0; q < n / 2; ++q) {
        const int a = 2 * q, b = 2 * q + 1;
        const bool r = bv[b] > bv[a];
        // the second: the losing side's best against the winning side's second
        const float xv = r ? bv[a] : sv[a], yv = r ? sv[b] : bv[b];
        const int xi = r ? bi[a] : si[a], yi = r ? si[b] : bi[b];
        const bool r2 = yv > xv;
        bv[q] = r ? bv[b] : bv[a];
        bi[q] = r ? bi[b] : bi[a];
        sv[q] = r2 ? yv : xv;
        si[q] = r2 ? yi : xi;
      }
    m = bv[0];
    sid[0] = bi[0];
    sid[1] = si[0];
    ex[0] = 1.0f;
    ex[1] = exp_diff(sv[0], m);
    if (norm) {
      two_sum_add(hi, lo, ex[0]);
      two_sum_add(hi, lo, ex[1]);
    }
  } else {
#pragma unroll
  for (int j = 0; j < K; ++j) {
    float tv[V];
    int ti[V];
#pragma unroll
    for (int i = 0; i < V; ++i) { tv[i] = w[i]; ti[i] = i; }
#pragma unroll
    for (int st = 1; st < V; st *= 2)
#pragma unroll
      for (int i = 0; i + st < V; i += 2 * st) {
        const bool right = tv[i + st] > tv[i];
        tv[i] = right ? tv[i + st] : tv[i];
        ti[i] = right ? ti[i + st] : ti[i];
      }
    if (j == 0) m = tv[0];
    sid[j] = ti[0];
    if (j + 1 < K) {
#pragma unroll
      for (int i = 0; i < V; ++i) w[i] = i == ti[0] ? -INFINITY : w[i];
    }
    ex[j] = j == 0 ? 1.0f : exp_diff(tv[0], m);
    if (norm) two_sum_add(hi, lo, ex[j]);
  }
  }
  if (!norm) {
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (i < E) two_sum_add(hi, lo, exp_diff(v[i], m));
  }
  const float denom = hi + lo;
  float wj[K];
#pragma unroll
  for (int j = 0; j < K; ++j) wj[j] = __fdiv_rn(ex[j], denom);
  if constexpr (K == 2) {   // whole rows as one 8-byte store each (outputs 16-byte aligned)
    reinterpret_cast<float2*>(w_out)[t] = make_float2(wj[0], wj[1]);
    reinterpret_cast<int2*>(idx_out)[t] = make_int2(sid[0], sid[1]);
  } else if constexpr (K == 4 || K == 8) {
#pragma unroll
    for (int q = 0; q < K / 4; ++q) {
      reinterpret_cast<float4*>(w_out)[t * (K / 4) + q] = make_float4(wj[4 * q], wj[4 * q + 1], wj[4 * q + 2], wj[4 * q + 3]);
      reinterpret_cast<int4*>(idx_out)[t * (K / 4) + q] = make_int4(sid[4 * q], sid[4 * q + 1], sid[4 * q + 2], sid[4 * q + 3]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < K; ++j) {
      w_out[t * K + j] = wj[j];
      idx_out[t * K + j] = sid[j];
    }
  }
}

// Top-k and softmax of one token's logits row by the L lanes of a group (V <= 64); lane
// g holds the contiguous experts [g*V, g*V + V) (vector loads when E % 4 == 0).
// Each of the k rounds takes the best remaining value of every lane (strictly
// greater wins, so the lower index stays first within a lane) and merges the
// lanes with a butterfly on (value desc, index asc). Round j's winner is
// written to slot j by lane j % L (its raw logit first); the denominator is a
// TwoSum-compensated float32 sum (identical in every lane), and a last pass
// turns each slot's logit into its weight with one correctly rounded division.
template <int L, int V, typename In = float>
__device__ __forceinline__ void gate_one_token(const In* __restrict__ logits, long t, int E, int k,
                                               int norm, float* __restrict__ w_out,
                                               int32_t* __restrict__ idx_out) {
  const int g = threadIdx.x & (L - 1);
  const unsigned gm = group_mask<L>();
  const int base = g * V;
  float v[V];
  load_row_part<V>(logits + t * (long)E, base, E, v);
  uint64_t taken = 0;
#pragma unroll
  for (int i = 0; i < V; ++i)
    if (base + i >= E) taken |= 1ull << i;

  float m = 0.0f, hi = 0.0f, lo = 0.0f;
  // one round: the best remaining (value, expert) over the group's lanes
  auto take = [&](float& bv, int& bi) {
    bv = 0.0f;
    bi = kNone;
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (!((taken >> i) & 1ull) && (bi == kNone || v[i] > bv)) { bv = v[i]; bi = base + i; }
#pragma unroll
    for (int off = L / 2; off >= 1; off >>= 1) {
      const float ov = __shfl_xor_sync(gm, bv, off, L);
      const int oi = __shfl_xor_sync(gm, bi, off, L);
      if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (bi / V == g) taken |= 1ull << (bi - base);
  };
  if (L == 1 && k <= kRegSel) {
    // one thread per token, the row in registers, k known at compile time (a loop
    // over runtime k would issue every round's instructions under predicates)
    switch (k) {
      case 1: return gate_row_regs<V, 1>(v, E, norm, t, w_out, idx_out);
      case 2: return gate_row_regs<V, 2>(v, E, norm, t, w_out, idx_out);
      case 3: return gate_row_regs<V, 3>(v, E, norm, t, w_out, idx_out);
      case 4: return gate_row_regs<V, 4>(v, E, norm, t, w_out, idx_out);
      case 5: return gate_row_regs<V, 5>(v, E, norm, t, w_out, idx_out);
      case 6: return gate_row_regs<V, 6>(v, E, norm, t, w_out, idx_out);
      case 7: return gate_row_regs<V, 7>(v, E, norm, t, w_out, idx_out);
      default: return gate_row_regs<V, 8>(v, E, norm, t, w_out, idx_out);
    }
  }
  for (int j = 0; j < k; ++j) {
    float bv;
    int bi;
    take(bv, bi);
    if (j == 0) m = bv;
    if (norm) two_sum_add(hi, lo, exp_diff(bv, m));
    if ((j & (L - 1)) == g) {
      idx_out[t * k + j] = bi;
      w_out[t * k + j] = bv;
    }
  }
  if (!norm) {
#pragma unroll
    for (int i = 0; i < V; ++i)
      if (base + i < E) two_sum_add(hi, lo, exp_diff(v[i], m));
#pragma unroll
    for (int off = L / 2; off >= 1; off >>= 1) {
      const float ohi = __shfl_xor_sync(gm, hi, off, L);
      const float olo = __shfl_xor_sync(gm, lo, off, L);
      two_sum_add(hi, lo, ohi);
      lo += olo;
    }
  }
  const float denom = hi + lo;
  for (int j = g; j < k; j += L) {
    const float x = w_out[t * k + j];        // this lane's own store above
    w_out[t * k + j] = __fdiv_rn(exp_diff(x, m), denom);
  }
}

// ---- thread-per-token top-k over rows parked in shared memory (E <= EP <= 128)
//
// A block of up to kStageRows rows is stored in 16-byte chunks: chunk q of row r
// (its elements q*VE .. q*VE + VE - 1, VE = 16 / sizeof(St)) sits at chunk index
// q * kStageLd + r. The padded stride makes both access patterns bank-conflict
// free per quarter warp: the staging writes (8 lanes, 8 consecutive chunks of one
// row) and the passes over a row (8 lanes, the same chunk of consecutive rows),
// so each is one 16-byte access per lane instead of VE scalar ones. The thread
// of row r selects with the tournament of topk_staged_row.
// Weights as in gate_one_token.
constexpr int kStageRows = 128;
constexpr int kStageLd = kStageRows + 1;

// Elements of a stage element type per 16-byte chunk.
template <typename St>
__host__ __device__ constexpr int chunk_elems() { return 16 / (int)sizeof(St); }

// Stage layouts: the index (in 16-byte units) of chunk q of staged row r.
// StagePadded: chunk columns of kStageLd chunks, the form filled by cp.async
// and thread stores (above). StageSwz128: the form a TMA load of 128-row x
// 128-byte boxes writes with the 128-byte swizzle (box b = chunks 8b .. 8b+7 of
// every row; in each 1 KB block of 8 rows, chunk u of row i sits at u ^ i): the
// 8 lanes of a quarter warp reading one chunk of 8 consecutive rows hit 8
// distinct bank groups whatever the chunk, so the rounds' reads of different
// groups by different rows are conflict-free too; the stage must start on a
// 1024-byte boundary.
struct StagePadded {
  static constexpr int kRowsLd = kStageLd;
  __host__ __device__ static constexpr int chunk(int q, int r) { return q * kStageLd + r; }
};
struct StageSwz128 {
  static constexpr int kRowsLd = kStageRows;
  __host__ __device__ static constexpr int chunk(int q, int r) {
    return (q >> 3) * (kStageRows * 8) + r * 8 + ((q & 7) ^ (r & 7));
  }
};

// Element e of staged row r.
template <typename St, typename Lay = StagePadded>
__host__ __device__ constexpr int sofs(int e, int r) {
  return Lay::chunk(e / chunk_elems<St>(), r) * chunk_elems<St>() + e % chunk_elems<St>();
}

// Staged logits are kept as float32, or for bf16 logits as their 16-bit
// patterns (half the shared memory per row, so more rows fit per SM); either
// way a value read back is the exact float32 of the logit.
__device__ __forceinline__ float st_get(const float* p) { return *p; }
__device__ __forceinline__ float st_get(const uint16_t* p) { return __uint_as_float((uint32_t)*p << 16); }
__device__ __forceinline__ void st_neg_inf(float* p) { *p = -INFINITY; }
__device__ __forceinline__ void st_neg_inf(uint16_t* p) { *p = 0xff80u; }   // bf16 -inf
__device__ __forceinline__ void put_one(float* p, const float* src) { *p = __ldg(src); }
__device__ __forceinline__ void put_one(float* p, const __nv_bfloat16* src) { *p = load_logit(src); }
__device__ __forceinline__ void put_one(uint16_t* p, const __nv_bfloat16* src) {
  *p = __ldg(reinterpret_cast<const unsigned short*>(src));
}

// 16-byte global -> shared copy without a register round trip (L2 only).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The cp.async copies of rows [t0, t0 + nt) into the chunked stage (one 16-byte
// logits vector per stage chunk: E % (16 / sizeof(In)) == 0 and sizeof(In) ==
// sizeof(St)), issued by threads tid = 0..nthr-1 (a multiple of 32) without
// waiting: a warp moves tiles of 4 rows x 8 vectors (4 full 128-byte segments of
// global memory, 8 conflict-free chunk stores per quarter warp).
template <typename In, typename St>
__device__ __forceinline__ void stage_rows_async(const In* __restrict__ logits, long t0, int nt, int E, St* col,
                                                 int tid, int nthr) {
  static_assert(sizeof(In) == sizeof(St), "one logits vector per stage chunk");
  constexpr int VEC = 16 / (int)sizeof(In);
  const int R = E / VEC;   // vectors per row
  const uint4* src = reinterpret_cast<const uint4*>(logits + t0 * (long)E);
  uint4* dst = reinterpret_cast<uint4*>(col);
  const int lane = tid & 31, w = tid >> 5, nw = nthr >> 5;
  const int nrt = (nt + 3) >> 2;   // tiles of 4 rows
  for (int c = lane & 7; c < ((R + 7) & ~7); c += 8)
    for (int rt = w; rt < nrt; rt += nw) {
      const int r = 4 * rt + (lane >> 3);
      if (c < R && r < nt) cp_async16(dst + c * kStageLd + r, src + r * R + c);
    }
}

// Stage rows [t0, t0 + nt) of logits (nt <= kStageRows) into the chunked stage,
// experts E..EP-1 as -inf, by threads tid = 0..nthr-1 (nthr >= kStageRows, a
// multiple of 32); the caller synchronises before reading. With 16-byte rows
// vectors (E a multiple of 4 float32 / 8 bf16 logits) a warp moves tiles of 4
// rows x 8 vectors (4 full 128-byte segments of global memory): by cp.async when
// a vector is one stage chunk (all of a thread's copies in flight at once), else
// (bf16 widened to float32) through registers, U vectors per round trip.
template <int EP, typename In = float, int U = 8, typename St = float>
__device__ __forceinline__ void stage_rows(const In* __restrict__ logits, long t0, int nt, int E,
                                           St* col, int tid, int nthr) {
  constexpr int VEC = 16 / (int)sizeof(In);   // logits per 16-byte vector
  const In* blk = logits + t0 * (long)E;   // the block's rows are contiguous
  if (E % VEC == 0) {
    const int R = E / VEC;                   // vectors per row
    const uint4* src = reinterpret_cast<const uint4*>(blk);
    const int lane = tid & 31, w = tid >> 5, nw = nthr >> 5;
    const int nrt = (nt + 3) >> 2;           // tiles of 4 rows
    if constexpr (sizeof(In) == sizeof(St)) {
      stage_rows_async(logits, t0, nt, E, col, tid, nthr);
      cp_async_wait_all();
    } else {   // 8 bf16 -> two float32 chunks
      float4* dst = reinterpret_cast<float4*>(col);
      for (int c = lane & 7; c < ((R + 7) & ~7); c += 8)
        for (int rt0 = w; rt0 < nrt; rt0 += U * nw) {
          uint4 q[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int r = 4 * (rt0 + u * nw) + (lane >> 3);
            if (c < R && r < nt) q[u] = __ldg(src + r * R + c);
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int r = 4 * (rt0 + u * nw) + (lane >> 3);
            if (c < R && r < nt) {
              dst[(2 * c) * kStageLd + r] = make_float4(lo_bf16(q[u].x), hi_bf16(q[u].x), lo_bf16(q[u].y), hi_bf16(q[u].y));
              dst[(2 * c + 1) * kStageLd + r] = make_float4(lo_bf16(q[u].z), hi_bf16(q[u].z), lo_bf16(q[u].w), hi_bf16(q[u].w));
            }
          }
        }
    }
  } else {
    for (int f = tid; f < nt * E; f += nthr) {
      const int r = f / E;
      put_one(col + sofs<St>(f - r * E, r), blk + f);
    }
  }
  if (tid < kStageRows)
    for (int e = E; e < EP; ++e) st_neg_inf(col + sofs<St>(e, tid));
}

// The 8 staged values of group g (experts 8g .. 8g + 7) of row r: two float32
// chunks, or one chunk of 16-bit patterns.
template <typename Lay = StagePadded>
__device__ __forceinline__ void load_group8(const float* col, int g, int r, float (&x)[8]) {
  const float4* c4 = reinterpret_cast<const float4*>(col);
  const float4 a = c4[Lay::chunk(2 * g, r)], b = c4[Lay::chunk(2 * g + 1, r)];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
template <typename Lay = StagePadded>
__device__ __forceinline__ void load_group8(const uint16_t* col, int g, int r, float (&x)[8]) {
  const uint4 q = reinterpret_cast<const uint4*>(col)[Lay::chunk(g, r)];
  x[0] = lo_bf16(q.x); x[1] = hi_bf16(q.x); x[2] = lo_bf16(q.y); x[3] = hi_bf16(q.y);
  x[4] = lo_bf16(q.z); x[5] = hi_bf16(q.z); x[6] = lo_bf16(q.w); x[7] = hi_bf16(q.w);
}

// The largest of the 8 staged values of group g of row r: float32 as a tree of
// maxima; 16-bit patterns of bf16 by packed bf16 pair maxima (the value is what
// matters: equal values, -0 and +0 included, compare equal as float32 later).
template <typename Lay = StagePadded>
__device__ __forceinline__ float group_max8(const float* col, int g, int r) {
  float y[8];
  load_group8<Lay>(col, g, r, y);
  return fmaxf(fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3])), fmaxf(fmaxf(y[4], y[5]), fmaxf(y[6], y[7])));
}
template <typename Lay = StagePadded>
__device__ __forceinline__ float group_max8(const uint16_t* col, int g, int r) {
  const uint4 q = reinterpret_cast<const uint4*>(col)[Lay::chunk(g, r)];
  auto h2 = [](uint32_t w) { return *reinterpret_cast<const __nv_bfloat162*>(&w); };
  const __nv_bfloat162 m = __hmax2(__hmax2(h2(q.x), h2(q.y)), __hmax2(h2(q.z), h2(q.w)));
  return fmaxf(__low2float(m), __high2float(m));
}

// Of the 8 staged values of group g of row r: eq, bit c set where value c equals v
// (as float32: -0 and +0 equal), and rest, the largest of the others (-inf if none).
// float32 stages as trees over the values; 16-bit stages on packed bf16 pairs (v is
// itself a staged value, so exact as bf16): pair comparisons give the mask, the
// matching halves become -inf by a bitwise select, and pair maxima give the rest.
template <typename Lay = StagePadded>
__device__ __forceinline__ void group_match8(const float* col, int g, int r, float v, unsigned& eq, float& rest) {
  float x[8];
  load_group8<Lay>(col, g, r, x);
  unsigned eqm[8];
  float ne[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    eqm[c] = x[c] == v ? 1u << c : 0u;
    ne[c] = x[c] == v ? -INFINITY : x[c];
  }
  eq = ((eqm[0] | eqm[1]) | (eqm[2] | eqm[3])) | ((eqm[4] | eqm[5]) | (eqm[6] | eqm[7]));
  rest = fmaxf(fmaxf(fmaxf(ne[0], ne[1]), fmaxf(ne[2], ne[3])), fmaxf(fmaxf(ne[4], ne[5]), fmaxf(ne[6], ne[7])));
}
template <typename Lay = StagePadded>
__device__ __forceinline__ void group_match8(const uint16_t* col, int g, int r, float v, unsigned& eq, float& rest) {
  const uint4 q = reinterpret_cast<const uint4*>(col)[Lay::chunk(g, r)];
  auto h2 = [](uint32_t w) { return *reinterpret_cast<const __nv_bfloat162*>(&w); };
  const __nv_bfloat162 vv = __float2bfloat162_rn(v);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  uint32_t m[4], k[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = __heq2_mask(h2(w[i]), vv);                   // 0xffff per equal half
    k[i] = (w[i] & ~m[i]) | (0xff80ff80u & m[i]);      // equal halves -> bf16 -inf
  }
  eq = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) eq |= ((m[i] & 1u) | ((m[i] >> 15) & 2u)) << (2 * i);
  const __nv_bfloat162 mx = __hmax2(__hmax2(h2(k[0]), h2(k[1])), __hmax2(h2(k[2]), h2(k[3])));
  rest = fmaxf(__low2float(mx), __high2float(mx));
}

// Shared memory (bytes) of a stage of kStageRows rows padded to EP experts: EP / VE
// chunk columns of Lay::kRowsLd 16-byte chunks, then (RM false) the float maxima
// of the rows' groups of 8 [EP / 8][kStageLd].
template <int EP, typename St = float, typename Lay = StagePadded>
__host__ __device__ constexpr int stage_rows_bytes() { return EP * Lay::kRowsLd * (int)sizeof(St); }
template <int EP, typename St = float, bool RM = false, typename Lay = StagePadded>
__host__ __device__ constexpr int stage_bytes() {
  return stage_rows_bytes<EP, St, Lay>() + (RM ? 0 : EP / 8 * kStageLd * 4);
}
template <int EP>
__host__ __device__ constexpr int stage_floats() { return stage_bytes<EP, float>() / 4; }

// Top-k and softmax of staged row r (called by one thread), written as token t. With
// s_w / s_idx (shared memory, indexed like the outputs) the results are also kept
// there.
//
// Selection is a tournament over groups of 8 experts. A round finds the largest
// group maximum and its first group holding it, reads that group's 8 values (one
// or two 16-byte reads), takes its first expert holding the value (scans in
// ascending index, so equal values go to the lower expert, as the page's strict
// '>' does), marks it taken (-inf; logits are finite) and refreshes the group's
// maximum. RM true: the group maxima live in registers and the first group is
// found by an arg-max tree (a right node wins only when strictly larger); the
// group read is the round's only shared-memory round trip (measured faster for
// float32 rows of 64-128 experts). RM false: the group maxima live in shared
// memory after the rows and the maxima of 4 consecutive groups ("supers") in
// registers (fewer instructions: faster for the 16-bit stages). Every choice is a select, not a branch: all threads of a warp run the
// same instructions.
//
// TO_COL (k <= kRegSel): instead of w_out / idx_out, the results go to the row's
// own first four chunks (its logits are no longer needed): weight j and index j
// (bits) as the 32-bit words j and kRegSel + j, word s being word s % 4 of chunk
// s / 4 for either element type.
template <int EP, bool TO_COL = false, typename St = float, bool RM = false, typename Lay = StagePadded>
__device__ __forceinline__ void topk_staged_row(St* col, int r, long t, int E, int k, int norm,
                                                float* __restrict__ w_out, int32_t* __restrict__ idx_out,
                                                float* s_w = nullptr, int32_t* s_idx = nullptr) {
  constexpr bool kHalf = sizeof(St) == 2;
  static_assert(!TO_COL || EP >= (kHalf ? 4 : 2) * kRegSel, "room for the parked results");
  constexpr int G = EP / 8;          // groups of 8 experts
  static_assert((G & (G - 1)) == 0, "a power-of-two number of groups");
  constexpr int S = (G + 3) / 4;     // supers of 4 groups (RM false)
  auto at = [&](int i) -> float { return st_get(col + sofs<St, Lay>(i, r)); };
  float* gcol = reinterpret_cast<float*>(reinterpret_cast<char*>(col) + stage_rows_bytes<EP, St, Lay>());
  auto gat = [&](int g) -> float& { return gcol[g * kStageLd + r]; };
  float gmx[RM ? G : 1];
  float sm[S];
#pragma unroll
  for (int q = 0; q < S; ++q) sm[q] = -INFINITY;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float x = group_max8<Lay>(col, g, r);
    if constexpr (RM) gmx[g] = x;
    else gat(g) = x;
    sm[g / 4] = fmaxf(sm[g / 4], x);
  }
  float m = sm[0];
#pragma unroll
  for (int q = 1; q < S; ++q) m = fmaxf(m, sm[q]);
  float hi = 0.0f, lo = 0.0f;
  if (!norm) {
    // The full-row denominator: each group's 8 terms exp(x - m) (x <= m, fast
    // exponential, no correction of the subtraction) summed as a tree, the group
    // sums added with TwoSum into two alternating compensated accumulators. Its
    // relative error stays below about 10 ulp (6e-7): the subtraction's rounding
    // perturbs term i by at most |x_i - m| ulp and the fast exponential by 2 +
    // 1.2 |x_i - m| ulp, and as the terms weigh e^(x_i - m) these average to a few
    // ulp over any row (the largest terms have the smallest |x_i - m|); a tree of
    // 8 positive terms adds 3 ulp. The selected numerators keep exp_diff.
    auto group_sum = [&](int g) {   // one or two 16-byte reads
      float y[8];
      load_group8<Lay>(col, g, r, y);
      float t[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) t[a] = __expf(y[a] - m);
      return ((t[0] + t[1]) + (t[2] + t[3])) + ((t[4] + t[5]) + (t[6] + t[7]));
    };
    float h0 = 0.0f, l0 = 0.0f, h1 = 0.0f, l1 = 0.0f;
    int i = 0;
    for (; i + 16 <= E; i += 16) {
      two_sum_add(h0, l0, group_sum(i / 8));
      two_sum_add(h1, l1, group_sum(i / 8 + 1));
    }
    if (i + 8 <= E) {
      two_sum_add(h0, l0, group_sum(i / 8));
      i += 8;
    }
    float tail = 0.0f;
    for (; i < E; ++i) tail += __expf(at(i) - m);
    two_sum_add(h0, l0, tail);
    hi = h0;
    lo = l0;
    two_sum_add(hi, lo, h1);
    lo += l1;
  }
  // one round: the largest remaining value and its lowest expert; refreshes the maxima
  auto take = [&](float& v, int& e) {
    int bg, bs = 0, bi = 0;
    float gv[4];
    if constexpr (RM) {
      float tv[G];
      int ti[G];
#pragma unroll
      for (int g = 0; g < G; ++g) { tv[g] = gmx[g]; ti[g] = g; }
#pragma unroll
      for (int w = 1; w < G; w *= 2)
#pragma unroll
        for (int g = 0; g + w < G; g += 2 * w) {
          const bool right = tv[g + w] > tv[g];
          tv[g] = right ? tv[g + w] : tv[g];
          ti[g] = right ? ti[g + w] : ti[g];
        }
      v = tv[0];
      bg = ti[0];
    } else {
      v = sm[0];
#pragma unroll
      for (int q = 1; q < S; ++q) v = fmaxf(v, sm[q]);
#pragma unroll
      for (int q = S - 1; q >= 0; --q) bs = sm[q] == v ? q : bs;
#pragma unroll
      for (int i = 0; i < 4; ++i) gv[i] = (G % 4 == 0 || 4 * bs + i < G) ? gat(4 * bs + i) : -INFINITY;
#pragma unroll
      for (int i = 3; i >= 0; --i) bi = gv[i] == v ? i : bi;
      bg = 4 * bs + bi;
    }
    // the group's first expert holding v, and its maximum without that expert
    // (v again when v occurs twice)
    unsigned eq;
    float rest;
    group_match8<Lay>(col, bg, r, v, eq, rest);
    const int bc = __ffs(eq) - 1;
    e = 8 * bg + bc;
    st_neg_inf(col + sofs<St, Lay>(e, r));
    const float nm = (eq & (eq - 1u)) ? v : rest;
    if constexpr (RM) {
#pragma unroll
      for (int g = 0; g < G; ++g) gmx[g] = g == bg ? nm : gmx[g];
    } else {
      gat(bg) = nm;
      float ns = -INFINITY;
#pragma unroll
      for (int i = 0; i < 4; ++i) ns = fmaxf(ns, i == bi ? nm : gv[i]);
#pragma unroll
      for (int q = 0; q < S; ++q) sm[q] = q == bs ? ns : sm[q];
    }
  };
  if (TO_COL || k <= kRegSel) {   // the selected logits stay in registers until the weights are formed
    float sel[kRegSel], ex[kRegSel];
    int sid[kRegSel];
#pragma unroll
    for (int j = 0; j < kRegSel; ++j) {
      if (j < k) {
        take(sel[j], sid[j]);
        ex[j] = exp_diff(sel[j], m);
        if (norm) two_sum_add(hi, lo, ex[j]);
      }
    }
    const float denom = hi + lo;
    if constexpr (TO_COL) {
      uint32_t pw[2 * kRegSel];
#pragma unroll
      for (int j = 0; j < kRegSel; ++j) {
        pw[j] = j < k ? __float_as_uint(__fdiv_rn(ex[j], denom)) : 0u;
        pw[kRegSel + j] = j < k ? (uint32_t)sid[j] : 0u;
      }
      uint4* c4 = reinterpret_cast<uint4*>(col);
#pragma unroll
      for (int h = 0; h < 2 * kRegSel / 4; ++h)
        c4[Lay::chunk(h, r)] = make_uint4(pw[4 * h], pw[4 * h + 1], pw[4 * h + 2], pw[4 * h + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < kRegSel; ++j)
        if (j < k) {
          const float wj = __fdiv_rn(ex[j], denom);
          w_out[t * k + j] = wj;
          idx_out[t * k + j] = sid[j];
          if (s_w) s_w[t * k + j] = wj;
          if (s_idx) s_idx[t * k + j] = sid[j];
        }
    }
    return;
  }
  if constexpr (!TO_COL) {   // k > kRegSel: the weights are formed in place after the k rounds
    for (int j = 0; j < k; ++j) {
      float bv;
      int bi;
      take(bv, bi);
      if (norm) two_sum_add(hi, lo, exp_diff(bv, m));
      idx_out[t * k + j] = bi;
      if (s_w) {
        s_idx[t * k + j] = bi;
        s_w[t * k + j] = bv;
      } else {
        w_out[t * k + j] = bv;
      }
    }
    const float denom = hi + lo;
    for (int j = 0; j < k; ++j) {
      const float x = s_w ? s_w[t * k + j] : w_out[t * k + j];
      const float wj = __fdiv_rn(exp_diff(x, m), denom);
      w_out[t * k + j] = wj;
      if (s_w) s_w[t * k + j] = wj;
    }
  }
}

// Routing of a small batch inside one CTA, every thread of the block taking
// part: the top-k experts of each of the T tokens (a warp per token, experts l
// and l + 32 in lane l, so E <= 64; largest logit first, the lower expert among
// equal logits, as the routing kernels choose), then every expert's count, its
// offset and its tokens in slot order (the stable expert order of the align
// step). All arrays in shared memory: idx[T*k], cnt[E], off[E+1], ids[T*k], run[E],
// and (when not null) pos[T*k]: the sorted position of every slot. One token (a
// decode step) takes a shorter path in warp 0 alone: every expert's rank in the
// row, and from the k best the counts, offsets and slot positions directly; it
// also writes (when not null) active[0, k): the chosen experts ascending, and
// *n_active = k (otherwise untouched).
__device__ __forceinline__ void route_block(const float* __restrict__ logits, int T, int E, int k,
                                            int32_t* idx, int32_t* cnt, int32_t* off, int32_t* ids,
                                            int32_t* run, int32_t* pos = nullptr, int32_t* active = nullptr,
                                            int* n_active = nullptr) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
  const int S = T * k;
  if (T == 1) {
    if (warp == 0) {
      unsigned key[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) key[i] = lane + 32 * i < E ? okey(__ldg(logits + lane + 32 * i)) : 0u;
      // rank of expert lane + 32 i: the experts ahead of it (larger logit, or an
      // equal one at a lower index); experts past E hold key 0 and come last
      int rk[2] = {0, 0};
#pragma unroll 8
      for (int src = 0; src < 32; ++src) {
        const unsigned o0 = __shfl_sync(0xffffffffu, key[0], src), o1 = __shfl_sync(0xffffffffu, key[1], src);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int me = lane + 32 * i;
          rk[i] += (o0 > key[i] || (o0 == key[i] && src < me)) + (o1 > key[i] || (o1 == key[i] && src + 32 < me));
        }
      }
      const bool sel0 = lane < E && rk[0] < k, sel1 = lane + 32 < E && rk[1] < k;
      const unsigned b0 = __ballot_sync(0xffffffffu, sel0), b1 = __ballot_sync(0xffffffffu, sel1);
      const unsigned below = (1u << lane) - 1u;
      const int o[2] = {__popc(b0 & below), __popc(b0) + __popc(b1 & below)};
      const bool sel[2] = {sel0, sel1};
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int me = lane + 32 * i;
        if (me < E) {
          cnt[me] = sel[i] ? 1 : 0;
          off[me] = o[i];
        }
        if (sel[i]) {
          idx[rk[i]] = me;
          ids[o[i]] = 0;
          if (pos) pos[rk[i]] = o[i];
          if (active) active[o[i]] = me;
        }
      }
      if (lane == 0) {
        off[E] = k;
        if (n_active) *n_active = k;
      }
    }
    __syncthreads();
    return;
  }
  for (int t = warp; t < T; t += nwarps) {
    const float* row = logits + (long)t * E;
    unsigned key[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) key[i] = lane + 32 * i < E ? okey(__ldg(row + lane + 32 * i)) : 0u;
    unsigned taken = 0;
    for (int j = 0; j < k; ++j) {
      unsigned kv;
      const int e = warp_argmax_round<2>(key, taken, lane, &kv);
      if ((e & 31) == lane) taken |= 1u << (e >> 5);
      if (lane == 0) idx[t * k + j] = e;
    }
  }
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  for (int q = tid; q < S; q += blockDim.x) atomicAdd(&cnt[idx[q]], 1);
  __syncthreads();
  if (warp == 0) {   // exclusive offsets, two experts per lane
    const int a = 2 * lane < E ? cnt[2 * lane] : 0, b = 2 * lane + 1 < E ? cnt[2 * lane + 1] : 0;
    int incl = a + b;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    if (2 * lane < E) off[2 * lane] = incl - a - b;
    if (2 * lane + 1 < E) off[2 * lane + 1] = incl - b;
    if (lane == 31) off[E] = incl;
  }
  __syncthreads();
  if (warp == 0) {   // rounds of 32 slots, ranked within their expert by __match_any_sync
    for (int e = lane; e < E; e += 32) run[e] = 0;
    __syncwarp();
    for (int q0 = 0; q0 < S; q0 += 32) {
      const int q = q0 + lane;
      const int e = q < S ? idx[q] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int below = __popc(peers & ((1u << lane) - 1u));
      const int prior = e >= 0 ? run[e] : 0;
      __syncwarp();
      if (e >= 0) {
        ids[off[e] + prior + below] = q / k;
        if (pos) pos[q] = off[e] + prior + below;
        if (below == 0) run[e] = prior + __popc(peers);
      }
      __syncwarp();
    }
  }
  __syncthreads();
}

}  // namespace gate
}  // namespace moe

// Dispatch on E: L lanes per row, V values per lane (L * V >= E).
#define MOE_DISPATCH_LV(E, FN, ...)                                        \
  do {                                                                     \
    if ((E) <= 8) return FN<1, 8>(__VA_ARGS__);                            \
    if ((E) <= 16) return FN<1, 16>(__VA_ARGS__);                          \
    if ((E) <= 32) return FN<1, 32>(__VA_ARGS__);                          \
    if ((E) <= 64) return FN<1, 64>(__VA_ARGS__);                          \
    if ((E) <= 128) return FN<2, 64>(__VA_ARGS__);                         \
    if ((E) <= 256) return FN<4, 64>(__VA_ARGS__);                         \
    if ((E) <= 512) return FN<8, 64>(__VA_ARGS__);                         \
    return FN<16, 64>(__VA_ARGS__);                                        \
  } while (0)
