// Align by expert: counts, exclusive offsets, stable sorted token ids / weights,
// reverse slot ids.
//
// mlc-llm moe_misc.py: moe_cumsum (the sorted position of slot (b, j) routed to
// e is cumsum[e*T + b] - 1 over the transposed expert mask), get_indptr
// (exclusive), get_indices; project_6 moe_expert_gemm.cpp moe_prefill_experts
// (counts, sorted ids, sorted weights).
//
// The E*T mask cumsum is never materialised. Because a row names distinct
// experts, "tokens t' < t routed to e" equals "flat slots s' < s holding e",
// so the sorted position of flat slot s = t*k + j is
//     offsets[e] + #{s' < s : idx[s'] == e}.
// Launches:
//   1. align_hist: each CTA counts its chunk of slots per expert (shared-memory
//      atomics; the counts are order-free) into chunk_hist[c][e];
//   2. (many chunks only) align_scan: one CTA per expert turns its column of
//      chunk_hist into an inclusive prefix over chunks, in place;
//   3. align_scatter: each CTA derives offsets and its chunk's per-expert base
//      from chunk_hist (summing the few chunks before it, or reading the
//      prefix), then ranks its slots in one round: warp w takes 256
//      consecutive slots in 8 sub-rounds of 32 (lanes of the same expert by
//      __match_any_sync, or per-bit ballots above 16 experts here, + popc of
//      lower lanes on top of the warp's running per-expert count), a
//      per-expert prefix over the warps' counts places the warps, the slots go
//      to an expert-sorted copy of the chunk in shared memory, and each
//      expert's run is copied out with consecutive threads (coalesced stores).
// A single-chunk problem runs as one launch (the CTA makes its own histogram).
#include <map>
#include <mutex>

#include "common.cuh"
#include "gating_device.cuh"

namespace moe {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 4096;   // slots per CTA
constexpr int kSub = kChunk / kThreads;   // sub-rounds of 32 slots per warp (its kChunk / kWarps slots)
constexpr int kScanAbove = 16; // chunks above which the per-expert prefix gets its own launch

__device__ __forceinline__ int valid_expert(int e, int E) { return (e >= 0 && e < E) ? e : -1; }

// Lanes of the warp holding the same expert as this lane (e >= 0), built from one
// ballot per bit of the expert id plus one for validity; `bits` = bits of E - 1.
// Measured against __match_any_sync in the many-CTA align ranking: 12-14% faster
// for E = 64 / 128, 5% slower for E = 8, so it is used there above 16 experts;
// the single-CTA small-batch routing (latency-bound) measured slower with it.
__device__ __forceinline__ unsigned same_expert_lanes(int e, int bits) {
  unsigned m = __ballot_sync(0xffffffffu, e >= 0);
  for (int b = 0; b < bits; ++b) {
    const unsigned bal = __ballot_sync(0xffffffffu, (e >> b) & 1);
    m &= ((e >> b) & 1) ? bal : ~bal;
  }
  return m;
}

// The same with the number of bits fixed at compile time (the ballots unrolled).
template <int BITS>
__device__ __forceinline__ unsigned same_expert_lanes_t(int e) {
  unsigned m = __ballot_sync(0xffffffffu, e >= 0);
#pragma unroll
  for (int b = 0; b < BITS; ++b) {
    const unsigned bal = __ballot_sync(0xffffffffu, (e >> b) & 1);
    m &= ((e >> b) & 1) ? bal : ~bal;
  }
  return m;
}

// Dynamic shared memory of align_chunk for E experts.
__host__ __device__ inline size_t align_smem_bytes(int E) {
  return (size_t)(3 * E + 2 + kWarps * E + 4 * kChunk) * sizeof(int);
}

__global__ void __launch_bounds__(kThreads) align_hist_kernel(const int32_t* __restrict__ idx,
                                                              long S, int E,
                                                              int32_t* __restrict__ chunk_hist,
                                                              int32_t* status) {
  extern __shared__ int hist[];
  pdl_wait();      // the routing was written by the previous kernel
  pdl_trigger();
  for (int e = threadIdx.x; e < E; e += kThreads) hist[e] = 0;
  __syncthreads();
  const long lo = (long)blockIdx.x * kChunk;
  const long hi = min(S, lo + kChunk);
  bool bad = false;
  auto count = [&](int e) {
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else bad = true;
  };
  if (hi - lo == kChunk) {   // a whole chunk: two 16-byte loads per thread, both in flight
    static_assert(kChunk == 8 * kThreads, "eight slots per thread");
    const int4 a = __ldg(reinterpret_cast<const int4*>(idx + lo) + threadIdx.x);
    const int4 b = __ldg(reinterpret_cast<const int4*>(idx + lo) + kThreads + threadIdx.x);
    count(a.x); count(a.y); count(a.z); count(a.w);
    count(b.x); count(b.y); count(b.z); count(b.w);
  } else {
    for (long s = lo + threadIdx.x; s < hi; s += kThreads) count(__ldg(idx + s));
  }
  if (bad && status) atomicOr(status, MOE_STATUS_BAD_INDEX);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) chunk_hist[(long)blockIdx.x * E + e] = hist[e];
}

// In place: chunk_hist[c][e] <- sum over c' <= c of chunk_hist[c'][e]; one CTA per expert,
// each thread a contiguous run of chunks, block scan of the run totals.
__global__ void __launch_bounds__(1024) align_scan_kernel(int32_t* __restrict__ chunk_hist, int nchunks, int E) {
  __shared__ int wsum[32];
  pdl_wait();      // the histograms of align_hist_kernel
  pdl_trigger();
  const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (nchunks + 1023) / 1024;
  const int c0 = min(nchunks, tid * per), c1 = min(nchunks, c0 + per);
  constexpr int kKeep = 4;   // runs this short stay in registers between the two passes
  int v[kKeep];
  int run = 0;
  if (per <= kKeep) {
#pragma unroll
    for (int i = 0; i < kKeep; ++i) v[i] = c0 + i < c1 ? chunk_hist[(long)(c0 + i) * E + e] : 0;
#pragma unroll
    for (int i = 0; i < kKeep; ++i) run += v[i];
  } else {
    for (int c = c0; c < c1; ++c) run += chunk_hist[(long)c * E + e];
  }
  int incl = run;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = wsum[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v, d);
      if (lane >= d) v += o;
    }
    wsum[lane] = v;   // inclusive over warps
  }
  __syncthreads();
  int acc = (warp ? wsum[warp - 1] : 0) + incl - run;
  if (per <= kKeep) {
#pragma unroll
    for (int i = 0; i < kKeep; ++i)
      if (c0 + i < c1) {
        acc += v[i];
        chunk_hist[(long)(c0 + i) * E + e] = acc;
      }
  } else {
    for (int c = c0; c < c1; ++c) {
      acc += chunk_hist[(long)c * E + e];
      chunk_hist[(long)c * E + e] = acc;
    }
  }
}

// Where align_chunk reads the routing (indices, weights) from: global memory
// through the read-only path, global memory through L2 (the same kernel has
// just written it), or a shared-memory copy made by the same CTA.
enum { kSrcGlobal = 0, kSrcFresh = 1, kSrcShared = 2 };
template <int SRC>
__device__ __forceinline__ int load_i(const int32_t* p) {
  return SRC == kSrcShared ? *p : (SRC == kSrcFresh ? __ldcg(p) : __ldg(p));
}
template <int SRC>
__device__ __forceinline__ float load_f(const float* p) {
  return SRC == kSrcShared ? *p : (SRC == kSrcFresh ? __ldcg(p) : __ldg(p));
}

// Exclusive scan of v[0..n) in place by warp 0 (lane l owns a run of entries);
// returns the total in lane 31.
__device__ __forceinline__ int warp0_exclusive_scan(int* v, int n) {
  const int lane = threadIdx.x & 31;
  const int per = (n + 31) / 32;
  const int e0 = min(n, lane * per), e1 = min(n, e0 + per);
  int run = 0;
  for (int e = e0; e < e1; ++e) run += v[e];
  int incl = run;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += o;
  }
  int acc = incl - run;
  for (int e = e0; e < e1; ++e) {
    const int c = v[e];
    v[e] = acc;
    acc += c;
  }
  return incl;
}

// Align chunk c of the slots (all kThreads threads of the CTA take part).
// Shared layout (ints): off[E+1] | cb[E] | cpre[E+1] | wcnt[kWarps][E]
//                       | staged token ids, slots, weights, destinations [kChunk] each.
// cb[e] is the number of expert e's slots in earlier chunks, cpre[e] the
// chunk-local start of e's slots, wcnt[w][e] warp w's count of e, then the
// number of e's slots in the chunk's warps before w. Slots are ranked into the
// staging arrays in expert-sorted order together with their global position,
// then copied out by consecutive threads (each expert's run is contiguous in
// both orders: coalesced stores). Slot indices are 32-bit (T*k < 2^31). With
// a power-of-two k the token of a staged slot is derived from the slot.
//
// Ranking. K8 (k == 8, a chunk is 512 tokens, one per thread): thread t holds
// token t's 8 slots, which name distinct experts, so a slot's rank among its
// warp's slots of the same expert is the number of lower lanes whose token
// names that expert: each lane sets its bit in the warp's 32-bit mask of every
// expert it names (shared-memory atomicOr), and the rank is the population
// count of the mask below the lane. A repeated expert within a row (outside
// what top-k routing produces; detected when the lane's bit was already set)
// sends the whole CTA to the general ranking. General: warp w takes the
// chunk's slots [w * 32 * kSub, (w + 1) * 32 * kSub) as kSub sub-rounds of 32,
// ranking each by its same-expert lanes on top of the warp's running
// per-expert count.
template <int SRC, int EB = 0, bool K8 = false>
__device__ __forceinline__ void align_chunk(
    int c, const int32_t* idx, const float* wts, long S, int k, int E, int nchunks, int hist_is_prefix,
    const int32_t* __restrict__ chunk_hist, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ sorted_ids, float* __restrict__ sorted_w, int32_t* __restrict__ reverse,
    int32_t* status, int* sm) {
  int* off = sm;
  int* cb = off + E + 1;
  int* cpre = cb + E;
  int* wcnt = cpre + E + 1;
  int* s_tok = wcnt + kWarps * E;
  int* s_rev = s_tok + kChunk;
  float* s_w = reinterpret_cast<float*>(s_rev + kChunk);
  int* s_dst = s_rev + 2 * kChunk;
  const int lo = c * kChunk;
  const int hi = (int)min(S, (long)lo + kChunk);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kshift = (k & (k - 1)) == 0 ? __ffs(k) - 1 : -1;   // token of slot s: s >> kshift or s / k
  const int wbase = lo + warp * 32 * kSub;

  // 0. this thread's slots (step 3), loaded first so that their latency overlaps steps 1-2;
  //    the barriers of steps 1-2 also order the zeroing of wcnt before step 3.
  //    Launched behind the histogram / scan kernels (programmatic serialization), the
  //    routing is two or more launches back and may be read before pdl_wait(); as the
  //    only align kernel (one chunk) it comes straight after the routing's producer.
  if constexpr (SRC == kSrcGlobal)
    if (!chunk_hist) pdl_wait();
  for (int i = tid; i < kWarps * E; i += kThreads) wcnt[i] = 0;
  int eu[kSub], ru[kSub];
  float wu[kSub];
  auto load_general = [&]() {
#pragma unroll
    for (int u = 0; u < kSub; ++u) {
      const int s = wbase + u * 32 + lane;
      eu[u] = s < hi ? load_i<SRC>(idx + s) : -1;
      wu[u] = s < hi ? load_f<SRC>(wts + s) : 0.0f;
    }
  };
  bool masks = K8;
  if constexpr (K8) {
    static_assert(kSub == 8 && SRC == kSrcGlobal, "one 8-slot token per thread, read from global memory");
    const int s0 = lo + 8 * tid;
    if (s0 + 8 <= hi) {
      const int4 a = __ldg(reinterpret_cast<const int4*>(idx + s0));
      const int4 b = __ldg(reinterpret_cast<const int4*>(idx + s0) + 1);
      const float4 x = __ldg(reinterpret_cast<const float4*>(wts + s0));
      const float4 y = __ldg(reinterpret_cast<const float4*>(wts + s0) + 1);
      eu[0] = a.x; eu[1] = a.y; eu[2] = a.z; eu[3] = a.w; eu[4] = b.x; eu[5] = b.y; eu[6] = b.z; eu[7] = b.w;
      wu[0] = x.x; wu[1] = x.y; wu[2] = x.z; wu[3] = x.w; wu[4] = y.x; wu[5] = y.y; wu[6] = y.z; wu[7] = y.w;
    } else {
#pragma unroll
      for (int u = 0; u < kSub; ++u) {
        eu[u] = s0 + u < hi ? __ldg(idx + s0 + u) : -1;
        wu[u] = s0 + u < hi ? __ldg(wts + s0 + u) : 0.0f;
      }
    }
  } else {
    load_general();
  }
  if constexpr (SRC == kSrcGlobal) {   // the histograms come from the launch just before
    if (chunk_hist) pdl_wait();
    pdl_trigger();
  }

  // 1. per-expert totals (off[]), slots of earlier chunks (cb[]) and this chunk's counts (cpre[])
  if (chunk_hist && hist_is_prefix) {
    for (int e = tid; e < E; e += kThreads) {
      const int before = c > 0 ? __ldg(chunk_hist + (long)(c - 1) * E + e) : 0;
      cb[e] = before;
      cpre[e] = __ldg(chunk_hist + (long)c * E + e) - before;
      off[e] = __ldg(chunk_hist + (long)(nchunks - 1) * E + e);
    }
    __syncthreads();
  } else if (chunk_hist) {
    for (int e = tid; e < E; e += kThreads) {
      int before = 0, total = 0;
      for (int cc = 0; cc < nchunks; ++cc) {
        const int h = __ldg(chunk_hist + (long)cc * E + e);
        before += cc < c ? h : 0;
        total += h;
      }
      cb[e] = before;
      cpre[e] = __ldg(chunk_hist + (long)c * E + e);
      off[e] = total;
    }
    __syncthreads();
  } else {   // single chunk: histogram here
    for (int e = tid; e < E; e += kThreads) { cb[e] = 0; off[e] = 0; }
    __syncthreads();
    bool bad = false;
    for (int s = lo + tid; s < hi; s += kThreads) {
      const int e = load_i<SRC>(idx + s);
      if (e >= 0 && e < E) atomicAdd(&off[e], 1);
      else bad = true;
    }
    if (bad && status) atomicOr(status, MOE_STATUS_BAD_INDEX);
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) cpre[e] = off[e];
    __syncthreads();
  }

  // 2. exclusive scans over experts: totals -> offsets (warp 0), chunk counts -> cpre (warp 1)
  if (warp == 0) {
    if (c == 0) {
      for (int e = lane; e < E; e += 32) counts[e] = off[e];
    }
    __syncwarp();
    const int total = warp0_exclusive_scan(off, E);
    if (lane == 31) {
      off[E] = total;
      if (c == 0) offsets[E] = total;
    }
  } else if (warp == 1) {
    const int total = warp0_exclusive_scan(cpre, E);
    if (lane == 31) cpre[E] = total;
  }
  __syncthreads();
  if (c == 0)
    for (int e = tid; e < E; e += kThreads) offsets[e] = off[e];

  // 3. ranking within the warp, then a per-expert prefix over the warps
  if constexpr (K8) {
    unsigned* msk = reinterpret_cast<unsigned*>(wcnt) + warp * E;
    const unsigned bit = 1u << lane;
    bool dup = false;
#pragma unroll
    for (int u = 0; u < kSub; ++u) {
      const int e = valid_expert(eu[u], E);
      eu[u] = e;
      if (e >= 0) dup |= (atomicOr(msk + e, bit) & bit) != 0u;
    }
    __syncwarp();
#pragma unroll
    for (int u = 0; u < kSub; ++u) ru[u] = eu[u] >= 0 ? __popc(msk[eu[u]] & (bit - 1u)) : 0;
    if (__syncthreads_or(dup)) {   // a repeated expert in some row: general ranking for this chunk
      masks = false;
      for (int i = tid; i < kWarps * E; i += kThreads) wcnt[i] = 0;
      load_general();
      __syncthreads();
    }
  }
  if (!masks) {
    const int ebits = 32 - __clz(max(E - 1, 1));
#pragma unroll
    for (int u = 0; u < kSub; ++u) {
      const int e = valid_expert(eu[u], E);
      const unsigned peers = EB > 0 ? same_expert_lanes_t<EB>(e)
                             : SRC == kSrcGlobal && ebits > 4 ? same_expert_lanes(e, ebits)
                                                              : __match_any_sync(0xffffffffu, e);
      const int below = __popc(peers & ((1u << lane) - 1u));
      const int prior = e >= 0 ? wcnt[warp * E + e] : 0;
      __syncwarp();
      if (e >= 0 && below == 0) wcnt[warp * E + e] = prior + __popc(peers);
      __syncwarp();
      eu[u] = e;
      ru[u] = prior + below;
    }
  }
  __syncthreads();
  for (int x = tid; x < E; x += kThreads) {
    int run = 0;
#pragma unroll 4
    for (int w = 0; w < kWarps; ++w) {
      const int v = wcnt[w * E + x];
      const int cnt = masks ? __popc((unsigned)v) : v;
      wcnt[w * E + x] = run;
      run += cnt;
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kSub; ++u) {
    const int e = eu[u];
    if (e >= 0) {
      const int s = masks ? lo + 8 * tid + u : wbase + u * 32 + lane;
      const int base = cpre[e];
      const int q = base + wcnt[warp * E + e] + ru[u];   // chunk-local, expert-sorted
      if (kshift < 0) s_tok[q] = (int)((uint32_t)s / (uint32_t)k);
      s_rev[q] = s;
      s_w[q] = wu[u];
      s_dst[q] = off[e] + cb[e] + (q - base);
    }
  }
  __syncthreads();

  // 4. copy the staged slots to their global positions (coalesced within each expert's run)
  const int n = cpre[E];
  for (int q = tid; q < n; q += kThreads) {
    const int p = s_dst[q];
    const int sl = s_rev[q];
    sorted_ids[p] = kshift >= 0 ? sl >> kshift : s_tok[q];
    reverse[p] = sl;
    sorted_w[p] = s_w[q];
  }
}

// EB: bits of E - 1 (5..10, the per-bit ballots unrolled), or 0 (E <= 16: __match_any_sync).
template <int EB, bool K8 = false>
__global__ void __launch_bounds__(kThreads) align_scatter_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ wts, long S, int k, int E,
    int nchunks, int hist_is_prefix, const int32_t* __restrict__ chunk_hist, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_ids,
    float* __restrict__ sorted_w, int32_t* __restrict__ reverse, int32_t* status) {
  extern __shared__ int sm[];
  align_chunk<kSrcGlobal, EB, K8>(blockIdx.x, idx, wts, S, k, E, nchunks, hist_is_prefix, chunk_hist, counts, offsets,
                     sorted_ids, sorted_w, reverse, status, sm);
}

// Small batches (at most kStageRows tokens, all routed slots in one align
// chunk): gating and align in one CTA and one launch. For E <= 128 the CTA
// stages the logits rows in shared memory and one thread per token runs the
// staged top-k (gate::topk_staged_row); wider rows take a warp per token
// (gate::gate_one_token). After a barrier the CTA ranks and scatters the slots
// it has just written.
template <int EP>
__global__ void __launch_bounds__(kThreads) route_small_staged_kernel(
    const float* logits, int T, int E, int k, int norm, float* w_out, int32_t* idx_out,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_ids,
    float* __restrict__ sorted_w, int32_t* __restrict__ reverse, int32_t* status, int32_t* clear) {
  extern __shared__ __align__(16) int sm[];
  // launched while the previous kernel on the stream finishes: its writes (the logits,
  // or the previous layer step's use of the counters cleared below) are complete after
  // the wait; only then may the FFN kernel, which reads the logits at once, launch
  pdl_wait();
  pdl_trigger();
  if (clear && threadIdx.x < kDecodeSyncWords) clear[threadIdx.x] = 0;
  float* col = reinterpret_cast<float*>(sm);
  int* asm_ = sm + gate::stage_floats<EP>();                  // align_chunk's shared memory
  int32_t* s_idx = asm_ + align_smem_bytes(E) / sizeof(int);  // shared copies of the routing
  float* s_w = reinterpret_cast<float*>(s_idx + T * k);
  gate::stage_rows<EP>(logits, 0, T, E, col, threadIdx.x, kThreads);
  __syncthreads();
  if ((int)threadIdx.x < T)
    gate::topk_staged_row<EP>(col, threadIdx.x, threadIdx.x, E, k, norm, w_out, idx_out, s_w, s_idx);
  __syncthreads();
  align_chunk<kSrcShared>(0, s_idx, s_w, (long)T * k, k, E, 1, 0, nullptr, counts, offsets, sorted_ids,
                          sorted_w, reverse, status, asm_);
}

template <int L, int V>
__global__ void __launch_bounds__(kThreads) route_small_kernel(
    const float* __restrict__ logits, int T, int E, int k, int norm, float* w_out, int32_t* idx_out,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_ids,
    float* __restrict__ sorted_w, int32_t* __restrict__ reverse, int32_t* status, int32_t* clear) {
  extern __shared__ int sm[];
  pdl_wait();   // as in route_small_staged_kernel
  pdl_trigger();
  if (clear && threadIdx.x < kDecodeSyncWords) clear[threadIdx.x] = 0;
  constexpr int groups = kThreads / L;
  for (long t = threadIdx.x / L; t < T; t += groups)
    gate::gate_one_token<L, V>(logits, t, E, k, norm, w_out, idx_out);
  __syncthreads();
  align_chunk<kSrcFresh>(0, idx_out, w_out, (long)T * k, k, E, 1, 0, nullptr, counts, offsets, sorted_ids,
                    sorted_w, reverse, status, sm);
}

template <typename Kernel>
int launch_route_small_k(Kernel kernel, size_t smem, size_t smem_max, const float* logits, int T, int E,
                         int k, int norm, float* w, int32_t* idx, int32_t* counts, int32_t* offsets,
                         int32_t* sorted_ids, float* sorted_w, int32_t* reverse, int32_t* status,
                         int32_t* clear, cudaStream_t s) {
  if (int rc = ensure_smem_limit(kernel, smem_max, "route_small")) return rc;
  ProfScope ps("route_small", s);
  const cudaError_t e = launch_pdl(kernel, 1, kThreads, smem, s, logits, T, E, k, norm, w, idx, counts, offsets,
                                   sorted_ids, sorted_w, reverse, status, clear);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "route_small: %s", cudaGetErrorString(e));
  return check_launch("route_small");
}

template <int EP>
int launch_route_staged(const float* logits, int T, int E, int k, int norm, float* w, int32_t* idx,
                        int32_t* counts, int32_t* offsets, int32_t* sorted_ids, float* sorted_w,
                        int32_t* reverse, int32_t* status, int32_t* clear, cudaStream_t s) {
  const size_t stage = (size_t)gate::stage_floats<EP>() * sizeof(float);
  const size_t copies = (size_t)T * k * (sizeof(int32_t) + sizeof(float));
  return launch_route_small_k(route_small_staged_kernel<EP>, stage + align_smem_bytes(E) + copies,
                              stage + align_smem_bytes(EP) + (size_t)kChunk * 8, logits, T, E, k, norm, w, idx,
                              counts, offsets, sorted_ids, sorted_w, reverse, status, clear, s);
}

template <int V>
int launch_route_warp(const float* logits, int T, int E, int k, int norm, float* w, int32_t* idx,
                      int32_t* counts, int32_t* offsets, int32_t* sorted_ids, float* sorted_w,
                      int32_t* reverse, int32_t* status, int32_t* clear, cudaStream_t s) {
  return launch_route_small_k(route_small_kernel<32, V>, align_smem_bytes(E), align_smem_bytes(MOE_MAX_EXPERTS),
                              logits, T, E, k, norm, w, idx, counts, offsets, sorted_ids, sorted_w, reverse,
                              status, clear, s);
}

}  // namespace

bool route_is_small(int T, int k) { return T <= gate::kStageRows && (long)T * k <= kChunk; }

int launch_route_small(const float* logits, int T, int E, int k, int norm, float* w, int32_t* idx,
                       int32_t* counts, int32_t* offsets, int32_t* sorted_ids, float* sorted_w,
                       int32_t* reverse, int32_t* status, int32_t* clear, cudaStream_t s) {
#define MOE_ROUTE_STAGED(EP) \
  return launch_route_staged<EP>(logits, T, E, k, norm, w, idx, counts, offsets, sorted_ids, sorted_w, reverse, \
                                 status, clear, s)
#define MOE_ROUTE_WARP(V) \
  return launch_route_warp<V>(logits, T, E, k, norm, w, idx, counts, offsets, sorted_ids, sorted_w, reverse, \
                              status, clear, s)
  if (E <= 8) MOE_ROUTE_STAGED(8);
  if (E <= 16) MOE_ROUTE_STAGED(16);
  if (E <= 32) MOE_ROUTE_STAGED(32);
  if (E <= 64) MOE_ROUTE_STAGED(64);
  if (E <= 128) MOE_ROUTE_STAGED(128);
  if (E <= 256) MOE_ROUTE_WARP(8);
  if (E <= 512) MOE_ROUTE_WARP(16);
  MOE_ROUTE_WARP(32);
#undef MOE_ROUTE_STAGED
#undef MOE_ROUTE_WARP
}

size_t align_scratch_bytes(long S, int E) {
  const size_t nchunks = S > 0 ? (size_t)((S + kChunk - 1) / kChunk) : 0;
  return nchunks > 1 ? nchunks * (size_t)E * sizeof(int32_t) : 0;
}

int launch_align(const int32_t* idx, const float* w, int T, int k, int E, int32_t* counts,
                 int32_t* offsets, int32_t* sorted_ids, float* sorted_w, int32_t* reverse,
                 void* scratch, int32_t* status, cudaStream_t s) {
  const long S = (long)T * k;
  const int nchunks = (int)((S + kChunk - 1) / kChunk);
  const size_t smem = align_smem_bytes(E);
  const int ebits = 32 - __builtin_clz((unsigned)(E > 1 ? E - 1 : 1));
  int32_t* hist = nullptr;
  if (nchunks > 1) {
    hist = static_cast<int32_t*>(scratch);
    ProfScope ps("align_hist", s);
    const cudaError_t e = launch_pdl(align_hist_kernel, nchunks, kThreads, E * sizeof(int), s, idx, S, E, hist, status);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "align_hist: %s", cudaGetErrorString(e));
    int rc = check_launch("align_hist");
    if (rc) return rc;
  }
  const int prefix = nchunks > kScanAbove;
  if (prefix) {
    ProfScope ps("align_scan", s);
    const cudaError_t e = launch_pdl(align_scan_kernel, E, 1024, 0, s, hist, nchunks, E);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "align_scan: %s", cudaGetErrorString(e));
    int rc = check_launch("align_scan");
    if (rc) return rc;
  }
  auto scatter = [&](auto kernel) -> int {
    if (int rc = ensure_smem_limit(kernel, align_smem_bytes(MOE_MAX_EXPERTS), "align_scatter")) return rc;
    ProfScope ps("align_scatter", s);
    const cudaError_t e = launch_pdl(kernel, nchunks > 0 ? nchunks : 1, kThreads, smem, s, idx, w, S, k, E, nchunks,
                                     prefix, hist, counts, offsets, sorted_ids, sorted_w, reverse, status);
    if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "align_scatter: %s", cudaGetErrorString(e));
    return check_launch("align_scatter");
  };
  if (k == 8) {   // one token per thread, ranked by per-warp expert masks
    switch (ebits) {
      case 5: return scatter(align_scatter_kernel<5, true>);
      case 6: return scatter(align_scatter_kernel<6, true>);
      case 7: return scatter(align_scatter_kernel<7, true>);
      case 8: return scatter(align_scatter_kernel<8, true>);
      case 9: return scatter(align_scatter_kernel<9, true>);
      case 10: return scatter(align_scatter_kernel<10, true>);
      default: return scatter(align_scatter_kernel<0, true>);
    }
  }
  switch (ebits) {
    case 5: return scatter(align_scatter_kernel<5>);
    case 6: return scatter(align_scatter_kernel<6>);
    case 7: return scatter(align_scatter_kernel<7>);
    case 8: return scatter(align_scatter_kernel<8>);
    case 9: return scatter(align_scatter_kernel<9>);
    case 10: return scatter(align_scatter_kernel<10>);
    default: return scatter(align_scatter_kernel<0>);
  }
}

// ---- fixed scratch for callers that cannot allocate --------------------------
//
// Some callers cannot obtain device memory at call time: host code that only
// receives tensors from a framework without access to its allocator, or a
// runtime whose device memory is planned once at start-up and may not grow.
// They cannot pass a workspace, so moe_align_by_expert_noalloc keeps the
// per-chunk histograms in this file-scope array instead. Every GPU that loads
// the library holds it (MOE_ALIGN_NOALLOC_SCRATCH_INTS int32 = 256 KiB) until
// the process exits. All calls share it: calls whose work overlaps on the GPU
// (different streams, or different host threads) race on it. The histograms
// are fully rewritten before they are read, so nothing needs clearing.
static __device__ __align__(256) int32_t g_align_scratch[MOE_ALIGN_NOALLOC_SCRATCH_INTS];

// Device address of g_align_scratch in the CUDA context current on this thread.
// In host code the array's name is only a host-side stand-in, so the address
// is looked up with cudaGetSymbolAddress, with the device current, on the first
// call that needs the array (ceil(T*k/4096) > 1) in that context: once per
// device for callers of the runtime's primary context, once more for each
// context of their own. That first call should come before any stream capture.
// The address belongs to the context (a context of its own, or the primary
// context after cudaDeviceReset, has its own copy of the array), so the cache
// is keyed by the context's process-unique id, never by the device ordinal.
static int align_scratch_address(int32_t** out) {
  static std::mutex mu;
  static std::map<unsigned long long, int32_t*> addr;
  const unsigned long long ctx = current_context_id();
  if (ctx != 0) {
    std::lock_guard<std::mutex> lk(mu);
    auto it = addr.find(ctx);
    if (it != addr.end()) {
      *out = it->second;
      return MOE_OK;
    }
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_align_scratch);
  if (e != cudaSuccess || p == nullptr)
    return fail(MOE_ERR_CUDA, "cudaGetSymbolAddress(align scratch): %s", cudaGetErrorString(e));
  if (ctx != 0) {   // without a context id the address is looked up on every call
    std::lock_guard<std::mutex> lk(mu);
    addr[ctx] = static_cast<int32_t*>(p);
  }
  *out = static_cast<int32_t*>(p);
  return MOE_OK;
}

int launch_align_noalloc(const int32_t* idx, const float* w, int T, int k, int E, int32_t* counts,
                         int32_t* offsets, int32_t* sorted_ids, float* sorted_w, int32_t* reverse,
                         int32_t* status, cudaStream_t s) {
  const long S = (long)T * k;
  const size_t need = align_scratch_bytes(S, E);
  if (need > sizeof(g_align_scratch))
    return fail(MOE_ERR_UNSUPPORTED,
                "align without workspace: T*k=%ld with E=%d needs %zu bytes of scratch, above the "
                "fixed %zu (ceil(T*k/4096)*E must not exceed %d)",
                S, E, need, sizeof(g_align_scratch), MOE_ALIGN_NOALLOC_SCRATCH_INTS);
  int32_t* scratch = nullptr;   // a single chunk needs no scratch
  if (need > 0) {
    const int rc = align_scratch_address(&scratch);
    if (rc) return rc;
  }
  return launch_align(idx, w, T, k, E, counts, offsets, sorted_ids, sorted_w, reverse, scratch, status, s);
}

}  // namespace moe
