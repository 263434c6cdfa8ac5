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
// Two launches:
//   1. align_hist: each CTA counts its chunk of slots per expert (shared-memory
//      atomics; the counts are order-free) into chunk_hist[c][e];
//   2. align_scatter: each CTA derives offsets and its chunk's per-expert base
//      from chunk_hist, then ranks its slots in order, 512 at a time: within a
//      warp by __match_any_sync + popc of lower lanes, across warps by a
//      per-expert prefix over the warps' counts. A single-chunk problem runs
//      as one launch (the CTA makes its own histogram).
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 4096;   // slots per CTA

__device__ __forceinline__ int valid_expert(int e, int E) { return (e >= 0 && e < E) ? e : -1; }

__global__ void __launch_bounds__(kThreads) align_hist_kernel(const int32_t* __restrict__ idx,
                                                              long S, int E,
                                                              int32_t* __restrict__ chunk_hist,
                                                              int32_t* status) {
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += kThreads) hist[e] = 0;
  __syncthreads();
  const long lo = (long)blockIdx.x * kChunk;
  const long hi = min(S, lo + kChunk);
  bool bad = false;
  for (long s = lo + threadIdx.x; s < hi; s += kThreads) {
    const int e = __ldg(idx + s);
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else bad = true;
  }
  if (bad && status) atomicOr(status, MOE_STATUS_BAD_INDEX);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads) chunk_hist[(long)blockIdx.x * E + e] = hist[e];
}

// Shared layout: base[E] | off[E+1] | wcnt[kWarps][E]
__global__ void __launch_bounds__(kThreads) align_scatter_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ wts, long S, int k, int E,
    int nchunks, const int32_t* __restrict__ chunk_hist, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_ids,
    float* __restrict__ sorted_w, int32_t* __restrict__ reverse, int32_t* status) {
  extern __shared__ int sm[];
  int* base = sm;
  int* off = sm + E;
  int* wcnt = sm + 2 * E + 1;
  const int c = blockIdx.x;
  const long lo = (long)c * kChunk;
  const long hi = min(S, lo + kChunk);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // 1. per-expert totals (into off[]) and the base of this chunk (into base[])
  if (chunk_hist) {
    for (int e = tid; e < E; e += kThreads) {
      int before = 0, total = 0;
      for (int cc = 0; cc < nchunks; ++cc) {
        const int h = __ldg(chunk_hist + (long)cc * E + e);
        before += cc < c ? h : 0;
        total += h;
      }
      base[e] = before;
      off[e] = total;
    }
    __syncthreads();
  } else {   // single chunk: histogram here
    for (int e = tid; e < E; e += kThreads) { base[e] = 0; off[e] = 0; }
    __syncthreads();
    bool bad = false;
    for (long s = lo + tid; s < hi; s += kThreads) {
      const int e = __ldg(idx + s);
      if (e >= 0 && e < E) atomicAdd(&off[e], 1);
      else bad = true;
    }
    if (bad && status) atomicOr(status, MOE_STATUS_BAD_INDEX);
    __syncthreads();
  }

  // 2. exclusive scan of the totals over experts (warp 0; lane l owns a run of experts)
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int run = 0;
    for (int e = e0; e < e1; ++e) run += off[e];
    int incl = run;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    int acc = incl - run;
    for (int e = e0; e < e1; ++e) {
      const int cnt = off[e];
      if (c == 0) counts[e] = cnt;
      off[e] = acc;
      acc += cnt;
    }
    if (lane == 31) {
      off[E] = incl;
      if (c == 0) offsets[E] = incl;
    }
  }
  __syncthreads();
  if (c == 0)
    for (int e = tid; e < E; e += kThreads) offsets[e] = off[e];

  // 3. ordered ranking and scatter, kThreads slots per round
  for (long r0 = lo; r0 < hi; r0 += kThreads) {
    for (int i = tid; i < kWarps * E; i += kThreads) wcnt[i] = 0;
    __syncthreads();
    const long s = r0 + tid;
    const int e = s < hi ? valid_expert(__ldg(idx + s), E) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int x = tid; x < E; x += kThreads) {
      int run = base[x];
#pragma unroll 4
      for (int w = 0; w < kWarps; ++w) {
        const int cnt = wcnt[w * E + x];
        wcnt[w * E + x] = run;
        run += cnt;
      }
      base[x] = run;
    }
    __syncthreads();
    if (e >= 0) {
      const int p = off[e] + wcnt[warp * E + e] + rank;
      sorted_ids[p] = (int)(s / k);
      reverse[p] = (int)s;
      sorted_w[p] = __ldg(wts + s);
    }
    __syncthreads();
  }
}

}  // namespace

size_t align_scratch_bytes(int S, int E) {
  const size_t nchunks = (size_t)(S + kChunk - 1) / kChunk;
  return nchunks > 1 ? nchunks * (size_t)E * sizeof(int32_t) : 0;
}

int launch_align(const int32_t* idx, const float* w, int T, int k, int E, int32_t* counts,
                 int32_t* offsets, int32_t* sorted_ids, float* sorted_w, int32_t* reverse,
                 void* scratch, int32_t* status, cudaStream_t s) {
  const long S = (long)T * k;
  const int nchunks = (int)((S + kChunk - 1) / kChunk);
  const size_t smem = (size_t)(2 * E + 1 + kWarps * E) * sizeof(int);
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaFuncSetAttribute(align_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)((2 * MOE_MAX_EXPERTS + 1 + kWarps * MOE_MAX_EXPERTS) * sizeof(int)));
    attr_set[dev] = true;
  }
  int32_t* hist = nullptr;
  if (nchunks > 1) {
    hist = static_cast<int32_t*>(scratch);
    ProfScope ps("align_hist", s);
    align_hist_kernel<<<nchunks, kThreads, E * sizeof(int), s>>>(idx, S, E, hist, status);
    int rc = check_launch("align_hist");
    if (rc) return rc;
  }
  ProfScope ps("align_scatter", s);
  align_scatter_kernel<<<nchunks > 0 ? nchunks : 1, kThreads, smem, s>>>(
      idx, w, S, k, E, nchunks, hist, counts, offsets, sorted_ids, sorted_w, reverse, status);
  return check_launch("align_scatter");
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

// Device address of g_align_scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress, once per device with that device current, on the first
// call that needs it (that first call should come before any stream capture).
static int align_scratch_address(int32_t** out) {
  static std::mutex mu;
  static int32_t* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(MOE_ERR_UNSUPPORTED, "device ordinal %d above 63", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_align_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(MOE_ERR_CUDA, "cudaGetSymbolAddress(align scratch): %s", cudaGetErrorString(e));
    addr[dev] = static_cast<int32_t*>(p);
  }
  *out = addr[dev];
  return MOE_OK;
}

int launch_align_noalloc(const int32_t* idx, const float* w, int T, int k, int E, int32_t* counts,
                         int32_t* offsets, int32_t* sorted_ids, float* sorted_w, int32_t* reverse,
                         int32_t* status, cudaStream_t s) {
  const size_t need = align_scratch_bytes(T * k, E);
  if (need > sizeof(g_align_scratch))
    return fail(MOE_ERR_UNSUPPORTED,
                "align without workspace: T*k=%ld with E=%d needs %zu bytes of scratch, above the "
                "fixed %zu (ceil(T*k/4096)*E must not exceed %d)",
                (long)T * k, E, need, sizeof(g_align_scratch), MOE_ALIGN_NOALLOC_SCRATCH_INTS);
  int32_t* scratch = nullptr;
  int rc = align_scratch_address(&scratch);
  if (rc) return rc;
  return launch_align(idx, w, T, k, E, counts, offsets, sorted_ids, sorted_w, reverse, scratch, status, s);
}

}  // namespace moe
