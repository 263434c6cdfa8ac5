// Internal helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "moe.h"

namespace moe {

// ---- host side -------------------------------------------------------------

// Records a message for moe_last_error() and returns `code`.
int fail(int code, const char* fmt, ...);
// Turns the last CUDA launch error into MOE_ERR_CUDA (or MOE_OK).
int check_launch(const char* what);
// Limit (ns of global time) of the tensor-core FFN kernels' waits on their other
// roles; set by moe_set_wait_limit_ns, read when a kernel is launched.
uint64_t wait_limit_ns();
// Multiprocessor count of the current device (cached per device).
int num_sms();
// Process-unique id of the CUDA context current on this thread (the device's
// primary context is made current first when none is). 0 if it cannot be read.
unsigned long long current_context_id();
// Raises `kernel`'s dynamic shared-memory limit to at least `bytes` in the
// context current on this thread. Function attributes belong to a context, not
// to a device ordinal (a caller may run the library under its own driver
// context beside the primary one), so the setting is remembered per
// (kernel, context) and made again in a context that has not seen it.
int ensure_smem_limit(const void* kernel, size_t bytes, const char* name);
template <typename... KArgs>
int ensure_smem_limit(void (*kernel)(KArgs...), size_t bytes, const char* name) {
  return ensure_smem_limit(reinterpret_cast<const void*>(kernel), bytes, name);
}

// Row of a flat grid-stride index: i / d for d > 0. A shift when d is a power of
// two (sh = log2(d), from pow2_shift on the host), else an unsigned 32-bit
// division while i fits, else the 64-bit division (a long instruction sequence).
__device__ __forceinline__ long div_idx(long i, long d, int sh) {
  if (sh >= 0) return i >> sh;
  if (i <= 0x7fffffffL && d <= 0x7fffffffL) return (long)((uint32_t)i / (uint32_t)d);
  return i / d;
}
inline int pow2_shift(long d) { return (d > 0 && (d & (d - 1)) == 0) ? __builtin_ctzl((unsigned long)d) : -1; }

// Kernel timing hooks (no-ops unless moe_profiler_enable(1)).
struct ProfScope {
  ProfScope(const char* name, cudaStream_t s);
  ~ProfScope();
  int slot;
  cudaStream_t stream;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Bump allocator over a caller workspace; every carve is 256-byte aligned.
struct Carver {
  char* base;
  size_t used;
  explicit Carver(void* b) : base(static_cast<char*>(b)), used(0) {}
  template <class T>
  T* take(size_t count) {
    used = align_up(used, 256);
    T* p = base ? reinterpret_cast<T*>(base + used) : nullptr;
    used += count * sizeof(T);
    return p;
  }
};

// ---- launchers (one per translation unit) -------------------------------

int launch_gating(const float* logits, int T, int E, int k, int norm, float* w, int32_t* idx,
                  cudaStream_t s);
// Same top-k on bf16 logits (widened exactly to float32 on load).
int launch_gating_bf16(const void* logits, int T, int E, int k, int norm, float* w, int32_t* idx,
                       cudaStream_t s);
int launch_group_limited_topk(const float* scores, const float* bias, int T, int E, int k, int n_group,
                              int topk_group, int noaux, float* w, int32_t* idx, cudaStream_t s);
int launch_indices_to_multihot(const int32_t* idx, const float* probs, int T, int k, int E,
                               uint8_t* mh, float* pm, int32_t* pos, cudaStream_t s);
int launch_multihot_to_indices(const float* pm, const int32_t* pos, int T, int E, int k,
                               float* probs, int32_t* idx, cudaStream_t s);

size_t align_scratch_bytes(long S, int E);
// Words of the one-kernel decode FFN's counters (per active expert, and of FC1
// units taken; a layer workspace region that the small-batch routing kernel zeroes).
constexpr int kDecodeSyncWords = 65;
// Gating + align in one single-CTA launch, for at most 128 tokens whose T*k
// slots fit one align chunk; it also zeroes clear[0, kDecodeSyncWords) (when not null).
bool route_is_small(int T, int k);
int launch_route_small(const float* logits, int T, int E, int k, int norm, float* w, int32_t* idx,
                       int32_t* counts, int32_t* offsets, int32_t* sorted_ids, float* sorted_w,
                       int32_t* reverse, int32_t* status, int32_t* clear, cudaStream_t s);
int launch_align_noalloc(const int32_t* idx, const float* w, int T, int k, int E, int32_t* counts,
                         int32_t* offsets, int32_t* sorted_ids, float* sorted_w, int32_t* reverse,
                         int32_t* status, cudaStream_t s);
int launch_align(const int32_t* idx, const float* w, int T, int k, int E, int32_t* counts,
                 int32_t* offsets, int32_t* sorted_ids, float* sorted_w, int32_t* reverse,
                 void* scratch, int32_t* status, cudaStream_t s);

struct FfnArgs {
  const void* hidden;
  const void* w13;
  const void* w2;
  int dtype, T, H, I, E, k;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* sorted_ids;
  const float* sorted_w;
  const int32_t* reverse;
  void* out;
  void* act;        // [S, I] dtype
  void* staging;    // [S, H]: bf16 on the tensor-core prefill path (staging_is_bf16), else float32
  void* xs;         // [S, H] dtype: expert-sorted copy of hidden (the FC1 A operand)
  int32_t* pos;     // [S]: sorted row of every slot (tensor-core prefill path)
  int32_t* status;
  // Router logits [T, E] (or null): with them the decode FC1 kernel derives the
  // routing of its tokens itself (the same top-k and expert order as the routing
  // kernel, whose outputs it then waits for only before FC2 may start).
  const float* logits;
  int norm;
  // kDecodeSyncWords words zeroed by the routing kernel launched just before (or
  // null): the per-expert FC1 counters of the one-kernel decode FFN (ffn_gemv.cu).
  int32_t* sync;
};

// bf16 matrix [rows, cols] row-major as a TMA tensor map: box = box_rows x 64
// columns, 128-byte swizzle, zero fill out of bounds.
int make_tmap(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);
// Row-major [rows, cols] matrix of 4- or 2-byte elements as a TMA tensor map whose
// box is box_rows rows x 128 bytes, 128-byte swizzle, zero fill out of bounds
// (cols * elem_bytes a multiple of 16, base 16-byte aligned).
int make_tmap_rows128(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, int elem_bytes,
                      uint32_t box_rows);
// x_sorted[p] = hidden[sorted_ids[p]] for p < offsets[E] (rows of row_bytes, a multiple of 16).
int launch_gather_rows(const void* hidden, const int32_t* sorted_ids, const int32_t* offsets, int E, int row_bytes,
                       void* xs, int32_t* status, cudaStream_t s);
// Expert-parallel index work (expert_parallel.cu).
size_t ep_receive_workspace_bytes(int G, int El);
int launch_ep_receive_index(const int32_t* recv_counts, int G, int El, int32_t* counts, int32_t* offsets,
                            int32_t* perm, void* ws, cudaStream_t s);
int launch_ep_combine(const void* y, const float* w, const int32_t* reverse, const int32_t* offsets, int dtype,
                      int T, int k, int H, int E, void* out, int32_t* pos, cudaStream_t s);
// Token-count threshold at or below which the weight-streaming decode kernels run.
constexpr int kDecodeMaxTokens = 64;
int launch_ffn_decode(const FfnArgs& a, cudaStream_t s);
// Batches of at most kGemvMaxTokens tokens: matrix-vector products on the CUDA
// cores with the combine folded into FC2 (ffn_gemv.cu); token rows and
// activation rows must fit kGemvSmemMax bytes of shared memory.
constexpr int kGemvMaxTokens = 2;
constexpr size_t kGemvSmemMax = 96 * 1024;
bool ffn_gemv_applies(int dtype, int T, int H, int I, int k);
int launch_ffn_gemv(const FfnArgs& a, cudaStream_t s);
// FC1 and FC2 on 2-SM clusters (tcgen05 cta_group::2), given the five tensor
// maps (A: 128-row boxes of x_sorted / act; B: 128-row boxes of w13 / w2;
// S2: 32-row boxes of act for FC2's swapped remainder tiles).
int launch_ffn_pair_gemms(const FfnArgs& a, const CUtensorMap& tA1, const CUtensorMap& tB1,
                          const CUtensorMap& tA2, const CUtensorMap& tB2, const CUtensorMap& tS2,
                          cudaStream_t s);

// Backward of the grouped FFN and the k-sum (bf16, tensor cores; ffn_bwd.cu).
struct FfnBwdArgs {
  const void* hidden;
  const void* w13;
  const void* w2;
  const void* d_out;
  int T, H, I, E, k;
  const int32_t* counts;
  const int32_t* offsets;
  const int32_t* sorted_ids;
  const float* sorted_w;
  const int32_t* reverse;
  void* d_hidden;   // [T, H] bf16
  void* d_w13;      // [E, 2I, H] bf16
  void* d_w2;       // [E, H, I] bf16
  float* d_weights; // [T, k] or null
  // workspace
  int32_t* poff;    // [E + 1]
  void* xs;         // [P, H] bf16, P = bwd_padded_rows(S, E)
  void* dos;        // [P, H] bf16
  void* dys;        // [P, H] bf16
  float* gu;        // [P, 2I] (separate recompute / dA path only, else null)
  void* act;        // [P, I] bf16
  void* dgu;        // [P, 2I] bf16
  float* dwp;       // [P, 2 ceil(I / 128)]: one partial per feature tile and epilogue half
  float* staging;   // [S, H]
  int32_t* status;
};
long bwd_padded_rows(long S, int E);
// FC1 recompute and dA in one kernel (no gu buffer) for this H.
bool bwd_uses_fused(int H);
int launch_ffn_backward(const FfnBwdArgs& a, cudaStream_t s);

bool ffn_uses_tensor_cores(int dtype, int H, int I);
size_t ffn_tc_extra_bytes(long S, int H);
size_t ffn_tc_pos_bytes(long S);
int launch_ffn_tc(const FfnArgs& a, cudaStream_t s);
int launch_ffn_simt(const FfnArgs& a, cudaStream_t s);
// The FFN's weighted slot rows ([S, H] staging) are bf16 on the tensor-core
// prefill path (bf16, T above the decode threshold) and float32 otherwise.
bool staging_is_bf16(int dtype, int T, int H, int I);
// Zeroes the staging rows (elem_bytes each) when the align step dropped slots (offsets[E] < S).
int launch_zero_dropped(const int32_t* offsets, int E, long S, int H, void* staging, int elem_bytes,
                        cudaStream_t s);
// out[t] = sum_j staging[t*k + j] (j ascending, fp32), rounded once to `dtype`.
int launch_combine(const void* staging, int staging_bf16, int T, int k, int H, int dtype, void* out,
                   cudaStream_t s);

// Launch with programmatic stream serialization (PDL): the kernel may start while
// the previous kernel on the stream is still running; it must execute
// pdl_wait() before touching anything that kernel writes, and every kernel
// calls pdl_trigger() only after its own pdl_wait(), so that everything two or
// more launches back is complete whenever a kernel starts.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- device side -----------------------------------------------------------

// One whole 32-byte sector per access (256-bit vector load / store). A warp
// whose lanes each move 16 bytes of different rows touches half of 32
// sectors per instruction; these keep every sector whole. The address must
// be 32-byte aligned (workspace buffers, rows a multiple of 32 bytes long).
__device__ __forceinline__ void st_v8(void* p, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void st_v8(float* p, const float (&v)[8]) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(v[0]), "f"(v[1]),
               "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}
__device__ __forceinline__ void ld_v8(const void* p, uint32_t (&v)[8]) {
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "l"(p)
               : "memory");
}

// Wait until the kernels this one depends on (programmatically) have completed
// and their writes are visible; returns at once without such a dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel on the stream to start launching.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

template <class T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// silu(z) = z / (1 + e^-z); e^-z overflows to +inf for very negative z, giving -0.
__device__ __forceinline__ float silu(float z) { return z / (1.0f + __expf(-z)); }

}  // namespace moe
