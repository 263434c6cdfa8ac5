// C ABI: argument checks, workspace layout, launch sequencing, timing hooks.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"

namespace moe {

static thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return MOE_OK;
}

namespace {
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
}  // namespace

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

int num_sms() {
  static int cache[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 1;
  if (dev < 64) cache[dev] = n;
  return n;
}

namespace {
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <class F>
F driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<F>(p);
  return nullptr;
}
}  // namespace

unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || c == nullptr) {
    // nothing current on this thread yet: bind (and initialise) the primary context
    // of the runtime's current device, which the next launch would use anyway
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  }
  unsigned long long id = 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id + 1;   // never 0 for a real context
}

int ensure_smem_limit(const void* kernel, size_t bytes, const char* name) {
  static std::mutex mu;
  static std::map<std::pair<const void*, unsigned long long>, size_t> done;
  const unsigned long long ctx = current_context_id();
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = done.find({kernel, ctx});
    if (ctx != 0 && it != done.end() && it->second >= bytes) return MOE_OK;
  }
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: shared-memory limit %zu: %s", name, bytes, cudaGetErrorString(e));
  if (ctx != 0) {
    std::lock_guard<std::mutex> lk(mu);
    size_t& v = done[{kernel, ctx}];
    if (v < bytes) v = bytes;
  }
  return MOE_OK;
}

// ---- kernel timing -------------------------------------------------------------

namespace {
struct ProfRec {
  std::string name;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t pool_get() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
}  // namespace

ProfScope::ProfScope(const char* name, cudaStream_t s) : slot(-1), stream(s) {
  if (!g_prof_on) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  ProfRec r{name, pool_get(), pool_get()};
  cudaEventRecord(r.a, s);
  g_prof.push_back(r);
  slot = (int)g_prof.size() - 1;
}

ProfScope::~ProfScope() {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (slot < (int)g_prof.size()) cudaEventRecord(g_prof[slot].b, stream);
}

// ---- argument checks ---------------------------------------------------------------

namespace {

// Device-memory check of a tensor argument. The allocation ranges already seen
// to be device (or managed) memory are remembered, so the driver is asked once
// per allocation rather than once per argument of every call. Device virtual
// addresses are never handed out as host memory, so a remembered range stays
// device memory (possibly another allocation) for the life of the process.
typedef CUresult (*MemGetAddressRangeFn)(CUdeviceptr*, size_t*, CUdeviceptr);
struct DevRange {
  uintptr_t lo, hi;
};
std::mutex g_range_mu;
DevRange g_ranges[64];
int g_nranges = 0, g_next_range = 0;

bool is_device_ptr(const void* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  {
    std::lock_guard<std::mutex> lk(g_range_mu);
    for (int i = 0; i < g_nranges; ++i)
      if (a >= g_ranges[i].lo && a < g_ranges[i].hi) return true;
  }
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return false;
  static MemGetAddressRangeFn range_fn = driver_fn<MemGetAddressRangeFn>("cuMemGetAddressRange");
  CUdeviceptr base = 0;
  size_t size = 0;
  if (range_fn && range_fn(&base, &size, (CUdeviceptr)a) == CUDA_SUCCESS && size > 0) {
    std::lock_guard<std::mutex> lk(g_range_mu);
    g_ranges[g_next_range] = DevRange{(uintptr_t)base, (uintptr_t)base + size};
    g_next_range = (g_next_range + 1) % 64;
    if (g_nranges < 64) ++g_nranges;
  }
  return true;
}

#define REQUIRE(cond, ...)                                   \
  do {                                                       \
    if (!(cond)) return fail(MOE_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

// A tensor argument: non-null, 16-byte aligned, device memory (when it holds data).
int check_tensor(const void* p, long count, const char* name) {
  if (count <= 0) return MOE_OK;
  REQUIRE(p != nullptr, "%s is null", name);
  REQUIRE(aligned(p, 16), "%s is not 16-byte aligned", name);
  REQUIRE(is_device_ptr(p), "%s is not device memory", name);
  return MOE_OK;
}

int check_routing_dims(int T, int E, int k) {
  REQUIRE(T >= 0, "T must be >= 0 (got %d)", T);
  REQUIRE(E >= 1 && E <= MOE_MAX_EXPERTS, "E must be in [1, %d] (got %d)", MOE_MAX_EXPERTS, E);
  REQUIRE(k >= 1 && k <= MOE_MAX_TOPK && k <= E, "k must be in [1, min(E, %d)] (got k=%d, E=%d)",
          MOE_MAX_TOPK, k, E);
  REQUIRE((long)T * k < (1L << 31), "T*k must be below 2^31");
  REQUIRE((long)T * E < (1L << 40), "T*E too large");
  return MOE_OK;
}

int check_ffn_dims(int dtype, int H, int I) {
  REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, "dtype must be MOE_F32 or MOE_BF16 (got %d)", dtype);
  REQUIRE(H >= 1 && I >= 1, "H and I must be >= 1 (got H=%d, I=%d)", H, I);
  return MOE_OK;
}

struct FfnWs {
  void* act;
  void* staging;
  void* xs;
  int32_t* pos;
  int32_t* sync;
};

size_t dsize(int dtype) { return dtype == MOE_F32 ? 4 : 2; }

FfnWs carve_ffn(Carver& c, int dtype, int T, long S, int H, int I) {
  FfnWs w;
  w.act = c.take<char>((size_t)S * I * dsize(dtype));
  w.staging = c.take<char>((size_t)S * H * (staging_is_bf16(dtype, T, H, I) ? 2 : 4));
  const size_t xs = ffn_uses_tensor_cores(dtype, H, I) ? ffn_tc_extra_bytes(S, H) : 0;
  w.xs = xs ? c.take<char>(xs) : nullptr;
  w.pos = xs ? c.take<int32_t>(ffn_tc_pos_bytes(S) / sizeof(int32_t)) : nullptr;
  w.sync = c.take<int32_t>(kDecodeSyncWords);
  return w;
}

struct AlignWs {
  int32_t *counts, *offsets, *sorted_ids, *reverse;
  float* sorted_w;
  void* scratch;
};

AlignWs carve_align(Carver& c, long S, int E) {
  AlignWs w;
  w.counts = c.take<int32_t>(E);
  w.offsets = c.take<int32_t>(E + 1);
  w.sorted_ids = c.take<int32_t>(S);
  w.sorted_w = c.take<float>(S);
  w.reverse = c.take<int32_t>(S);
  const size_t sb = align_scratch_bytes(S, E);
  w.scratch = c.take<char>(sb ? sb : 1);
  return w;
}

int check_ws(void* ws, size_t have, size_t need) {
  if (need == 0) return MOE_OK;
  if (ws == nullptr || !aligned(ws, 256))
    return fail(MOE_ERR_WORKSPACE, "workspace is null or not 256-byte aligned");
  if (have < need)
    return fail(MOE_ERR_WORKSPACE, "workspace too small: %zu bytes given, %zu needed", have, need);
  if (!is_device_ptr(ws)) return fail(MOE_ERR_WORKSPACE, "workspace is not device memory");
  return MOE_OK;
}

int run_ffn(const void* hidden, const void* w13, const void* w2, int dtype, int T, int H, int I,
            int E, int k, const int32_t* counts, const int32_t* offsets, const int32_t* ids,
            const float* sw, const int32_t* rev, void* out, const FfnWs& w, int32_t* status,
            cudaStream_t s, bool may_drop = true, const float* logits = nullptr, int norm = 0,
            int32_t* sync = nullptr) {
  FfnArgs a{hidden, w13, w2, dtype, T, H, I, E, k, counts, offsets, ids, sw, rev,
            out, w.act, w.staging, w.xs, w.pos, status, logits, norm, sync};
  // caller routing may hold indices outside [0, E): their staging rows are zero (the
  // matrix-vector path has no staging rows: it skips dropped slots itself)
  if (may_drop && !ffn_gemv_applies(dtype, T, H, I, k)) {
    const int rc = launch_zero_dropped(offsets, E, (long)T * k, H, w.staging,
                                       staging_is_bf16(dtype, T, H, I) ? 2 : 4, s);
    if (rc) return rc;
  }
  return ffn_uses_tensor_cores(dtype, H, I) ? launch_ffn_tc(a, s) : launch_ffn_simt(a, s);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

MOE_API const char* moe_last_error(void) { return g_err; }

MOE_API const char* moe_version(void) { return "moe-gb300 0.1 (sm_103a, tcgen05 grouped FFN)"; }

MOE_API int moe_gating_softmax_topk(const float* logits, int T, int E, int k, int norm_topk_prob,
                                    float* weights, int32_t* indices, void* stream) {
  g_err[0] = 0;
  int rc;
  if ((rc = check_routing_dims(T, E, k))) return rc;
  if ((rc = check_tensor(logits, (long)T * E, "logits"))) return rc;
  if ((rc = check_tensor(weights, (long)T * k, "weights"))) return rc;
  if ((rc = check_tensor(indices, (long)T * k, "indices"))) return rc;
  return launch_gating(logits, T, E, k, norm_topk_prob != 0, weights, indices, (cudaStream_t)stream);
}

MOE_API int moe_gating_softmax_topk_bf16(const void* logits, int T, int E, int k, int norm_topk_prob,
                                         float* weights, int32_t* indices, void* stream) {
  g_err[0] = 0;
  int rc;
  if ((rc = check_routing_dims(T, E, k))) return rc;
  if ((rc = check_tensor(logits, (long)T * E, "logits"))) return rc;
  if ((rc = check_tensor(weights, (long)T * k, "weights"))) return rc;
  if ((rc = check_tensor(indices, (long)T * k, "indices"))) return rc;
  return launch_gating_bf16(logits, T, E, k, norm_topk_prob != 0, weights, indices, (cudaStream_t)stream);
}

MOE_API int moe_group_limited_topk(const float* scores, const float* bias, int T, int E, int k,
                                   int n_group, int topk_group, int method, float* weights,
                                   int32_t* indices, void* stream) {
  g_err[0] = 0;
  int rc;
  if ((rc = check_routing_dims(T, E, k))) return rc;
  REQUIRE(method == MOE_GROUP_TOPK_GREEDY || method == MOE_GROUP_TOPK_NOAUX_TC, "unknown method %d", method);
  REQUIRE(n_group >= 1 && n_group <= 32 && E % n_group == 0, "n_group must be in [1, 32] and divide E");
  REQUIRE(topk_group >= 1 && topk_group <= n_group, "topk_group must be in [1, n_group]");
  REQUIRE((long)k <= (long)topk_group * (E / n_group), "k must not exceed topk_group * E / n_group");
  REQUIRE(method != MOE_GROUP_TOPK_NOAUX_TC || E / n_group >= 2, "noaux_tc needs two experts per group");
  REQUIRE(method != MOE_GROUP_TOPK_NOAUX_TC || bias != nullptr, "noaux_tc needs a bias");
  if ((rc = check_tensor(scores, (long)T * E, "scores"))) return rc;
  if (bias && (rc = check_tensor(bias, E, "bias"))) return rc;
  if ((rc = check_tensor(weights, (long)T * k, "weights"))) return rc;
  if ((rc = check_tensor(indices, (long)T * k, "indices"))) return rc;
  return launch_group_limited_topk(scores, bias, T, E, k, n_group, topk_group,
                                   method == MOE_GROUP_TOPK_NOAUX_TC, weights, indices, (cudaStream_t)stream);
}

MOE_API int moe_indices_to_multihot(const int32_t* indices, const float* probs, int T, int k, int E,
                                    uint8_t* multihot, float* probs_in_multihot,
                                    int32_t* position_map, void* stream) {
  g_err[0] = 0;
  int rc;
  if ((rc = check_routing_dims(T, E, k))) return rc;
  if ((rc = check_tensor(indices, (long)T * k, "indices"))) return rc;
  if ((rc = check_tensor(probs, (long)T * k, "probs"))) return rc;
  if ((rc = check_tensor(multihot, (long)T * E, "multihot"))) return rc;
  if ((rc = check_tensor(probs_in_multihot, (long)T * E, "probs_in_multihot"))) return rc;
  if ((rc = check_tensor(position_map, (long)T * E, "position_map"))) return rc;
  return launch_indices_to_multihot(indices, probs, T, k, E, multihot, probs_in_multihot, position_map,
                                    (cudaStream_t)stream);
}

MOE_API int moe_multihot_to_indices(const float* probs_in_multihot, const int32_t* position_map,
                                    int T, int E, int k, float* probs, int32_t* indices_or_null,
                                    void* stream) {
  g_err[0] = 0;
  int rc;
  if ((rc = check_routing_dims(T, E, k))) return rc;
  if ((rc = check_tensor(probs_in_multihot, (long)T * E, "probs_in_multihot"))) return rc;
  if ((rc = check_tensor(position_map, (long)T * E, "position_map"))) return rc;
  if ((rc = check_tensor(probs, (long)T * k, "probs"))) return rc;
  if (indices_or_null && (rc = check_tensor(indices_or_null, (long)T * k, "indices"))) return rc;
  return launch_multihot_to_indices(probs_in_multihot, position_map, T, E, k, probs, indices_or_null,
                                    (cudaStream_t)stream);
}

MOE_API size_t moe_align_workspace_size(int T, int k, int E) {
  if (T < 0 || k < 1 || E < 1) return 0;
  return align_up(align_scratch_bytes((long)T * k, E), 256);
}

MOE_API int moe_align_by_expert(const int32_t* indices, const float* weights, int T, int k, int E,
                                int32_t* counts, int32_t* offsets, int32_t* sorted_token_ids,
                                float* sorted_weights, int32_t* reverse_indices, void* ws,
                                size_t ws_bytes, int32_t* status, void* stream) {
  g_err[0] = 0;
  int rc;
  if ((rc = check_routing_dims(T, E, k))) return rc;
  const long S = (long)T * k;
  if ((rc = check_tensor(indices, S, "indices"))) return rc;
  if ((rc = check_tensor(weights, S, "weights"))) return rc;
  if ((rc = check_tensor(counts, E, "counts"))) return rc;
  if ((rc = check_tensor(offsets, E + 1, "offsets"))) return rc;
  if ((rc = check_tensor(sorted_token_ids, S, "sorted_token_ids"))) return rc;
  if ((rc = check_tensor(sorted_weights, S, "sorted_weights"))) return rc;
  if ((rc = check_tensor(reverse_indices, S, "reverse_indices"))) return rc;
  if (status && (rc = check_tensor(status, 1, "status"))) return rc;
  if ((rc = check_ws(ws, ws_bytes, align_scratch_bytes(S, E)))) return rc;
  return launch_align(indices, weights, T, k, E, counts, offsets, sorted_token_ids, sorted_weights,
                      reverse_indices, ws, status, (cudaStream_t)stream);
}

MOE_API int moe_align_by_expert_noalloc(const int32_t* indices, const float* weights, int T, int k,
                                        int E, int32_t* counts, int32_t* offsets,
                                        int32_t* sorted_token_ids, float* sorted_weights,
                                        int32_t* reverse_indices, int32_t* status, void* stream) {
  g_err[0] = 0;
  int rc;
  if ((rc = check_routing_dims(T, E, k))) return rc;
  const long S = (long)T * k;
  if ((rc = check_tensor(indices, S, "indices"))) return rc;
  if ((rc = check_tensor(weights, S, "weights"))) return rc;
  if ((rc = check_tensor(counts, E, "counts"))) return rc;
  if ((rc = check_tensor(offsets, E + 1, "offsets"))) return rc;
  if ((rc = check_tensor(sorted_token_ids, S, "sorted_token_ids"))) return rc;
  if ((rc = check_tensor(sorted_weights, S, "sorted_weights"))) return rc;
  if ((rc = check_tensor(reverse_indices, S, "reverse_indices"))) return rc;
  if (status && (rc = check_tensor(status, 1, "status"))) return rc;
  return launch_align_noalloc(indices, weights, T, k, E, counts, offsets, sorted_token_ids,
                              sorted_weights, reverse_indices, status, (cudaStream_t)stream);
}

MOE_API size_t moe_grouped_ffn_workspace_size(int dtype, int T, int H, int I, int E, int k) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || k < 1) return 0;
  Carver c(nullptr);
  carve_ffn(c, dtype, T, (long)T * k, H, I);
  return align_up(c.used, 256);
}

MOE_API int moe_grouped_ffn(const void* hidden, const void* w13, const void* w2, int dtype, int T,
                            int H, int I, int E, int k, const int32_t* counts,
                            const int32_t* offsets, const int32_t* sorted_token_ids,
                            const float* sorted_weights, const int32_t* reverse_indices,
                            void* out, void* ws, size_t ws_bytes, int32_t* status, void* stream) {
  g_err[0] = 0;
  int rc;
  if ((rc = check_routing_dims(T, E, k))) return rc;
  if ((rc = check_ffn_dims(dtype, H, I))) return rc;
  const long S = (long)T * k;
  if ((rc = check_tensor(hidden, (long)T * H, "hidden"))) return rc;
  if ((rc = check_tensor(w13, (long)E * 2 * I * H, "w13"))) return rc;
  if ((rc = check_tensor(w2, (long)E * H * I, "w2"))) return rc;
  if ((rc = check_tensor(counts, E, "counts"))) return rc;
  if ((rc = check_tensor(offsets, E + 1, "offsets"))) return rc;
  if ((rc = check_tensor(sorted_token_ids, S, "sorted_token_ids"))) return rc;
  if ((rc = check_tensor(sorted_weights, S, "sorted_weights"))) return rc;
  if ((rc = check_tensor(reverse_indices, S, "reverse_indices"))) return rc;
  if ((rc = check_tensor(out, (long)T * H, "out"))) return rc;
  if (status && (rc = check_tensor(status, 1, "status"))) return rc;
  const size_t need = moe_grouped_ffn_workspace_size(dtype, T, H, I, E, k);
  if ((rc = check_ws(ws, ws_bytes, need))) return rc;
  Carver c(ws);
  const FfnWs w = carve_ffn(c, dtype, T, S, H, I);
  return run_ffn(hidden, w13, w2, dtype, T, H, I, E, k, counts, offsets, sorted_token_ids,
                 sorted_weights, reverse_indices, out, w, status, (cudaStream_t)stream);
}

namespace moe {
namespace {

size_t carve_bwd(Carver& c, FfnBwdArgs* a, long S, int H, int I, int E) {
  const long P = bwd_padded_rows(S, E);
  int32_t* poff = c.take<int32_t>((size_t)E + 1);
  void* xs = c.take<uint16_t>((size_t)P * H);
  void* dos = c.take<uint16_t>((size_t)P * H);
  void* dys = c.take<uint16_t>((size_t)P * H);
  float* gu = bwd_uses_fused(H) ? nullptr : c.take<float>((size_t)P * 2 * I);
  void* act = c.take<uint16_t>((size_t)P * I);
  void* dgu = c.take<uint16_t>((size_t)P * 2 * I);
  float* dwp = c.take<float>((size_t)P * 2 * ((I + 127) / 128));
  float* staging = c.take<float>((size_t)S * H);
  if (a) {
    a->poff = poff;
    a->xs = xs;
    a->dos = dos;
    a->dys = dys;
    a->gu = gu;
    a->act = act;
    a->dgu = dgu;
    a->dwp = dwp;
    a->staging = staging;
  }
  return align_up(c.used, 256);
}

}  // namespace
}  // namespace moe

MOE_API size_t moe_grouped_ffn_backward_workspace_size(int dtype, int T, int H, int I, int E, int k) {
  if (dtype != MOE_BF16 || T < 0 || H < 1 || I < 1 || E < 1 || k < 1) return 0;
  Carver c(nullptr);
  return carve_bwd(c, nullptr, (long)T * k, H, I, E);
}

MOE_API int moe_grouped_ffn_backward(const void* hidden, const void* w13, const void* w2, int dtype, int T,
                                     int H, int I, int E, int k, const int32_t* counts,
                                     const int32_t* offsets, const int32_t* sorted_token_ids,
                                     const float* sorted_weights, const int32_t* reverse_indices,
                                     const void* d_out, void* d_hidden, void* d_w13, void* d_w2,
                                     float* d_weights_or_null, void* ws, size_t ws_bytes, int32_t* status,
                                     void* stream) {
  g_err[0] = 0;
  int rc;
  if ((rc = check_routing_dims(T, E, k))) return rc;
  if ((rc = check_ffn_dims(dtype, H, I))) return rc;
  if (dtype != MOE_BF16 || !ffn_uses_tensor_cores(dtype, H, I))
    return fail(MOE_ERR_UNSUPPORTED, "the FFN backward runs bf16 with H %% 64 == 0 and I %% 64 == 0 only");
  const long S = (long)T * k;
  if ((rc = check_tensor(hidden, (long)T * H, "hidden"))) return rc;
  if ((rc = check_tensor(w13, (long)E * 2 * I * H, "w13"))) return rc;
  if ((rc = check_tensor(w2, (long)E * H * I, "w2"))) return rc;
  if ((rc = check_tensor(counts, E, "counts"))) return rc;
  if ((rc = check_tensor(offsets, E + 1, "offsets"))) return rc;
  if ((rc = check_tensor(sorted_token_ids, S, "sorted_token_ids"))) return rc;
  if ((rc = check_tensor(sorted_weights, S, "sorted_weights"))) return rc;
  if ((rc = check_tensor(reverse_indices, S, "reverse_indices"))) return rc;
  if ((rc = check_tensor(d_out, (long)T * H, "d_out"))) return rc;
  if ((rc = check_tensor(d_hidden, (long)T * H, "d_hidden"))) return rc;
  if ((rc = check_tensor(d_w13, (long)E * 2 * I * H, "d_w13"))) return rc;
  if ((rc = check_tensor(d_w2, (long)E * H * I, "d_w2"))) return rc;
  if (d_weights_or_null && (rc = check_tensor(d_weights_or_null, S, "d_weights"))) return rc;
  if (status && (rc = check_tensor(status, 1, "status"))) return rc;
  const size_t need = moe_grouped_ffn_backward_workspace_size(dtype, T, H, I, E, k);
  if ((rc = check_ws(ws, ws_bytes, need))) return rc;
  if (T == 0) {   // no rows: the weight gradients are zero
    cudaError_t e = cudaMemsetAsync(d_w13, 0, (size_t)E * 2 * I * H * 2, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(d_w2, 0, (size_t)E * H * I * 2, (cudaStream_t)stream);
    return e == cudaSuccess ? MOE_OK : fail(MOE_ERR_CUDA, "zeroing weight gradients: %s", cudaGetErrorString(e));
  }
  FfnBwdArgs a{};
  a.hidden = hidden;
  a.w13 = w13;
  a.w2 = w2;
  a.d_out = d_out;
  a.T = T;
  a.H = H;
  a.I = I;
  a.E = E;
  a.k = k;
  a.counts = counts;
  a.offsets = offsets;
  a.sorted_ids = sorted_token_ids;
  a.sorted_w = sorted_weights;
  a.reverse = reverse_indices;
  a.d_hidden = d_hidden;
  a.d_w13 = d_w13;
  a.d_w2 = d_w2;
  a.d_weights = d_weights_or_null;
  a.status = status;
  Carver c(ws);
  carve_bwd(c, &a, S, H, I, E);
  return launch_ffn_backward(a, (cudaStream_t)stream);
}

MOE_API size_t moe_layer_workspace_size(int dtype, int T, int H, int I, int E, int k) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || k < 1) return 0;
  const long S = (long)T * k;
  Carver c(nullptr);
  c.take<float>(S);
  c.take<int32_t>(S);
  carve_align(c, S, E);
  carve_ffn(c, dtype, T, S, H, I);
  return align_up(c.used, 256);
}

MOE_API int moe_layer_forward(const void* hidden, const float* router_logits, const void* w13,
                              const void* w2, int dtype, int T, int H, int I, int E, int k,
                              int norm_topk_prob, void* out, float* topk_weights_or_null,
                              int32_t* topk_indices_or_null, void* ws, size_t ws_bytes,
                              int32_t* status, void* stream) {
  g_err[0] = 0;
  int rc;
  if ((rc = check_routing_dims(T, E, k))) return rc;
  if ((rc = check_ffn_dims(dtype, H, I))) return rc;
  const long S = (long)T * k;
  if ((rc = check_tensor(hidden, (long)T * H, "hidden"))) return rc;
  if ((rc = check_tensor(router_logits, (long)T * E, "router_logits"))) return rc;
  if ((rc = check_tensor(w13, (long)E * 2 * I * H, "w13"))) return rc;
  if ((rc = check_tensor(w2, (long)E * H * I, "w2"))) return rc;
  if ((rc = check_tensor(out, (long)T * H, "out"))) return rc;
  if (topk_weights_or_null && (rc = check_tensor(topk_weights_or_null, S, "topk_weights"))) return rc;
  if (topk_indices_or_null && (rc = check_tensor(topk_indices_or_null, S, "topk_indices"))) return rc;
  if (status && (rc = check_tensor(status, 1, "status"))) return rc;
  const size_t need = moe_layer_workspace_size(dtype, T, H, I, E, k);
  if ((rc = check_ws(ws, ws_bytes, need))) return rc;
  if (T == 0) return MOE_OK;

  cudaStream_t s = (cudaStream_t)stream;
  Carver c(ws);
  float* tw = c.take<float>(S);
  int32_t* ti = c.take<int32_t>(S);
  if (topk_weights_or_null) tw = topk_weights_or_null;
  if (topk_indices_or_null) ti = topk_indices_or_null;
  const AlignWs al = carve_align(c, S, E);
  const FfnWs fw = carve_ffn(c, dtype, T, S, H, I);

  const bool small = route_is_small(T, k);
  if (small) {
    if ((rc = launch_route_small(router_logits, T, E, k, norm_topk_prob != 0, tw, ti, al.counts, al.offsets,
                                 al.sorted_ids, al.sorted_w, al.reverse, status, fw.sync, s)))
      return rc;
  } else {
    if ((rc = launch_gating(router_logits, T, E, k, norm_topk_prob != 0, tw, ti, s))) return rc;
    if ((rc = launch_align(ti, tw, T, k, E, al.counts, al.offsets, al.sorted_ids, al.sorted_w,
                           al.reverse, al.scratch, status, s)))
      return rc;
  }
  // the layer's own gating only produces indices in [0, E): no slot is dropped. The
  // logits let the decode kernels start on the experts' weights before routing ends;
  // the words the small-batch routing kernel zeroes are the decode FFN's counters.
  return run_ffn(hidden, w13, w2, dtype, T, H, I, E, k, al.counts, al.offsets, al.sorted_ids,
                 al.sorted_w, al.reverse, out, fw, status, s, /*may_drop=*/false, router_logits,
                 norm_topk_prob != 0, small ? fw.sync : nullptr);
}

MOE_API int moe_gather_rows(const void* hidden, const int32_t* sorted_token_ids, const int32_t* offsets,
                            int dtype, int T, int H, int E, int k, void* x_sorted, void* stream) {
  g_err[0] = 0;
  int rc;
  if ((rc = check_routing_dims(T, E, k))) return rc;
  REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, "dtype must be MOE_F32 or MOE_BF16 (got %d)", dtype);
  REQUIRE(H >= 1, "H must be >= 1 (got %d)", H);
  const long S = (long)T * k;
  if ((rc = check_tensor(hidden, (long)T * H, "hidden"))) return rc;
  if ((rc = check_tensor(sorted_token_ids, S, "sorted_token_ids"))) return rc;
  if ((rc = check_tensor(offsets, E + 1, "offsets"))) return rc;
  if ((rc = check_tensor(x_sorted, S * H, "x_sorted"))) return rc;
  if (S == 0) return MOE_OK;
  return launch_gather_rows(hidden, sorted_token_ids, offsets, E, H * (int)dsize(dtype), x_sorted, nullptr,
                            (cudaStream_t)stream);
}

MOE_API size_t moe_ep_receive_workspace_size(int G, int E_local) {
  if (G < 1 || E_local < 1) return 0;
  return align_up(ep_receive_workspace_bytes(G, E_local), 256);
}

MOE_API int moe_ep_receive_index(const int32_t* recv_counts, int G, int E_local, int R, int32_t* local_counts,
                                 int32_t* local_offsets, int32_t* perm, void* ws, size_t ws_bytes, void* stream) {
  g_err[0] = 0;
  int rc;
  REQUIRE(G >= 1 && E_local >= 1 && E_local <= MOE_MAX_EXPERTS, "need G >= 1 and 1 <= E_local <= %d",
          MOE_MAX_EXPERTS);
  REQUIRE((long)G * E_local <= 65536, "G * E_local must not exceed 65536");
  REQUIRE(R >= 0, "R must be >= 0");
  if ((rc = check_tensor(recv_counts, (long)G * E_local, "recv_counts"))) return rc;
  if ((rc = check_tensor(local_counts, E_local, "local_counts"))) return rc;
  if ((rc = check_tensor(local_offsets, E_local + 1, "local_offsets"))) return rc;
  if ((rc = check_tensor(perm, R, "perm"))) return rc;
  if ((rc = check_ws(ws, ws_bytes, ep_receive_workspace_bytes(G, E_local)))) return rc;
  return launch_ep_receive_index(recv_counts, G, E_local, local_counts, local_offsets, perm, ws,
                                 (cudaStream_t)stream);
}

MOE_API size_t moe_ep_combine_workspace_size(int T, int k) {
  if (T < 0 || k < 1) return 0;
  return align_up((size_t)T * k * sizeof(int32_t), 256);
}

MOE_API int moe_ep_combine(const void* y_sorted, const float* topk_weights, const int32_t* reverse_indices,
                           const int32_t* offsets, int dtype, int T, int k, int H, int E, void* out, void* ws,
                           size_t ws_bytes, void* stream) {
  g_err[0] = 0;
  int rc;
  if ((rc = check_routing_dims(T, E, k))) return rc;
  REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, "dtype must be MOE_F32 or MOE_BF16 (got %d)", dtype);
  REQUIRE(H >= 1, "H must be >= 1 (got %d)", H);
  const long S = (long)T * k;
  if ((rc = check_tensor(y_sorted, S * H, "y_sorted"))) return rc;
  if ((rc = check_tensor(topk_weights, S, "topk_weights"))) return rc;
  if ((rc = check_tensor(reverse_indices, S, "reverse_indices"))) return rc;
  if ((rc = check_tensor(offsets, E + 1, "offsets"))) return rc;
  if ((rc = check_tensor(out, (long)T * H, "out"))) return rc;
  if ((rc = check_ws(ws, ws_bytes, (size_t)S * sizeof(int32_t)))) return rc;
  if (S == 0) return MOE_OK;
  return launch_ep_combine(y_sorted, topk_weights, reverse_indices, offsets, dtype, T, k, H, E, out,
                           static_cast<int32_t*>(ws), (cudaStream_t)stream);
}

MOE_API uint64_t moe_set_wait_limit_ns(uint64_t ns) {
  return g_wait_ns.exchange(ns ? ns : kDefaultWaitNs);
}

MOE_API int moe_profiler_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = on != 0;
  return MOE_OK;
}

MOE_API int moe_profiler_report(char* buf, size_t len) {
  std::map<std::string, std::pair<long, double>> agg;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (auto& r : g_prof) {
      float ms = 0.f;
      cudaEventSynchronize(r.b);
      if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
        cudaGetLastError();
        ms = 0.f;
      }
      auto& a = agg[r.name];
      a.first += 1;
      a.second += ms;
      g_pool.push_back(r.a);
      g_pool.push_back(r.b);
    }
    g_prof.clear();
  }
  std::string js = "{";
  bool first = true;
  for (auto& kv : agg) {
    char tmp[256];
    snprintf(tmp, sizeof(tmp), "%s\"%s\": {\"launches\": %ld, \"total_ms\": %.6f}", first ? "" : ", ",
             kv.first.c_str(), kv.second.first, kv.second.second);
    js += tmp;
    first = false;
  }
  js += "}";
  if (buf && len) {
    const size_t n = js.size() < len - 1 ? js.size() : len - 1;
    memcpy(buf, js.data(), n);
    buf[n] = 0;
  }
  return (int)js.size();
}

}  // extern "C"
