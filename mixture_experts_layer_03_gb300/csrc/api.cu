// C ABI entry points: argument validation on the host, workspace layout, and the
// launch sequence of the forward. Nothing here allocates device memory.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"

namespace moe {

namespace {
thread_local char g_err[512] = {0};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int32_t problem_reason(const moe_problem& p) {
  if (p.T < 0 || p.T > (int64_t{1} << 24)) return MOE_REASON_T_RANGE;
  if (p.E < 1 || p.E > 256) return MOE_REASON_E_RANGE;
  if (p.k < 1 || p.k > 8) return MOE_REASON_TOPK_RANGE;
  if (p.H < 64 || p.H % 64 != 0 || p.H > 32768) return MOE_REASON_H_ALIGN;
  if (p.I < 64 || p.I % 64 != 0 || p.I > 65536) return MOE_REASON_I_ALIGN;
  if (p.shared_I < 0 || p.shared_I % 64 != 0 || p.shared_I > 65536) return MOE_REASON_SHARED_I_ALIGN;
  const int64_t rows = p.T * p.k + (p.shared_I > 0 ? p.T : 0);
  if (rows >= (int64_t{1} << 31)) return MOE_REASON_ROWS;
  return MOE_REASON_OK;
}

int32_t route_reason(int64_t T, const moe_route_params& r) {
  if (T < 0 || T > (int64_t{1} << 31) / 8) return MOE_REASON_T_RANGE;
  if (r.num_experts < 1 || r.num_experts > 256) return MOE_REASON_E_RANGE;
  if (r.top_k < 1 || r.top_k > 8 || r.top_k > r.num_experts) return MOE_REASON_TOPK_RANGE;
  switch (r.method) {
    case MOE_ROUTE_DEFAULT:
    case MOE_ROUTE_RENORMALIZE:
    case MOE_ROUTE_LLAMA4:
    case MOE_ROUTE_RENORMALIZE_NAIVE:
    case MOE_ROUTE_MINIMAX2:
    case MOE_ROUTE_SIGMOID_RENORM:
      return MOE_REASON_OK;
    case MOE_ROUTE_DEEPSEEKV3: {
      // Fused-routing limits of the TensorRT-LLM MoE page, section "融合算子与回退阈值":
      // top_k <= 8, E <= 256, experts per group <= 32, experts per group * topk_group <= 256.
      if (r.n_group < 1 || r.n_group > 32 || r.num_experts % r.n_group != 0) return MOE_REASON_GROUPS;
      const int epg = r.num_experts / r.n_group;
      if (epg < 2 || epg > 32) return MOE_REASON_GROUPS;
      if (r.topk_group < 1 || r.topk_group > r.n_group) return MOE_REASON_GROUPS;
      if (epg * r.topk_group > 256 || r.top_k > epg * r.topk_group) return MOE_REASON_GROUPS;
      return MOE_REASON_OK;
    }
    case MOE_ROUTE_GROUPED_TOPK: {
      // vLLM GroupedTopKRouter: k / topk_group experts from each of topk_group groups. One
      // warp lane scores each group, hence n_group <= 32.
      if (r.n_group < 1 || r.n_group > 32 || r.num_experts % r.n_group != 0) return MOE_REASON_GROUPS;
      if (r.topk_group < 1 || r.topk_group > r.n_group) return MOE_REASON_GROUPS;
      if (r.top_k % r.topk_group != 0 || r.top_k / r.topk_group > r.num_experts / r.n_group)
        return MOE_REASON_GROUPS;
      return MOE_REASON_OK;
    }
    case MOE_ROUTE_GROUPED_TOPK_SOFTMAX:
      // A softmax taken inside each group sums to 1 in every group: the group choice would
      // be decided by tie-breaking alone.
      return MOE_REASON_DEGENERATE;
    default:
      return MOE_REASON_METHOD;
  }
}

// Per-device SM counts, filled on first use (any thread may fill one; all write the same).
std::atomic<int> g_sm_count[64];

}  // namespace

moe_status set_error(moe_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int n = g_sm_count[dev].load(std::memory_order_acquire);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    g_sm_count[dev].store(n, std::memory_order_release);
  }
  return n;
}

bool compute_layout(const moe_problem& p, moe_ws_layout* out) {
  if (problem_reason(p) != MOE_REASON_OK) return false;
  moe_ws_layout L;
  memset(&L, 0, sizeof(L));
  const int64_t P = p.T * p.k;
  const int G = p.E + (p.shared_I > 0 ? 1 : 0);
  const int nb = static_cast<int>((P + kPermChunk - 1) / kPermChunk);
  const int Ih = p.shared_I > p.I ? p.shared_I : p.I;
  const int64_t R = P + (p.shared_I > 0 ? p.T : 0);
  const size_t A = 1024;
  size_t o = 0;
  L.status = o;      o = align_up(o + 16, A);
  L.counts = o;      o = align_up(o + 4 * size_t(G), A);
  L.starts = o;      o = align_up(o + 4 * size_t(G), A);
  L.offsets = o;     o = align_up(o + 4 * size_t(p.E + 1), A);
  L.tile_off1 = o;   o = align_up(o + 8 * size_t(G + 1), A);
  L.tile_off2 = o;   o = align_up(o + 8 * size_t(G + 1), A);
  L.sched = o;       o = align_up(o + 4 * size_t(kSchedCounters + G), A);
  L.block_hist = o;  o = align_up(o + 4 * size_t(nb) * size_t(p.E), A);
  L.perm_src = o;    o = align_up(o + 4 * size_t(P), A);
  L.perm_inv = o;    o = align_up(o + 4 * size_t(P), A);
  L.x_perm = o;      o = align_up(o + 2 * size_t(R) * size_t(p.H), A);
  L.h = o;           o = align_up(o + 2 * size_t(R) * size_t(Ih), A);
  L.out_perm = o;    o = align_up(o + 2 * size_t(R) * size_t(p.H), A);
  L.total = o;
  L.rows = R;
  L.groups = G;
  L.n_chunks = nb;
  L.h_ld = Ih;
  *out = L;
  return true;
}

}  // namespace moe

using namespace moe;

namespace {

moe_status check_forward_common(const moe_problem* p, void* workspace, size_t ws_bytes,
                                moe_ws_layout* L) {
  if (!p) return set_error(MOE_ERR_INVALID_ARG, "problem is NULL");
  const int32_t reason = problem_reason(*p);
  if (reason != MOE_REASON_OK)
    return set_error(MOE_ERR_UNSUPPORTED, "problem outside the supported envelope (reason %d)", reason);
  compute_layout(*p, L);
  if (p->T == 0) return MOE_OK;
  if (!workspace) return set_error(MOE_ERR_INVALID_ARG, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(workspace) & 1023u) != 0)
    return set_error(MOE_ERR_INVALID_ARG, "workspace must be 1024-byte aligned");
  if (ws_bytes < L->total)
    return set_error(MOE_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", ws_bytes, L->total);
  return MOE_OK;
}

bool shared_args_ok(const moe_problem* p, const void* a, const void* b) {
  if (p->shared_I > 0) return a && b && aligned16(a) && aligned16(b);
  return true;
}

}  // namespace

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported problem";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_BAD_ID: return "device saw an expert id outside [0, E)";
    case MOE_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out";
    case MOE_ERR_NOT_IMPLEMENTED: return "not implemented";
  }
  return "unknown status";
}

const char* moe_last_error(void) { return g_err; }

moe_status moe_can_implement(const moe_problem* p, int32_t* reason) {
  if (!p) {
    if (reason) *reason = MOE_REASON_OK;
    return MOE_ERR_INVALID_ARG;
  }
  const int32_t r = problem_reason(*p);
  if (reason) *reason = r;
  return r == MOE_REASON_OK ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

size_t moe_workspace_bytes(const moe_problem* p) {
  moe_ws_layout L;
  if (!p || !compute_layout(*p, &L)) return 0;
  return L.total;
}

moe_status moe_workspace_layout(const moe_problem* p, moe_ws_layout* out) {
  if (!p || !out) return set_error(MOE_ERR_INVALID_ARG, "NULL argument");
  if (!compute_layout(*p, out)) return set_error(MOE_ERR_UNSUPPORTED, "problem outside the envelope");
  return MOE_OK;
}

moe_status moe_route(const float* logits, int64_t T, const float* bias, const moe_route_params* p,
                     int32_t* ids, float* scales, void* stream) {
  if (!p) return set_error(MOE_ERR_INVALID_ARG, "route params are NULL");
  const int32_t r = route_reason(T, *p);
  if (r == MOE_REASON_DEGENERATE)
    return set_error(MOE_ERR_UNSUPPORTED, "grouped top-k with softmax scoring: every group's score "
                     "is 1, so the group choice would rest on tie-breaking alone");
  if (r != MOE_REASON_OK) return set_error(MOE_ERR_UNSUPPORTED, "routing outside the envelope (reason %d)", r);
  if (T == 0) return MOE_OK;
  if (!logits || !ids || !scales) return set_error(MOE_ERR_INVALID_ARG, "NULL logits/ids/scales");
  if (!aligned16(logits) || !aligned16(ids) || !aligned16(scales) || (bias && !aligned16(bias)))
    return set_error(MOE_ERR_INVALID_ARG, "route pointers must be 16-byte aligned");
  if (bias && p->method == MOE_ROUTE_GROUPED_TOPK)
    return set_error(MOE_ERR_INVALID_ARG, "the grouped top-k routing takes no bias");
  return launch_route(logits, T, bias, *p, ids, scales, static_cast<cudaStream_t>(stream));
}

moe_status moe_permute(const moe_problem* p, const void* x, const int32_t* ids, void* workspace,
                       size_t ws_bytes, void* stream) {
  moe_ws_layout L;
  moe_status st = check_forward_common(p, workspace, ws_bytes, &L);
  if (st != MOE_OK || p->T == 0) return st;
  if (!x || !ids || !aligned16(x) || !aligned16(ids))
    return set_error(MOE_ERR_INVALID_ARG, "x/ids NULL or not 16-byte aligned");
  return launch_permute(*p, L, x, ids, 0, p->E, static_cast<char*>(workspace),
                        static_cast<cudaStream_t>(stream));
}

moe_status moe_fc1(const moe_problem* p, const void* w13, const void* w13_s, void* workspace,
                   size_t ws_bytes, void* stream) {
  moe_ws_layout L;
  moe_status st = check_forward_common(p, workspace, ws_bytes, &L);
  if (st != MOE_OK || p->T == 0) return st;
  if (!w13 || !aligned16(w13) || !shared_args_ok(p, w13_s, w13_s))
    return set_error(MOE_ERR_INVALID_ARG, "w13/w13_s NULL or not 16-byte aligned");
  return launch_fc1(*p, L, w13, w13_s, 0, p->E, static_cast<char*>(workspace),
                    static_cast<cudaStream_t>(stream));
}

moe_status moe_fc2(const moe_problem* p, const void* w2, const void* w2_s, void* workspace,
                   size_t ws_bytes, void* stream) {
  moe_ws_layout L;
  moe_status st = check_forward_common(p, workspace, ws_bytes, &L);
  if (st != MOE_OK || p->T == 0) return st;
  if (!w2 || !aligned16(w2) || !shared_args_ok(p, w2_s, w2_s))
    return set_error(MOE_ERR_INVALID_ARG, "w2/w2_s NULL or not 16-byte aligned");
  return launch_fc2(*p, L, w2, w2_s, 0, p->E, static_cast<char*>(workspace),
                    static_cast<cudaStream_t>(stream));
}

moe_status moe_fc1_fc2(const moe_problem* p, const void* w13, const void* w13_s, const void* w2,
                       const void* w2_s, void* workspace, size_t ws_bytes, void* stream) {
  moe_ws_layout L;
  moe_status st = check_forward_common(p, workspace, ws_bytes, &L);
  if (st != MOE_OK || p->T == 0) return st;
  if (!w13 || !aligned16(w13) || !w2 || !aligned16(w2))
    return set_error(MOE_ERR_INVALID_ARG, "w13/w2 NULL or not 16-byte aligned");
  if (!shared_args_ok(p, w13_s, w2_s))
    return set_error(MOE_ERR_INVALID_ARG, "shared expert weights NULL or not 16-byte aligned");
  return launch_fc12(*p, L, w13, w13_s, w2, w2_s, 0, p->E, static_cast<char*>(workspace),
                     static_cast<cudaStream_t>(stream));
}

moe_status moe_finalize(const moe_problem* p, const float* scales, void* y, void* workspace,
                        size_t ws_bytes, void* stream) {
  moe_ws_layout L;
  moe_status st = check_forward_common(p, workspace, ws_bytes, &L);
  if (st != MOE_OK || p->T == 0) return st;
  if (!scales || !y || !aligned16(scales) || !aligned16(y))
    return set_error(MOE_ERR_INVALID_ARG, "scales/y NULL or not 16-byte aligned");
  return launch_finalize(*p, L, scales, nullptr, y, static_cast<const char*>(workspace),
                         static_cast<cudaStream_t>(stream));
}

moe_status moe_gate(const void* x, const void* wg, int64_t T, int32_t H, int32_t E,
                    int32_t n_shared, float* routed_logits, float* shared_logits, void* stream) {
  if (T < 0 || T > (int64_t{1} << 31) / 8 || H < 64 || H % 64 != 0 || H > 32768 || E < 1 ||
      E > 256 || n_shared < 0 || n_shared > 1)
    return set_error(MOE_ERR_UNSUPPORTED, "gate shape outside the envelope (T %lld, H %d, E %d, "
                     "n_shared %d)", static_cast<long long>(T), H, E, n_shared);
  if (T == 0) return MOE_OK;
  if (!x || !wg || !routed_logits || (n_shared == 1 && !shared_logits))
    return set_error(MOE_ERR_INVALID_ARG, "NULL gate argument");
  if (!aligned16(x) || !aligned16(wg) || !aligned16(routed_logits) ||
      (shared_logits && !aligned16(shared_logits)))
    return set_error(MOE_ERR_INVALID_ARG, "gate pointers must be 16-byte aligned");
  return launch_gate(x, wg, T, H, E, n_shared, routed_logits, n_shared ? shared_logits : nullptr,
                     nullptr, static_cast<cudaStream_t>(stream));
}

moe_status moe_gate_route(const void* x, const void* wg, int64_t T, int32_t H, int32_t n_shared,
                          const float* bias, const moe_route_params* p, int32_t* ids,
                          float* scales, float* routed_logits, float* shared_logits,
                          void* stream) {
  if (!p) return set_error(MOE_ERR_INVALID_ARG, "route params are NULL");
  const int32_t E = p->num_experts;
  if (T < 0 || T > (int64_t{1} << 31) / 8 || H < 64 || H % 64 != 0 || H > 32768 || E < 1 ||
      E > 256 || n_shared < 0 || n_shared > 1)
    return set_error(MOE_ERR_UNSUPPORTED, "gate shape outside the envelope (T %lld, H %d, E %d, "
                     "n_shared %d)", static_cast<long long>(T), H, E, n_shared);
  const int32_t r = route_reason(T, *p);
  if (r == MOE_REASON_DEGENERATE)
    return set_error(MOE_ERR_UNSUPPORTED, "grouped top-k with softmax scoring: every group's score "
                     "is 1, so the group choice would rest on tie-breaking alone");
  if (r != MOE_REASON_OK) return set_error(MOE_ERR_UNSUPPORTED, "routing outside the envelope (reason %d)", r);
  if (T == 0) return MOE_OK;
  if (!x || !wg || !ids || !scales || (n_shared == 1 && !shared_logits))
    return set_error(MOE_ERR_INVALID_ARG, "NULL gate or routing argument");
  if (!aligned16(x) || !aligned16(wg) || !aligned16(ids) || !aligned16(scales) ||
      (routed_logits && !aligned16(routed_logits)) || (shared_logits && !aligned16(shared_logits)) ||
      (bias && !aligned16(bias)))
    return set_error(MOE_ERR_INVALID_ARG, "gate and routing pointers must be 16-byte aligned");
  if (bias && p->method == MOE_ROUTE_GROUPED_TOPK)
    return set_error(MOE_ERR_INVALID_ARG, "the grouped top-k routing takes no bias");
  GateRouteArgs ra;
  ra.params = *p;
  ra.bias = bias;
  ra.ids = ids;
  ra.scales = scales;
  return launch_gate(x, wg, T, H, E, n_shared, routed_logits, n_shared ? shared_logits : nullptr,
                     nullptr, static_cast<cudaStream_t>(stream), &ra);
}

moe_status moe_forward_partial(const moe_problem* p, int32_t e_lo, int32_t e_hi, const void* x,
                               const int32_t* ids, const float* scales, const void* w13,
                               const void* w2, const void* w13_s, const void* w2_s,
                               const float* shared_gate, void* y, void* workspace,
                               size_t ws_bytes, void* stream) {
  moe_ws_layout L;
  moe_status st = check_forward_common(p, workspace, ws_bytes, &L);
  if (st != MOE_OK || p->T == 0) return st;
  if (e_lo < 0 || e_hi > p->E || e_lo >= e_hi)
    return set_error(MOE_ERR_INVALID_ARG, "expert range [%d, %d) not inside [0, %d)", e_lo, e_hi, p->E);
  if (!x || !ids || !scales || !w13 || !w2 || !y)
    return set_error(MOE_ERR_INVALID_ARG, "NULL tensor argument");
  if (!aligned16(x) || !aligned16(ids) || !aligned16(scales) || !aligned16(w13) || !aligned16(w2) ||
      !aligned16(y))
    return set_error(MOE_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (!shared_args_ok(p, w13_s, w2_s))
    return set_error(MOE_ERR_INVALID_ARG, "shared expert weights NULL or not 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  if ((st = launch_permute(*p, L, x, ids, e_lo, e_hi, ws, s)) != MOE_OK) return st;
  if ((st = launch_fc12(*p, L, w13, w13_s, w2, w2_s, e_lo, e_hi, ws, s)) != MOE_OK) return st;
  return launch_finalize(*p, L, scales, shared_gate, y, ws, s);
}

moe_status moe_forward(const moe_problem* p, const void* x, const int32_t* ids, const float* scales,
                       const void* w13, const void* w2, const void* w13_s, const void* w2_s, void* y,
                       void* workspace, size_t ws_bytes, void* stream) {
  return moe_forward_partial(p, 0, p ? p->E : 0, x, ids, scales, w13, w2, w13_s, w2_s, nullptr,
                             y, workspace, ws_bytes, stream);
}

}  // extern "C"

// Scratch of moe_forward_static: one fixed array per GPU, in this library's device
// image. The extra 1024 bytes let the workspace start on a 1024-byte boundary.
static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES + 1024];

namespace {

std::mutex g_static_mu;
void* g_static_addr[64] = {nullptr};

// Device address of g_static_scratch on the current device, looked up once per device
// with that device current (the symbol's name is only a host-side stand-in).
moe_status static_scratch_base(char** base) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64)
    return set_error(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_static_scratch);
    if (e != cudaSuccess || !addr)
      return set_error(MOE_ERR_CUDA, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
    g_static_addr[dev] = addr;
  }
  const uintptr_t a = reinterpret_cast<uintptr_t>(g_static_addr[dev]);
  *base = reinterpret_cast<char*>((a + 1023u) & ~static_cast<uintptr_t>(1023u));
  return MOE_OK;
}

// Reads the status word at `status` after the work queued on `s`, then clears it.
moe_status read_status_word(void* status, cudaStream_t s, int32_t* flags) {
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, status, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, sizeof(v), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (flags) *flags = v;
  if (v & MOE_DEVICE_FLAG_TIMEOUT) return MOE_ERR_DEVICE_TIMEOUT;
  if (v & MOE_DEVICE_FLAG_BAD_ID) return MOE_ERR_DEVICE_BAD_ID;
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_forward_static(const moe_problem* p, const void* x, const int32_t* ids,
                              const float* scales, const void* w13, const void* w2,
                              const void* w13_s, const void* w2_s, void* y, void* stream) {
  if (!p) return set_error(MOE_ERR_INVALID_ARG, "problem is NULL");
  const int32_t reason = problem_reason(*p);
  if (reason != MOE_REASON_OK)
    return set_error(MOE_ERR_UNSUPPORTED, "problem outside the supported envelope (reason %d)", reason);
  moe_ws_layout L;
  compute_layout(*p, &L);
  if (p->T == 0) return MOE_OK;
  if (L.total > MOE_STATIC_SCRATCH_BYTES)
    return set_error(MOE_ERR_WORKSPACE_TOO_SMALL,
                     "problem needs %zu bytes of scratch; the static scratch holds %zu", L.total,
                     static_cast<size_t>(MOE_STATIC_SCRATCH_BYTES));
  if (!x || !ids || !scales || !w13 || !w2 || !y)
    return set_error(MOE_ERR_INVALID_ARG, "NULL tensor argument");
  if (!aligned16(x) || !aligned16(ids) || !aligned16(scales) || !aligned16(w13) || !aligned16(w2) ||
      !aligned16(y))
    return set_error(MOE_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (!shared_args_ok(p, w13_s, w2_s))
    return set_error(MOE_ERR_INVALID_ARG, "shared expert weights NULL or not 16-byte aligned");
  char* ws = nullptr;
  moe_status st = static_scratch_base(&ws);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The permute step clears the status word and the GEMM tile counters in the scratch.
  if ((st = launch_permute(*p, L, x, ids, 0, p->E, ws, s)) != MOE_OK) return st;
  if ((st = launch_fc12(*p, L, w13, w13_s, w2, w2_s, 0, p->E, ws, s)) != MOE_OK) return st;
  return launch_finalize(*p, L, scales, nullptr, y, ws, s);
}

moe_status moe_read_device_status(void* workspace, void* stream, int32_t* flags) {
  if (!workspace) return set_error(MOE_ERR_INVALID_ARG, "workspace is NULL");
  return read_status_word(workspace, static_cast<cudaStream_t>(stream), flags);
}

moe_status moe_static_read_device_status(void* stream, int32_t* flags) {
  char* ws = nullptr;
  const moe_status st = static_scratch_base(&ws);
  if (st != MOE_OK) return st;
  return read_status_word(ws, static_cast<cudaStream_t>(stream), flags);
}

moe_status moe_selftest_wait(void* workspace, void* stream) {
  if (!workspace) return set_error(MOE_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned16(workspace)) return set_error(MOE_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = cudaMemsetAsync(workspace, 0, 2 * sizeof(int32_t), s);
  if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
  return launch_wait_selftest(static_cast<int32_t*>(workspace), s);
}

moe_status moe_cast_f32_to_bf16(const float* in, void* out, int64_t n, void* stream) {
  if (n < 0) return set_error(MOE_ERR_INVALID_ARG, "negative length");
  if (n == 0) return MOE_OK;
  if (!in || !out) return set_error(MOE_ERR_INVALID_ARG, "NULL pointer");
  return launch_cast_f32_bf16(in, out, n, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
