// Declarations shared by the translation units of the library (not public).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

// Permute: one block handles a chunk of this many (token, slot) pairs.
constexpr int kPermChunk = 1024;
constexpr int kPermThreads = 512;

// The workspace's sched region: kSchedCounters grouped-GEMM work counters (FC1 pair,
// FC1 single, FC2 pair, FC2 single: a claim counter and a finished-CTA count each), then,
// for the launch that runs both GEMMs, one FC1-tiles-finished counter per group. The
// permute step zeroes all of them every forward.
constexpr int kSchedCounters = 8;

// Grouped GEMM tiling.
constexpr int kTileRows = 128;    // token rows of a full (token-major) tile
constexpr int kFc1Cols = 128;     // FC1 output channels per tile (gate and up each)
constexpr int kFc2Cols = 256;     // FC2 output channels per tile

// Narrow weight-major tiles. In a launch whose groups average at most kNarrowRows rows
// (T * k <= kNarrowRows * E: decode batches), a single-SM group of at most kNarrowRows rows
// is tiled by 128 weight rows instead of 256 (FC1: 64 gate + 64 up rows of kFc1NarrowCols
// channels; FC2: kFc2NarrowCols channels), each pipeline stage carrying two adjacent K
// blocks of them. A CTA then streams half as many weight rows at once, 256 contiguous bytes
// of each per stage: a bare TMA stream of [128, 1536, 2048] bf16 weights ran 5% faster so
// than 256 rows x 128 bytes on GB300. Measured on whole layers, this took 1% off the
// decode batches; in launches of larger groups it cost 2-4% (the x rows are re-read once
// per half-width tile), hence the launch-level rule. Returns the narrow row limit, 0 for
// none.
constexpr int kNarrowRows = 32;
constexpr int kFc1NarrowCols = 64;
constexpr int kFc2NarrowCols = 128;
inline int narrow_max_rows(const moe_problem& p) {
  return p.T * p.k <= static_cast<int64_t>(kNarrowRows) * p.E ? kNarrowRows : 0;
}

// Which GEMM kernel tiles the groups. When the routed groups average at least one full
// CTA-pair unit (T * k >= 256 * E), the CTA-pair kernel takes every group (groups of
// fewer than 256 rows become its masked or weight-major units) and the single-SM kernel
// is not launched; otherwise every group goes to the single-SM kernel and the pair kernel
// is not launched. (Measured: at 128 rows per expert the single-SM kernel is 11-17%
// faster, at 512 and 1024 the pair kernel 3% and 9%.) Returns the fewest rows of a group
// in the pair kernel's list.
inline int pair_min_rows(const moe_problem& p) {
  return p.T * p.k >= static_cast<int64_t>(2 * kTileRows) * p.E ? 1 : INT32_MAX;
}

// Fills the layout; returns false when the problem is outside the envelope.
bool compute_layout(const moe_problem& p, moe_ws_layout* out);

// Records a message for moe_last_error() and returns the status.
moe_status set_error(moe_status s, const char* fmt, ...);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// ---- launchers (each returns MOE_OK or MOE_ERR_CUDA; arguments already validated)

moe_status launch_route(const float* logits, int64_t T, const float* bias,
                        const moe_route_params& p, int32_t* ids, float* scales,
                        cudaStream_t s);

// Experts [e_lo, e_hi) are this call's (all of them: 0, E). Routed weights hold those
// experts only (plane g - e_lo for expert g).
moe_status launch_permute(const moe_problem& p, const moe_ws_layout& L, const void* x,
                          const int32_t* ids, int e_lo, int e_hi, char* ws, cudaStream_t s);

moe_status launch_fc1(const moe_problem& p, const moe_ws_layout& L, const void* w13,
                      const void* w13_s, int e_lo, int e_hi, char* ws, cudaStream_t s);

moe_status launch_fc2(const moe_problem& p, const moe_ws_layout& L, const void* w2,
                      const void* w2_s, int e_lo, int e_hi, char* ws, cudaStream_t s);

// FC1 then FC2 of one forward. When the single-SM kernel tiles the groups, one persistent
// launch runs both work lists (FC2 tiles wait for their group's FC1 tiles); at CTA-pair
// sizes, the two launches of launch_fc1 and launch_fc2.
moe_status launch_fc12(const moe_problem& p, const moe_ws_layout& L, const void* w13,
                       const void* w13_s, const void* w2, const void* w2_s, int e_lo, int e_hi,
                       char* ws, cudaStream_t s);

// shared_gate: fp32 [T] gate logits of the shared expert (weight sigmoid) or NULL (1).
moe_status launch_finalize(const moe_problem& p, const moe_ws_layout& L, const float* scales,
                           const float* shared_gate, void* y, const char* ws, cudaStream_t s);

// Device failure-path self-test (selftest.cu): status = the workspace status words.
moe_status launch_wait_selftest(int32_t* status, cudaStream_t s);

// Routing fused into the gate's epilogue (moe_gate_route); arguments as for moe_route.
struct GateRouteArgs {
  moe_route_params params;
  const float* bias;
  int32_t* ids;
  float* scales;
};

// logits may be NULL when `route` is given (the routed logits are then not written).
moe_status launch_gate(const void* x, const void* wg, int64_t T, int H, int E, int n_shared,
                       float* logits, float* shared_logits, int32_t* status, cudaStream_t s,
                       const GateRouteArgs* route = nullptr);

moe_status launch_cast_f32_bf16(const float* in, void* out, int64_t n, cudaStream_t s);

}  // namespace moe
