// Step 1: routing. One warp per token; lane l holds experts l, l+32, ... (E <= 256).
//
// Methods (RoutingMethodType of the TensorRT-LLM MoE page, section "路由方法枚举"):
//   Default          softmax over all E, top-k, weights = the selected probabilities
//   Renormalize      top-k, softmax over the k selected logits
//   RenormalizeNaive softmax over all E, top-k, divide by the selected sum
//   SigmoidRenorm    sigmoid, top-k, divide by the selected sum
//   DeepSeekV3       noaux_tc (same page, section "DeepSeek-V3 的 noaux_tc"): sigmoid
//                    scores, + e_score_correction_bias for selection only, group score =
//                    sum of the top-2 biased scores, keep topk_group groups, top-k among
//                    their experts, weights = unbiased scores / (sum + 1e-20) * rsf.
//
// Selection keys are fp32 so ids are exact: the logit itself for the softmax and
// sigmoid methods (both maps are increasing), and fl32(fl32(sigmoid_fp64(l)) + b) for
// DeepSeekV3. Ties go to the lower expert index; slots are listed by descending key.
// Weights are computed in fp64 and rounded once to fp32.
#include <cfloat>
#include <cmath>
#include <cstdint>

#include "internal.h"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;
constexpr int kMaxPerLane = 8;    // 256 experts / 32 lanes
constexpr int kMaxTopK = 8;

struct KeyIdx {
  float key;
  int idx;    // INT32_MAX = no candidate
};

// a beats b: larger key, or equal key and lower index.
__device__ __forceinline__ bool beats(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

__device__ __forceinline__ KeyIdx warp_best(KeyIdx v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float ok = __shfl_xor_sync(0xffffffffu, v.key, off);
    int oi = __shfl_xor_sync(0xffffffffu, v.idx, off);
    if (beats(ok, oi, v.key, v.idx)) {
      v.key = ok;
      v.idx = oi;
    }
  }
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ double sigmoid_d(double l) { return 1.0 / (1.0 + exp(-l)); }

__global__ void __launch_bounds__(kRouteWarps * 32)
route_kernel(const float* __restrict__ logits, int64_t T, int E, const float* __restrict__ bias,
             int method, int k, int n_group, int topk_group, float rsf,
             int32_t* __restrict__ ids, float* __restrict__ scales) {
  __shared__ float s_key[kRouteWarps][256];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kRouteWarps + warp;
  if (t >= T) return;   // warp-uniform
  const float* row = logits + t * E;

  // Load: l = logit (non-finite -> -inf), key = selection key.
  float l[kMaxPerLane], key[kMaxPerLane];
  bool present[kMaxPerLane];
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int e = lane + 32 * i;
    present[i] = e < E;
    float v = present[i] ? row[e] : -INFINITY;
    if (!isfinite(v)) v = -INFINITY;
    l[i] = v;
    if (method == MOE_ROUTE_DEEPSEEKV3 && present[i]) {
      const float s32 = __double2float_rn(sigmoid_d(static_cast<double>(v)));
      key[i] = __fadd_rn(s32, bias ? bias[e] : 0.0f);
    } else {
      key[i] = v;
    }
  }

  if (method == MOE_ROUTE_DEEPSEEKV3) {
    // Group scores: lane g < n_group sums the top-2 keys of its group.
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
      if (present[i]) s_key[warp][lane + 32 * i] = key[i];
    __syncwarp();
    const int epg = E / n_group;
    float gscore = -INFINITY;
    int gidx = INT32_MAX;
    if (lane < n_group) {
      float a = -INFINITY, b = -INFINITY;   // a >= b: the two largest
      for (int j = 0; j < epg; ++j) {
        const float v = s_key[warp][lane * epg + j];
        if (v > a) {
          b = a;
          a = v;
        } else if (v > b) {
          b = v;
        }
      }
      gscore = __fadd_rn(a, b);
      gidx = lane;
    }
    // Keep topk_group groups: repeated warp argmax.
    uint32_t chosen = 0;
    bool taken = false;
    for (int r = 0; r < topk_group; ++r) {
      KeyIdx v = taken ? KeyIdx{-INFINITY, INT32_MAX} : KeyIdx{gscore, gidx};
      v = warp_best(v);
      if (v.idx == lane) taken = true;
      chosen |= 1u << v.idx;
    }
    // Experts outside the chosen groups cannot be selected.
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      if (present[i] && !((chosen >> (e / epg)) & 1u)) key[i] = -INFINITY;
    }
  }

  // Top-k by repeated warp argmax; every lane ends with the same sel_* arrays.
  int sel_idx[kMaxTopK];
  float sel_l[kMaxTopK];
  uint32_t taken_mask = 0;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    sel_idx[j] = 0;
    sel_l[j] = 0.f;
    if (j < k) {
      KeyIdx best{-INFINITY, INT32_MAX};
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        const int e = lane + 32 * i;
        if (present[i] && !((taken_mask >> i) & 1u) && beats(key[i], e, best.key, best.idx)) {
          best.key = key[i];
          best.idx = e;
        }
      }
      best = warp_best(best);
      const int owner = best.idx & 31;
      const int slot = best.idx >> 5;
      float lv = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i)
        if (i == slot) lv = l[i];
      lv = __shfl_sync(0xffffffffu, lv, owner);
      if (lane == owner) taken_mask |= 1u << slot;
      sel_idx[j] = best.idx;
      sel_l[j] = lv;
    }
  }

  // Weights in fp64.
  double w[kMaxTopK];
  if (method == MOE_ROUTE_DEFAULT || method == MOE_ROUTE_RENORMALIZE_NAIVE) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) m = fmaxf(m, l[i]);
    m = warp_max_f(m);
    double z = 0.0;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
      if (present[i]) z += exp(static_cast<double>(l[i]) - static_cast<double>(m));
    z = warp_sum_d(z);
    double psum = 0.0;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      w[j] = (j < k) ? exp(static_cast<double>(sel_l[j]) - static_cast<double>(m)) / z : 0.0;
      psum += w[j];
    }
    if (method == MOE_ROUTE_RENORMALIZE_NAIVE) {
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) w[j] /= psum;
    }
  } else if (method == MOE_ROUTE_RENORMALIZE) {
    const double m = static_cast<double>(sel_l[0]);
    double z = 0.0;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      w[j] = (j < k) ? exp(static_cast<double>(sel_l[j]) - m) : 0.0;
      z += w[j];
    }
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) w[j] /= z;
  } else {   // SigmoidRenorm, DeepSeekV3: unbiased sigmoid of the selected logits
    double z = 0.0;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      w[j] = (j < k) ? sigmoid_d(static_cast<double>(sel_l[j])) : 0.0;
      z += w[j];
    }
    if (method == MOE_ROUTE_DEEPSEEKV3) {
      const double denom = z + 1e-20;
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) w[j] = w[j] / denom * static_cast<double>(rsf);
    } else {
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) w[j] /= z;
    }
  }

  // Lane j < k writes slot j.
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k && lane == j) {
      ids[t * k + j] = sel_idx[j];
      scales[t * k + j] = __double2float_rn(w[j]);
    }
  }
}

}  // namespace

moe_status launch_route(const float* logits, int64_t T, const float* bias,
                        const moe_route_params& p, int32_t* ids, float* scales,
                        cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const int64_t blocks = (T + kRouteWarps - 1) / kRouteWarps;
  const bool grouped = p.method == MOE_ROUTE_DEEPSEEKV3;
  route_kernel<<<static_cast<unsigned>(blocks), kRouteWarps * 32, 0, s>>>(
      logits, T, p.num_experts, grouped ? bias : nullptr, p.method, p.top_k,
      grouped ? p.n_group : 1, grouped ? p.topk_group : 1,
      grouped ? p.routed_scaling_factor : 1.0f, ids, scales);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "route_kernel launch: %s", cudaGetErrorString(err));
  return MOE_OK;
}

}  // namespace moe
