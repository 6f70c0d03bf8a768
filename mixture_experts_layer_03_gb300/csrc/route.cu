// Step 1: routing. One warp selects the experts of one token; the block then computes
// the weights of all its (token, slot) pairs packed across threads.
//
// Methods (RoutingMethodType of the TensorRT-LLM MoE page, section "路由方法枚举"):
//   Default          softmax over all E, top-k, weights = the selected probabilities
//   Renormalize      top-k, softmax over the k selected logits
//   RenormalizeNaive softmax over all E, top-k, divide by the selected sum
//   SigmoidRenorm    sigmoid, top-k, divide by the selected sum
//   Llama4           "Top1 -> Sigmoid": top-k by logit, each weight the sigmoid of its own
//                    logit, not renormalised
//   MiniMax2         "Sigmoid -> RoutingBiasAdd -> TopK -> Renormalize(without bias)": the
//                    DeepSeekV3 keys over all E (one group), weights = unbiased scores / sum
//   DeepSeekV3       noaux_tc (same page, section "DeepSeek-V3 的 noaux_tc"): sigmoid
//                    scores, + e_score_correction_bias for selection only, group score =
//                    sum of the top-2 biased scores, keep topk_group groups, top-k among
//                    their experts, weights = unbiased scores / (sum + 1e-20) * rsf.
//
//   GroupedTopK      vLLM's GroupedTopKRouter (vLLM MoE page, section "GroupedTopKRouter"),
//                    sigmoid scoring: group score = sum of the group's scores, keep
//                    topk_group groups, k / topk_group experts inside each, renormalise
//                    (route_grouped_topk_kernel below).
//
// Selection keys are fp32 so ids are exact: the logit itself for the softmax and sigmoid
// methods (both maps are increasing), and kappa = fl32(fl32(sigmoid_fp64(l)) + b) for
// DeepSeekV3 and MiniMax2. Ties go to the lower expert index; slots are listed by
// descending key.
//
// FP64 runs at 1/64 of the FP32 rate on this part, so it is used only where the result
// depends on it:
//  * weights: exp/sigmoid of the k selected logits and the divisions, in fp64, for all
//    (token, slot) pairs of a block packed across threads; the Default normaliser over
//    all E uses fp32 expf terms (relative error <= 2 ulp each) accumulated in fp64.
//  * DeepSeekV3 / MiniMax2 keys: every kappa is first approximated in fp32 (|error| <= D,
//    a bound with a wide margin). When every decision (the chosen groups, then each
//    place of the top-k) is separated from the next candidate by more than twice its
//    error bound, the approximate keys decide exactly as the exact ones would and no
//    fp64 key is computed. Otherwise the token takes the exact path: the fp64-derived
//    kappa only for the experts that can still decide a group's top-2 sum or the final
//    top-k (every other expert is provably below the decision threshold). Either way the
//    ids equal those from exact keys.
#include <cfloat>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "launch.cuh"
#include "route_device.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 4;

// EPL = experts per lane (lane l holds experts l, l + 32, ...; E <= 32 * EPL).
// kGrouped: selection on the biased sigmoid keys (DeepSeekV3 with groups, MiniMax2 with
// one group); otherwise on the logits (the softmax/sigmoid methods and Llama4).
template <int EPL, bool kGrouped>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_kernel(const float* __restrict__ logits, int64_t T, int E, const float* __restrict__ bias,
             int method, int k, int n_group, int topk_group, float rsf,
             int32_t* __restrict__ ids, float* __restrict__ scales) {
  __shared__ float s_key[kRouteWarps][256];
  __shared__ uint8_t s_exact[kRouteWarps][256];
  __shared__ uint8_t s_list[kRouteWarps][256];
  __shared__ int s_sel[kRouteWarps * kMaxTopK];
  __shared__ float s_sel_l[kRouteWarps * kMaxTopK];
  __shared__ double s_e[kRouteWarps * kMaxTopK];
  __shared__ double s_z[kRouteWarps];
  const PairSlots ps{s_sel, s_sel_l, s_e, nullptr, s_z};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kRouteWarps;
  const int64_t t = t0 + warp;
  pdl_trigger();
  pdl_wait();

  if (t < T) {   // warp-uniform; every warp reaches the block barriers below
    const float* row = logits + t * E;
    int sel[kMaxTopK];
    double z = 0.0;
    select_token<EPL, kGrouped>(row, E, bias, method, k, n_group, topk_group, lane, s_key[warp],
                                s_exact[warp], s_list[warp], sel, &z);
    record_selection(row, sel, k, lane, ps, warp);
    if (!kGrouped && method == MOE_ROUTE_DEFAULT && lane == 0) s_z[warp] = z;
  }
  __syncthreads();
  block_pair_weights<kGrouped ? 1 : 0>(kRouteWarps, t0, T, k, method, rsf, ps, ids, scales);
}

// vLLM grouped top-k: the same block structure, selection by grouped_topk_select_token.
template <int EPL>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_grouped_topk_kernel(const float* __restrict__ logits, int64_t T, int E, int k, int n_group,
                          int topk_group, float rsf, int32_t* __restrict__ ids,
                          float* __restrict__ scales) {
  __shared__ float s_key[kRouteWarps][256];
  __shared__ int s_sel[kRouteWarps * kMaxTopK];
  __shared__ float s_sel_l[kRouteWarps * kMaxTopK];
  __shared__ double s_e[kRouteWarps * kMaxTopK];
  __shared__ float s_ek[kRouteWarps * kMaxTopK];
  const PairSlots ps{s_sel, s_sel_l, s_e, s_ek, nullptr};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kRouteWarps;
  const int64_t t = t0 + warp;
  pdl_trigger();
  pdl_wait();
  if (t < T) {
    const float* row = logits + t * E;
    int sel[kMaxTopK];
    grouped_topk_select_token<EPL>(row, E, k, n_group, topk_group, lane, s_key[warp], sel);
    record_selection(row, sel, k, lane, ps, warp);
  }
  __syncthreads();
  block_pair_weights<2>(kRouteWarps, t0, T, k, MOE_ROUTE_GROUPED_TOPK, rsf, ps, ids, scales);
}

template <int EPL>
cudaError_t launch_grouped_topk_t(const float* logits, int64_t T, const moe_route_params& p,
                                  int32_t* ids, float* scales, cudaStream_t s) {
  const int64_t blocks = (T + kRouteWarps - 1) / kRouteWarps;
  return launch_pdl(route_grouped_topk_kernel<EPL>, dim3(static_cast<unsigned>(blocks)),
                    dim3(kRouteWarps * 32), 0, s, logits, T, p.num_experts, p.top_k, p.n_group,
                    p.topk_group, p.routed_scaling_factor, ids, scales);
}

template <int EPL, bool kGrouped>
cudaError_t launch_route_t(const float* logits, int64_t T, const float* bias,
                           const moe_route_params& p, int32_t* ids, float* scales, cudaStream_t s) {
  const int64_t blocks = (T + kRouteWarps - 1) / kRouteWarps;
  // Groups and the routed scaling factor belong to DeepSeekV3; MiniMax2 has one group.
  const bool dsv3 = p.method == MOE_ROUTE_DEEPSEEKV3;
  return launch_pdl(route_kernel<EPL, kGrouped>, dim3(static_cast<unsigned>(blocks)),
                    dim3(kRouteWarps * 32), 0, s, logits, T, p.num_experts,
                    kGrouped ? bias : nullptr, p.method, p.top_k, dsv3 ? p.n_group : 1,
                    dsv3 ? p.topk_group : 1, dsv3 ? p.routed_scaling_factor : 1.0f, ids, scales);
}

template <bool kGrouped>
cudaError_t launch_route_e(const float* logits, int64_t T, const float* bias,
                           const moe_route_params& p, int32_t* ids, float* scales, cudaStream_t s) {
  const int E = p.num_experts;
  if (E <= 32) return launch_route_t<1, kGrouped>(logits, T, bias, p, ids, scales, s);
  if (E <= 64) return launch_route_t<2, kGrouped>(logits, T, bias, p, ids, scales, s);
  if (E <= 128) return launch_route_t<4, kGrouped>(logits, T, bias, p, ids, scales, s);
  return launch_route_t<8, kGrouped>(logits, T, bias, p, ids, scales, s);
}

}  // namespace

moe_status launch_route(const float* logits, int64_t T, const float* bias,
                        const moe_route_params& p, int32_t* ids, float* scales,
                        cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const bool keyed = p.method == MOE_ROUTE_DEEPSEEKV3 || p.method == MOE_ROUTE_MINIMAX2;
  cudaError_t err;
  if (p.method == MOE_ROUTE_GROUPED_TOPK) {
    const int E = p.num_experts;
    err = E <= 32    ? launch_grouped_topk_t<1>(logits, T, p, ids, scales, s)
          : E <= 64  ? launch_grouped_topk_t<2>(logits, T, p, ids, scales, s)
          : E <= 128 ? launch_grouped_topk_t<4>(logits, T, p, ids, scales, s)
                     : launch_grouped_topk_t<8>(logits, T, p, ids, scales, s);
  } else {
    err = keyed ? launch_route_e<true>(logits, T, bias, p, ids, scales, s)
                : launch_route_e<false>(logits, T, bias, p, ids, scales, s);
  }
  if (err != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "route_kernel launch: %s", cudaGetErrorString(err));
  return MOE_OK;
}

}  // namespace moe
