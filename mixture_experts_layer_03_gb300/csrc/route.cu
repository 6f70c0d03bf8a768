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

namespace moe {
namespace {

constexpr int kRouteWarps = 4;
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
    const float ok = __shfl_xor_sync(0xffffffffu, v.key, off);
    const int oi = __shfl_xor_sync(0xffffffffu, v.idx, off);
    if (beats(ok, oi, v.key, v.idx)) {
      v.key = ok;
      v.idx = oi;
    }
  }
  return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__device__ __forceinline__ double sigmoid_d(double l) { return 1.0 / (1.0 + exp(-l)); }

__device__ __forceinline__ float exact_kappa(float l, float b) {
  return __fadd_rn(__double2float_rn(sigmoid_d(static_cast<double>(l))), b);
}

// k rounds of warp argmax over this lane's keys; returns the winners (uniform in the
// warp). Keys of absent or excluded experts must be passed as absent via `live`.
template <int EPL>
__device__ __forceinline__ void warp_topk(const float (&key)[EPL], uint32_t live, int k,
                                          int lane, int (&sel)[kMaxTopK], float* kth_key) {
  uint32_t taken = 0;
  float last = -INFINITY;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    sel[j] = 0;
    if (j < k) {
      KeyIdx best{-INFINITY, INT32_MAX};
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (((live & ~taken) >> i) & 1u && beats(key[i], e, best.key, best.idx)) {
          best.key = key[i];
          best.idx = e;
        }
      }
      best = warp_best(best);
      if (best.idx == INT32_MAX) best.idx = 0;   // unreachable: callers pass >= k live keys
      if ((best.idx & 31) == lane) taken |= 1u << (best.idx >> 5);
      sel[j] = best.idx;
      last = best.key;
    }
  }
  if (kth_key) *kth_key = last;
}

// k + 1 rounds of warp argmax over approximate keys: the k winners in sel, and whether
// every two consecutive keys among the k + 1 best (the (k+1)-th taken as -inf when there
// is none) differ by more than 2 * D. Keys within D of the exact ones then select and
// order exactly the same experts.
template <int EPL>
__device__ __forceinline__ bool warp_topk_separated(const float (&key)[EPL], uint32_t live, int k,
                                                    int lane, float D, int (&sel)[kMaxTopK]) {
  uint32_t taken = 0;
  float prev = INFINITY;
  bool sep = true;
  for (int j = 0; j <= k; ++j) {
    KeyIdx best{-INFINITY, INT32_MAX};
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (((live & ~taken) >> i) & 1u && beats(key[i], e, best.key, best.idx)) {
        best.key = key[i];
        best.idx = e;
      }
    }
    best = warp_best(best);
    const float cur = best.idx == INT32_MAX ? -INFINITY : best.key;
    if (j > 0 && !(prev - cur > 2.0f * D)) sep = false;
    if (j < k) {
      if (best.idx == INT32_MAX) best.idx = 0;   // unreachable: callers pass >= k live keys
      if ((best.idx & 31) == lane) taken |= 1u << (best.idx >> 5);
      sel[j] = best.idx;
    }
    prev = cur;
  }
  return sep;
}

// EPL = experts per lane (lane l holds experts l, l + 32, ...; E <= 32 * EPL).
// kGrouped: selection on the biased sigmoid keys (DeepSeekV3 with groups, MiniMax2 with
// one group); otherwise on the logits (the softmax/sigmoid methods and Llama4).
template <int EPL, bool kGrouped>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_kernel(const float* __restrict__ logits, int64_t T, int E, const float* __restrict__ bias,
             int method, int k, int n_group, int topk_group, float rsf,
             int32_t* __restrict__ ids, float* __restrict__ scales) {
  constexpr int kMaxPerLane = EPL;
  __shared__ float s_key[kRouteWarps][256];
  __shared__ uint8_t s_exact[kRouteWarps][256];
  __shared__ float s_sel_l[kRouteWarps][kMaxTopK];
  __shared__ double s_e[kRouteWarps][kMaxTopK];
  __shared__ double s_z[kRouteWarps];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kRouteWarps + warp;
  const bool valid = t < T;   // warp-uniform; invalid warps still reach the block barriers
  pdl_trigger();
  pdl_wait();

  if (valid) {
    const float* row = logits + t * E;
    float l[kMaxPerLane], key[kMaxPerLane];
    uint32_t present = 0;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int e = lane + 32 * i;
      float v = -INFINITY;
      if (e < E) {
        present |= 1u << i;
        v = row[e];
        if (!isfinite(v)) v = -INFINITY;
      }
      l[i] = v;
      key[i] = v;
    }

    if (kGrouped) {
      // fp32 approximation of every kappa, and a bound D on |kappa_exact - kappa_approx|:
      // the fp32 sigmoid is within 4e-7 of the true value and both roundings add at most
      // one ulp of the key, so 1e-6 + 2.5e-7 * |kappa| holds with room to spare.
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        const int e = lane + 32 * i;
        if ((present >> i) & 1u) {
          const float b = bias ? bias[e] : 0.0f;
          const bool fin = l[i] != -INFINITY;
          const float sa = fin ? 1.0f / (1.0f + expf(-l[i])) : 0.0f;
          key[i] = __fadd_rn(sa, b);
          s_key[warp][e] = key[i];
          s_exact[warp][e] = fin ? 0 : 1;   // sigmoid(-inf) = 0 exactly
          amax = fmaxf(amax, fabsf(key[i]));
        }
      }
      const float D = 1e-6f + 2.5e-7f * warp_max_f(amax);
      __syncwarp();

      const int epg = E / n_group;
      int sel[kMaxTopK];

      // Certified path: every decision taken on the approximate keys, accepted only when
      // each one has a margin above the keys' error bound, so that the exact keys would
      // decide the same way. (1) The chosen groups: the approximate group score (sum of
      // the approximate top-2) is within 2D of the exact top-2 sum, plus one rounding of
      // each sum, so Eg = 2D + 2.4e-7 |score| bounds its error; the last chosen group must
      // beat the best left out by more than 2 Eg. (2) The top-k inside them: consecutive
      // keys of the k + 1 best must differ by more than 2D.
      bool certain = true;
      uint32_t chosen = n_group > 1 ? 0u : 1u;
      if (n_group > 1) {
        float ga = -INFINITY;
        int gi = INT32_MAX;
        if (lane < n_group) {
          const int e0 = lane * epg;
          float a1 = -INFINITY, a2 = -INFINITY;
          for (int j = 0; j < epg; ++j) {
            const float v = s_key[warp][e0 + j];
            if (v > a1) { a2 = a1; a1 = v; } else if (v > a2) { a2 = v; }
          }
          ga = __fadd_rn(a1, a2);
          gi = lane;
        }
        const float Eg = 2.0f * D + 2.4e-7f * warp_max_f(lane < n_group ? fabsf(ga) : 0.0f);
        bool gt = false;
        float last = INFINITY, next = -INFINITY;
        for (int r = 0; r <= topk_group && r < n_group; ++r) {
          KeyIdx v = gt ? KeyIdx{-INFINITY, INT32_MAX} : KeyIdx{ga, gi};
          v = warp_best(v);
          if (r < topk_group) {
            if (v.idx == lane) gt = true;
            chosen |= 1u << v.idx;
            last = v.key;
          } else {
            next = v.key;
          }
        }
        if (topk_group < n_group && !(last - next > 2.0f * Eg)) certain = false;
      }
      if (certain) {
        uint32_t live = 0;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
          const int e = lane + 32 * i;
          if (((present >> i) & 1u) && ((chosen >> (e / epg)) & 1u)) live |= 1u << i;
        }
        certain = warp_topk_separated(key, live, k, lane, D, sel);
      }

      if (!certain) {
        // Exact path (rare): exact keys wherever a decision could depend on them.
        // Group scores: lane g sums the exact top-2 keys of its group. Only experts whose
        // approximate key is within 2D of the approximate second-largest can be in the
        // exact top-2; their keys are made exact first.
        float gscore = -INFINITY;
        int gidx = INT32_MAX;
        if (n_group > 1 && lane < n_group) {
          const int e0 = lane * epg;
          float a1 = -INFINITY, a2 = -INFINITY;
          for (int j = 0; j < epg; ++j) {
            const float v = s_key[warp][e0 + j];
            if (v > a1) { a2 = a1; a1 = v; } else if (v > a2) { a2 = v; }
          }
          const float thr = a2 - 2.0f * D;
          float x1 = -INFINITY, x2 = -INFINITY;
          for (int j = 0; j < epg; ++j) {
            const int e = e0 + j;
            float v = s_key[warp][e];
            if (v >= thr) {
              if (!s_exact[warp][e]) {
                v = exact_kappa(row[e], bias ? bias[e] : 0.0f);
                s_key[warp][e] = v;
                s_exact[warp][e] = 1;
              }
              if (v > x1) { x2 = x1; x1 = v; } else if (v > x2) { x2 = v; }
            }
          }
          gscore = __fadd_rn(x1, x2);
          gidx = lane;
        }
        // Keep topk_group groups by repeated warp argmax (ties: lower group index). A single
        // group is kept without scoring it.
        chosen = n_group > 1 ? 0u : 1u;
        bool gtaken = false;
        for (int r = 0; n_group > 1 && r < topk_group; ++r) {
          KeyIdx v = gtaken ? KeyIdx{-INFINITY, INT32_MAX} : KeyIdx{gscore, gidx};
          v = warp_best(v);
          if (v.idx == lane) gtaken = true;
          chosen |= 1u << v.idx;
        }
        __syncwarp();

        // Final top-k inside the chosen groups. Bounds per expert (exact: lb = ub = kappa);
        // the k-th largest lower bound is a threshold no non-candidate can reach.
        float lb[kMaxPerLane];
        uint32_t live = 0;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
          const int e = lane + 32 * i;
          lb[i] = -INFINITY;
          if (((present >> i) & 1u) && ((chosen >> (e / epg)) & 1u)) {
            live |= 1u << i;
            key[i] = s_key[warp][e];
            lb[i] = s_exact[warp][e] ? key[i] : key[i] - D;
          }
        }
        int tmp[kMaxTopK];
        float kth_lb;
        warp_topk(lb, live, k, lane, tmp, &kth_lb);
        uint32_t cand = 0;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
          const int e = lane + 32 * i;
          if ((live >> i) & 1u) {
            const bool ex = s_exact[warp][e];
            const float ub = ex ? key[i] : key[i] + D;
            if (ub >= kth_lb) {
              cand |= 1u << i;
              if (!ex) key[i] = exact_kappa(row[e], bias ? bias[e] : 0.0f);
            }
          }
        }
        warp_topk(key, cand, k, lane, sel, nullptr);
      }
      // Selected logits for the weights.
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        if (j < k && lane == j) {
          ids[t * k + j] = sel[j];
          const float v = row[sel[j]];
          s_sel_l[warp][j] = isfinite(v) ? v : -INFINITY;
        }
      }
    } else {
      int sel[kMaxTopK];
      warp_topk(key, present, k, lane, sel, nullptr);
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        if (j < k && lane == j) {
          ids[t * k + j] = sel[j];
          const float v = row[sel[j]];
          s_sel_l[warp][j] = isfinite(v) ? v : -INFINITY;
        }
      }
      if (method == MOE_ROUTE_DEFAULT) {
        // Normaliser over all E: fp32 exp terms, fp64 accumulation.
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) m = fmaxf(m, l[i]);
        m = warp_max_f(m);
        double z = 0.0;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i)
          if ((present >> i) & 1u) z += static_cast<double>(expf(l[i] - m));
        z = warp_sum_d(z);
        if (lane == 0) s_z[warp] = z;
      }
    }
  }
  __syncthreads();

  // Weights of the block's (token, slot) pairs, packed across threads.
  const int npairs = kRouteWarps * k;
  for (int pidx = threadIdx.x; pidx < npairs; pidx += blockDim.x) {
    const int w = pidx / k, j = pidx - w * k;
    const int64_t tt = static_cast<int64_t>(blockIdx.x) * kRouteWarps + w;
    if (tt >= T) continue;
    const double lv = static_cast<double>(s_sel_l[w][j]);
    double e;
    if (kGrouped || method == MOE_ROUTE_SIGMOID_RENORM || method == MOE_ROUTE_LLAMA4)
      e = sigmoid_d(lv);
    else
      e = exp(lv - static_cast<double>(s_sel_l[w][0]));   // slot 0 holds the largest logit
    s_e[w][j] = e;
  }
  __syncthreads();
  for (int pidx = threadIdx.x; pidx < npairs; pidx += blockDim.x) {
    const int w = pidx / k, j = pidx - w * k;
    const int64_t tt = static_cast<int64_t>(blockIdx.x) * kRouteWarps + w;
    if (tt >= T) continue;
    double s = 0.0;
    for (int q = 0; q < k; ++q) s += s_e[w][q];
    double wgt;
    if (method == MOE_ROUTE_DEFAULT)
      wgt = s_e[w][j] / s_z[w];
    else if (method == MOE_ROUTE_LLAMA4)
      wgt = s_e[w][j];
    else if (method == MOE_ROUTE_MINIMAX2)
      wgt = s_e[w][j] / s;
    else if (kGrouped)
      wgt = s_e[w][j] / (s + 1e-20) * static_cast<double>(rsf);
    else
      wgt = s_e[w][j] / s;
    scales[tt * k + j] = __double2float_rn(wgt);
  }
}


// vLLM grouped top-k with sigmoid scoring, one warp per token. The selection key of
// expert e is fl32(sigmoid_fp64(l_e)); group g's score is the sum of its keys added in
// fp32 in expert order (lane g adds them one by one); the topk_group best groups are
// kept (ties: lower group index); inside each, its k / topk_group best keys (ties: lower
// expert index). Slots are listed by descending key; weights = s / sum(s) * rsf with the
// fp64 scores s of the chosen experts.
//
// Every key is first approximated in fp32 (1 / (1 + expf(-l)), within D of the exact key).
// The decisions on approximate keys are accepted when each has a margin the error cannot
// close: the last kept group's score beats the best dropped one by more than 2 Eg, where
// Eg bounds a score's error (epg keys off by D each, plus one rounding of each partial
// sum on either side: u * m per step, m <= epg the partial sum); and inside each kept
// group the last chosen key beats the next by more than 2 D. Then the chosen set equals
// the exact one; otherwise the token recomputes every key exactly and decides again. The
// slot order and the weights always come from the exact keys and scores of the chosen k,
// computed one per lane.
template <int EPL>
__device__ __forceinline__ bool grouped_topk_select(const float (&key)[EPL], const float* skey,
                                                    int E, int n_group, int topk_group, int per,
                                                    int lane, bool check, float D,
                                                    int (&sel)[kMaxTopK]) {
  const int epg = E / n_group;
  float tot = -INFINITY;
  if (lane < n_group) {
    const float* gk = skey + lane * epg;
    float acc = gk[0];
    for (int j = 1; j < epg; ++j) acc = __fadd_rn(acc, gk[j]);
    tot = acc;
  }
  bool certain = true;
  // Groups: topk_group rounds of warp argmax (one more to read the best dropped score).
  const float Eg = static_cast<float>(epg) * D + 6.0e-8f * static_cast<float>(epg) *
                                                     static_cast<float>(epg + 1);
  bool gtaken = false;
  int groups[32];
  float last = INFINITY;
  for (int r = 0; r < topk_group; ++r) {
    KeyIdx v = gtaken ? KeyIdx{-INFINITY, INT32_MAX} : KeyIdx{tot, lane < n_group ? lane : INT32_MAX};
    v = warp_best(v);
    if (v.idx == lane) gtaken = true;
    groups[r] = v.idx;
    last = v.key;
  }
  if (check && topk_group < n_group) {
    KeyIdx v = gtaken ? KeyIdx{-INFINITY, INT32_MAX} : KeyIdx{tot, lane < n_group ? lane : INT32_MAX};
    v = warp_best(v);
    if (!(last - v.key > 2.0f * Eg)) certain = false;
  }
  // Experts: per rounds inside each kept group (one more for the margin).
  int n = 0;
  for (int r = 0; r < topk_group; ++r) {
    const int lo = groups[r] * epg, hi = lo + epg;
    uint32_t live = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e >= lo && e < hi) live |= 1u << i;
    }
    float kth = INFINITY;
    for (int j = 0; j <= per; ++j) {
      if (j == per && !check) break;
      KeyIdx best{-INFINITY, INT32_MAX};
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if ((live >> i) & 1u && beats(key[i], e, best.key, best.idx)) {
          best.key = key[i];
          best.idx = e;
        }
      }
      best = warp_best(best);
      if (j < per) {
        if ((best.idx & 31) == lane) live &= ~(1u << (best.idx >> 5));
        // n < k <= kMaxTopK: every kept group contributes exactly per experts
#pragma unroll
        for (int q = 0; q < kMaxTopK; ++q)
          if (q == n) sel[q] = best.idx;
        ++n;
        kth = best.key;
      } else {
        const float next = best.idx == INT32_MAX ? -INFINITY : best.key;
        if (!(kth - next > 2.0f * D)) certain = false;
      }
    }
  }
  return certain;
}

template <int EPL>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_grouped_topk_kernel(const float* __restrict__ logits, int64_t T, int E, int k, int n_group,
                          int topk_group, float rsf, int32_t* __restrict__ ids,
                          float* __restrict__ scales) {
  __shared__ float s_key[kRouteWarps][256];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kRouteWarps + warp;
  pdl_trigger();
  pdl_wait();
  if (t >= T) return;   // warp-uniform; the kernel has no block-wide barrier

  const float* row = logits + t * E;
  float l[EPL], key[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    float v = -INFINITY;
    key[i] = -INFINITY;
    if (e < E) {
      v = row[e];
      if (!isfinite(v)) v = -INFINITY;
      key[i] = v == -INFINITY ? 0.0f : 1.0f / (1.0f + expf(-v));   // sigmoid(-inf) = 0 exactly
      s_key[warp][e] = key[i];
    }
    l[i] = v;
  }
  __syncwarp();
  // The fp32 sigmoid is within a few ulp of the true value (keys lie in [0, 1]) and the
  // exact key adds one rounding: 1.25e-6 bounds the difference with a wide margin.
  constexpr float D = 1.25e-6f;
  const int per = k / topk_group;
  int sel[kMaxTopK];
  bool certain = grouped_topk_select(key, s_key[warp], E, n_group, topk_group, per, lane, true, D, sel);
  if (!certain) {
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        key[i] = l[i] == -INFINITY ? 0.0f : __double2float_rn(sigmoid_d(static_cast<double>(l[i])));
        s_key[warp][e] = key[i];
      }
    }
    __syncwarp();
    grouped_topk_select(key, s_key[warp], E, n_group, topk_group, per, lane, false, 0.0f, sel);
  }

  // Lane j < k: the j-th chosen expert's exact score and key; its slot is the number of
  // chosen experts that beat it (larger key, or the same key and a lower index).
  int me = INT32_MAX;
#pragma unroll
  for (int q = 0; q < kMaxTopK; ++q)
    if (q < k && q == lane) me = sel[q];
  double s = 0.0;
  float ek = -INFINITY;
  if (lane < k) {
    const float v = row[me];
    s = isfinite(v) ? sigmoid_d(static_cast<double>(v)) : 0.0;   // non-finite counts as -inf
    ek = __double2float_rn(s);
  }
  int slot = 0;
  for (int q = 0; q < k; ++q) {
    const float ok = __shfl_sync(0xffffffffu, ek, q);
    const int oe = __shfl_sync(0xffffffffu, me, q);
    if (q != lane && beats(ok, oe, ek, me)) ++slot;
  }
  const double sum = warp_sum_d(s);
  if (lane < k) {
    ids[t * k + slot] = me;
    scales[t * k + slot] = __double2float_rn(s / sum * static_cast<double>(rsf));
  }
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
