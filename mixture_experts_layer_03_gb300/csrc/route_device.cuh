// Per-token routing shared by the route kernel (route.cu) and the routing epilogue of
// the fused gate (gate.cu): one warp selects the experts of one token and computes their
// weights. The methods, keys and the certified fp32 / exact fp64 decision scheme are
// described at the top of route.cu.
#pragma once

#include <cfloat>
#include <cmath>
#include <cstdint>

#include "internal.h"

namespace moe {
namespace {

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

// Replaces the approximate keys of the experts marked 2 in s_exact by their exact keys
// fl32(fl32(sigmoid_fp64(l)) + b) and marks them 1. The marked experts are first listed in
// s_list (expert ids, 256 bytes per warp), then each lane takes every 32nd entry.
template <int EPL>
__device__ __forceinline__ void make_marked_exact(const float* row, const float* bias, int E,
                                                  int lane, float* s_key, uint8_t* s_exact,
                                                  uint8_t* s_list) {
  int n = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    const bool m = e < E && s_exact[e] == 2;
    const uint32_t b = __ballot_sync(0xffffffffu, m);
    if (m) s_list[n + __popc(b & ((1u << lane) - 1u))] = static_cast<uint8_t>(e);
    n += __popc(b);
  }
  __syncwarp();
  for (int j = lane; j < n; j += 32) {
    const int e = s_list[j];
    s_key[e] = exact_kappa(row[e], bias ? bias[e] : 0.0f);
    s_exact[e] = 1;
  }
  __syncwarp();
}

// Selection of one token's k experts by one warp: `row` holds the token's E fp32 logits
// (global or shared memory); s_key / s_exact are this warp's scratch (256 floats and 256
// bytes of shared memory). On return sel[0..k) holds the chosen experts by descending key
// (uniform across the warp); for Default, *z_out = the softmax normaliser over all E
// (fp32 exp terms of l - max l, accumulated in fp64).
// kGrouped: selection on the biased sigmoid keys (DeepSeekV3 with groups, MiniMax2 with
// one group); otherwise on the logits (the softmax/sigmoid methods and Llama4).
template <int EPL, bool kGrouped>
__device__ __forceinline__ void select_token(const float* row, int E, const float* bias,
                                             int method, int k, int n_group, int topk_group,
                                             int lane, float* s_key, uint8_t* s_exact,
                                             uint8_t* s_list, int (&sel)[kMaxTopK],
                                             double* z_out) {
  float l[EPL], key[EPL];
  uint32_t present = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
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
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if ((present >> i) & 1u) {
        const float b = bias ? bias[e] : 0.0f;
        const bool fin = l[i] != -INFINITY;
        const float sa = fin ? 1.0f / (1.0f + expf(-l[i])) : 0.0f;
        key[i] = __fadd_rn(sa, b);
        s_key[e] = key[i];
        s_exact[e] = fin ? 0 : 1;   // sigmoid(-inf) = 0 exactly
        amax = fmaxf(amax, fabsf(key[i]));
      }
    }
    const float D = 1e-6f + 2.5e-7f * warp_max_f(amax);
    __syncwarp();

    const int epg = E / n_group;

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
          const float v = s_key[e0 + j];
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
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (((present >> i) & 1u) && ((chosen >> (e / epg)) & 1u)) live |= 1u << i;
      }
      certain = warp_topk_separated(key, live, k, lane, D, sel);
    }

    if (!certain) {
      // Exact path (rare): exact keys wherever a decision could depend on them, computed
      // one per lane over a list of the experts concerned (marked 2 in s_exact), so that
      // the fp64 sigmoids of a token run side by side rather than lane after lane.
      // Group scores: only experts whose approximate key is within 2D of their group's
      // approximate second largest can be in its exact top-2 (every other expert's exact
      // key lies below the exact second largest), so those are made exact first.
      if (n_group > 1 && lane < n_group) {
        const int e0 = lane * epg;
        float a1 = -INFINITY, a2 = -INFINITY;
        for (int j = 0; j < epg; ++j) {
          const float v = s_key[e0 + j];
          if (v > a1) { a2 = a1; a1 = v; } else if (v > a2) { a2 = v; }
        }
        const float thr = a2 - 2.0f * D;
        for (int j = 0; j < epg; ++j)
          if (s_key[e0 + j] >= thr && !s_exact[e0 + j]) s_exact[e0 + j] = 2;
      }
      __syncwarp();
      make_marked_exact<EPL>(row, bias, E, lane, s_key, s_exact, s_list);
      float gscore = -INFINITY;
      int gidx = INT32_MAX;
      if (n_group > 1 && lane < n_group) {
        const int e0 = lane * epg;
        float x1 = -INFINITY, x2 = -INFINITY;
        for (int j = 0; j < epg; ++j) {
          const float v = s_key[e0 + j];
          if (v > x1) { x2 = x1; x1 = v; } else if (v > x2) { x2 = v; }
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

      // Final top-k inside the chosen groups. Bounds per expert (exact: lb = ub = kappa);
      // the k-th largest lower bound is a threshold no non-candidate can reach.
      float lb[EPL];
      uint32_t live = 0;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        lb[i] = -INFINITY;
        if (((present >> i) & 1u) && ((chosen >> (e / epg)) & 1u)) {
          live |= 1u << i;
          key[i] = s_key[e];
          lb[i] = s_exact[e] ? key[i] : key[i] - D;
        }
      }
      int tmp[kMaxTopK];
      float kth_lb;
      warp_topk(lb, live, k, lane, tmp, &kth_lb);
      uint32_t cand = 0;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if ((live >> i) & 1u) {
          const bool ex = s_exact[e];
          const float ub = ex ? key[i] : key[i] + D;
          if (ub >= kth_lb) {
            cand |= 1u << i;
            if (!ex) s_exact[e] = 2;
          }
        }
      }
      __syncwarp();
      make_marked_exact<EPL>(row, bias, E, lane, s_key, s_exact, s_list);
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if ((cand >> i) & 1u) key[i] = s_key[lane + 32 * i];
      warp_topk(key, cand, k, lane, sel, nullptr);
    }
  } else {
    warp_topk(key, present, k, lane, sel, nullptr);
    if (method == MOE_ROUTE_DEFAULT) {
      // Normaliser over all E: fp32 exp terms, fp64 accumulation.
      float m = -INFINITY;
#pragma unroll
      for (int i = 0; i < EPL; ++i) m = fmaxf(m, l[i]);
      m = warp_max_f(m);
      double z = 0.0;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if ((present >> i) & 1u) z += static_cast<double>(expf(l[i] - m));
      z = warp_sum_d(z);
      *z_out = z;
    }
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

// vLLM grouped top-k (sigmoid scoring) of one token by one warp: `row` holds its E fp32
// logits (global or shared memory), s_key is this warp's scratch (256 floats of shared
// memory). On return sel[0..k) holds the chosen experts (uniform across the warp), group
// by group; block_pair_weights orders them by key and weights them.
template <int EPL>
__device__ __forceinline__ void grouped_topk_select_token(const float* row, int E, int k,
                                                          int n_group, int topk_group, int lane,
                                                          float* s_key, int (&sel)[kMaxTopK]) {
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
      s_key[e] = key[i];
    }
    l[i] = v;
  }
  __syncwarp();
  // The fp32 sigmoid is within a few ulp of the true value (keys lie in [0, 1]) and the
  // exact key adds one rounding: 1.25e-6 bounds the difference with a wide margin.
  constexpr float D = 1.25e-6f;
  const int per = k / topk_group;
  const bool certain = grouped_topk_select(key, s_key, E, n_group, topk_group, per, lane, true, D,
                                           sel);
  if (!certain) {
    // Every key exact (fp64 sigmoid rounded once), EPL per lane side by side.
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        key[i] = l[i] == -INFINITY ? 0.0f : __double2float_rn(sigmoid_d(static_cast<double>(l[i])));
        s_key[e] = key[i];
      }
    }
    __syncwarp();
    grouped_topk_select(key, s_key, E, n_group, topk_group, per, lane, false, 0.0f, sel);
  }
}

// Per-token routing record of a block, kept in shared memory between the selection (one
// warp per token) and block_pair_weights: slot j of token r is entry r * kMaxTopK + j.
struct PairSlots {
  int* sel;        // chosen expert
  float* sel_l;    // its logit (non-finite as -inf)
  double* e;       // its fp64 score
  float* ek;       // its exact fp32 key (grouped top-k ordering)
  double* z;       // [rows] Default: softmax normaliser over all E
};

// Lane j < k of the warp that selected token r records slot j.
__device__ __forceinline__ void record_selection(const float* row, const int (&sel)[kMaxTopK],
                                                 int k, int lane, const PairSlots& ps, int r) {
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k && lane == j) {
      const float v = row[sel[j]];
      ps.sel[r * kMaxTopK + j] = sel[j];
      ps.sel_l[r * kMaxTopK + j] = isfinite(v) ? v : -INFINITY;
    }
  }
}

// Weights of the block's nrows tokens (t0 + r, r < nrows; tokens at or past T skipped),
// their (token, slot) pairs packed across the block's threads: FP64 runs at 1/64 of the
// FP32 rate on this part, so a warp that held one token's k pairs would issue mostly idle
// fp64 instructions. Scores: fp64 sigmoid of the chosen logit (sigmoid methods, keyed and
// grouped top-k) or exp(l - l_max) (softmax methods; slot 0 holds the largest logit); their
// sum taken in slot order; one rounding to fp32. kMode: 0 logit-keyed methods, 1 biased
// sigmoid keys (DeepSeekV3, MiniMax2), 2 vLLM grouped top-k (slots ordered here by the
// exact key, ties to the lower expert index). Called by every thread of the block; it
// synchronises the block twice.
template <int kMode>
__device__ __forceinline__ void block_pair_weights(int nrows, int64_t t0, int64_t T, int k,
                                                   int method, float rsf, const PairSlots& ps,
                                                   int32_t* ids, float* scales) {
  const int npairs = nrows * k;
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    const int r = p / k, j = p - r * k;
    if (t0 + r >= T) continue;
    const double lv = static_cast<double>(ps.sel_l[r * kMaxTopK + j]);
    double e;
    if (kMode != 0 || method == MOE_ROUTE_SIGMOID_RENORM || method == MOE_ROUTE_LLAMA4)
      e = sigmoid_d(lv);
    else
      e = exp(lv - static_cast<double>(ps.sel_l[r * kMaxTopK]));
    ps.e[r * kMaxTopK + j] = e;
    if (kMode == 2) ps.ek[r * kMaxTopK + j] = __double2float_rn(e);
  }
  __syncthreads();
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    const int r = p / k, j = p - r * k;
    const int64_t t = t0 + r;
    if (t >= T) continue;
    const double* er = ps.e + r * kMaxTopK;
    double s = 0.0;
    for (int q = 0; q < k; ++q) s += er[q];
    double wgt;
    if (kMode == 2)
      wgt = er[j] / s * static_cast<double>(rsf);
    else if (method == MOE_ROUTE_DEFAULT)
      wgt = er[j] / ps.z[r];
    else if (method == MOE_ROUTE_LLAMA4)
      wgt = er[j];
    else if (method == MOE_ROUTE_MINIMAX2)
      wgt = er[j] / s;
    else if (kMode == 1)
      wgt = er[j] / (s + 1e-20) * static_cast<double>(rsf);
    else
      wgt = er[j] / s;
    const int me = ps.sel[r * kMaxTopK + j];
    int slot = j;
    if (kMode == 2) {
      const float* ekr = ps.ek + r * kMaxTopK;
      const int* sr = ps.sel + r * kMaxTopK;
      slot = 0;
      for (int q = 0; q < k; ++q)
        if (q != j && beats(ekr[q], sr[q], ekr[j], me)) ++slot;
    }
    ids[t * k + slot] = me;
    scales[t * k + slot] = __double2float_rn(wgt);
  }
  __syncthreads();
}

}  // namespace
}  // namespace moe
