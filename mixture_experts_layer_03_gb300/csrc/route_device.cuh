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
                                             int (&sel)[kMaxTopK], double* z_out) {
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
          const float v = s_key[e0 + j];
          if (v > a1) { a2 = a1; a1 = v; } else if (v > a2) { a2 = v; }
        }
        const float thr = a2 - 2.0f * D;
        float x1 = -INFINITY, x2 = -INFINITY;
        for (int j = 0; j < epg; ++j) {
          const int e = e0 + j;
          float v = s_key[e];
          if (v >= thr) {
            if (!s_exact[e]) {
              v = exact_kappa(row[e], bias ? bias[e] : 0.0f);
              s_key[e] = v;
              s_exact[e] = 1;
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
            if (!ex) key[i] = exact_kappa(row[e], bias ? bias[e] : 0.0f);
          }
        }
      }
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
// memory); writes the token's k ids and weights (ids_row, scales_row: its k slots).
template <int EPL>
__device__ __forceinline__ void grouped_topk_token(const float* row, int E, int k, int n_group,
                                                   int topk_group, float rsf, int lane,
                                                   float* s_key, int32_t* ids_row,
                                                   float* scales_row) {
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
  int sel[kMaxTopK];
  bool certain = grouped_topk_select(key, s_key, E, n_group, topk_group, per, lane, true, D, sel);
  if (!certain) {
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
    ids_row[slot] = me;
    scales_row[slot] = __double2float_rn(s / sum * static_cast<double>(rsf));
  }
}


// Weights of one token's k chosen experts (sel, from select_token), one per lane j < k,
// written with the ids to the token's slots. The same arithmetic as the route kernel's
// packed weights: fp64 sigmoid (sigmoid methods) or exp(l - l_max) (softmax methods) of
// the chosen logits, their sum taken in slot order, one rounding to fp32.
template <bool kGrouped>
__device__ __forceinline__ void token_weights_warp(const float* row, const int (&sel)[kMaxTopK],
                                                   int k, int method, double z, float rsf,
                                                   int lane, int32_t* ids_row,
                                                   float* scales_row) {
  int me = 0;
#pragma unroll
  for (int q = 0; q < kMaxTopK; ++q)
    if (q < k && q == lane) me = sel[q];
  float lv = -INFINITY;
  if (lane < k) {
    const float v = row[me];
    lv = isfinite(v) ? v : -INFINITY;
  }
  const double l0 = static_cast<double>(__shfl_sync(0xffffffffu, lv, 0));   // the largest
  double e = 0.0;
  if (lane < k) {
    if (kGrouped || method == MOE_ROUTE_SIGMOID_RENORM || method == MOE_ROUTE_LLAMA4)
      e = sigmoid_d(static_cast<double>(lv));
    else
      e = exp(static_cast<double>(lv) - l0);
  }
  double s = 0.0;
  for (int q = 0; q < k; ++q) s += __shfl_sync(0xffffffffu, e, q);
  if (lane < k) {
    double wgt;
    if (method == MOE_ROUTE_DEFAULT)
      wgt = e / z;
    else if (method == MOE_ROUTE_LLAMA4)
      wgt = e;
    else if (method == MOE_ROUTE_MINIMAX2)
      wgt = e / s;
    else if (kGrouped)
      wgt = e / (s + 1e-20) * static_cast<double>(rsf);
    else
      wgt = e / s;
    ids_row[lane] = me;
    scales_row[lane] = __double2float_rn(wgt);
  }
}

}  // namespace
}  // namespace moe
