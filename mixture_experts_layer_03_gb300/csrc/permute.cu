// Step 2: permute (Dense GEMM -> GroupedGEMM article, sections 2.1-2.2: rows of each
// expert gathered into one contiguous block; blocks concatenated in expert order and
// described by an offset array; one grouped launch then covers every expert).
//
// Deterministic, no atomics in the ordering:
//   hist_kernel    per chunk of kPermChunk (token, slot) pairs: histogram over experts
//                  (skipped when there is a single chunk: the plan kernel counts it)
//   plan_kernel    every chunk: column sums + exclusive scan of the histograms give each
//                  (chunk, expert) its base row; inside the chunk, ranks come from
//                  warp match_any and a running per-expert count, so rows of an expert
//                  keep ascending flat index f = t*k + j. Chunk 0 also writes counts,
//                  starts, offsets and the FC1/FC2 tile lists.
//   gather_kernel  x_perm[r] = x[perm_src[r] / k] (and x[t] for the shared rows),
//                  16-byte vector copies, one warp per row (decode-sized batches).
//   plan_gather_kernel  plan and row copy in one launch when the problem is one chunk
//                  and copied row by row: every block plans (block 0 publishes the plan)
//                  and copies its rows from its own shared-memory perm_src.
//   scatter_kernel the same rows, token-major: one warp per token reads x[t] once and
//                  writes it to each of its permuted rows perm_inv[t*k + j] (and the
//                  shared row). With many tokens, x is then read from HBM once instead
//                  of once per slot through L2 (batches of at least kScatterMinTokens).
#include <cstdint>

#include <cuda_bf16.h>

#include "internal.h"
#include "launch.cuh"

namespace moe {
namespace {

constexpr int kPermWarps = kPermThreads / 32;
// Batches with at least this many tokens copy rows token-major (scatter_kernel): enough
// warps (one per token) to keep every SM busy. Smaller batches copy row by row.
constexpr int64_t kScatterMinTokens = 2048;

__global__ void __launch_bounds__(kPermThreads)
hist_kernel(const int32_t* __restrict__ ids, int64_t P, int E, int e_lo, int e_hi,
            int32_t* __restrict__ block_hist, int32_t* __restrict__ status) {
  __shared__ int32_t h[256];
  pdl_trigger();
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  pdl_wait();
  // This forward's status bits start from zero (the plan and GEMM kernels run after).
  if (blockIdx.x == 0 && threadIdx.x < 4) status[threadIdx.x] = 0;
  __syncthreads();
  const int64_t f0 = static_cast<int64_t>(blockIdx.x) * kPermChunk;
  const int64_t f1 = (P < f0 + kPermChunk ? P : f0 + kPermChunk);
  for (int64_t f = f0 + threadIdx.x; f < f1; f += blockDim.x) {
    const int e = ids[f];
    if (e >= e_lo && e < e_hi) atomicAdd(&h[e], 1);   // local experts only
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) block_hist[blockIdx.x * E + e] = h[e];
}

// Block-wide exclusive scan of v over the first n <= kPermThreads threads.
// Returns the exclusive prefix; *total receives the sum.
__device__ int block_exclusive_scan(int v, int n, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (static_cast<int>(threadIdx.x) >= n) v = 0;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kPermWarps ? s_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    if (lane < kPermWarps) s_warp[lane] = wi - w;   // exclusive warp prefix
    if (lane == kPermWarps - 1) s_warp[kPermWarps] = wi;
  }
  __syncthreads();
  const int res = s_warp[warp] + incl - v;
  *total = s_warp[kPermWarps];
  __syncthreads();
  return res;
}

struct PlanArgs {
  const int32_t* ids;
  int64_t P;
  int T;
  int E;
  int e_lo, e_hi;      // the experts of this call; slots of others contribute nothing
  int k;
  int nb;
  int has_shared;
  int I;
  int shared_I;
  int H;
  int pair_min_rows;   // groups with at least this many rows go to the CTA-pair list
  int narrow_rows;     // single-SM groups with 1..narrow_rows rows get narrow tiles
  const int32_t* block_hist;
  int32_t* counts;     // [G]
  int32_t* starts;     // [G]
  int32_t* offsets;    // [E+1]
  int32_t* tile_off1;  // [2][G+1]: FC1 offsets into the pair list, then the single-SM list
  int32_t* tile_off2;  // [2][G+1]: FC2 offsets into the pair list, then the single-SM list
  int32_t* perm_src;   // [P]
  int32_t* perm_inv;   // [P]
  int32_t* status;
  int32_t* sched;      // [kSchedCounters + G] grouped-GEMM counters, zeroed here every forward
};

// The plan of chunk b, by one block of kPermThreads threads. kSingleChunk: the whole
// problem is one chunk; the block counts its own histogram (no hist_kernel ran before it).
// publish: write the plan to the workspace (counts, starts, offsets, tile lists, perm_src,
// perm_inv; clear the status word, flag invalid ids, zero the GEMM counters). s_src (or
// NULL): also receives perm_src in shared memory. Returns the number of valid rows P'.
template <bool kSingleChunk>
__device__ __forceinline__ int plan_body(const PlanArgs& a, int b, bool publish,
                                         int32_t* s_src) {
  __shared__ int32_t s_run[256];                // next free row per expert in this chunk
  __shared__ int32_t s_wcnt[kPermWarps][256];   // rows per (warp, expert) in a sub-chunk
  __shared__ int s_warp[kPermWarps + 1];
  const int tid = threadIdx.x;
  const int E = a.E;

  // Column sums and this chunk's prefix over earlier chunks.
  int tot = 0, before = 0;
  if (kSingleChunk) {
    for (int e = tid; e < 256; e += blockDim.x) s_run[e] = 0;
    if (publish && tid < 4) a.status[tid] = 0;
    __syncthreads();
    for (int64_t f = tid; f < a.P; f += blockDim.x) {
      const int e = a.ids[f];
      if (e >= a.e_lo && e < a.e_hi) atomicAdd(&s_run[e], 1);
    }
    __syncthreads();
    if (tid < E) tot = s_run[tid];
    __syncthreads();
  } else if (tid < E) {
    for (int c = 0; c < a.nb; ++c) {
      const int v = a.block_hist[c * E + tid];
      if (c < b) before += v;
      tot += v;
    }
  }
  int p_valid = 0;
  const int off = block_exclusive_scan(tot, E, s_warp, &p_valid);
  if (tid < E) s_run[tid] = off + before;
  for (int i = tid; i < kPermWarps * 256; i += blockDim.x) (&s_wcnt[0][0])[i] = 0;

  if (b == 0 && publish) {
    // Group table: routed experts 0..E-1, then the shared expert (all T tokens, rows
    // starting at P). Tiles per group: full 128-row tiles plus one remainder tile, times
    // the output-channel tiles of the GEMM.
    const int G = E + a.has_shared;
    int cnt = 0, start = 0, np1 = 0, ns1 = 0, np2 = 0, ns2 = 0;
    if (tid < E) {
      cnt = tot;
      start = off;
      a.offsets[tid] = off;
    } else if (tid == E && a.has_shared) {
      cnt = a.T;
      start = static_cast<int>(a.P);
    }
    if (tid == E) a.offsets[E] = p_valid;
    if (tid < G) {
      a.counts[tid] = cnt;
      a.starts[tid] = start;
      // Work of the grouped GEMM, per output-channel tile. A group of >= pair_min_rows
      // rows goes to the CTA-pair kernel: floor(m / 256) units of two full 128-row tiles
      // plus one unit for the rows left over. Any other group goes to the single-SM
      // kernel: one tile per 128 rows (full tiles and/or the partial last one), or, for a
      // group of at most narrow_rows rows, one narrow weight-major tile per channel tile
      // of the narrow width.
      const int nI = (tid < E) ? a.I : a.shared_I;
      const int c1 = (nI + kFc1Cols - 1) / kFc1Cols;
      const int c2 = (a.H + kFc2Cols - 1) / kFc2Cols;
      if (cnt >= a.pair_min_rows) {
        const int units = (cnt >> 8) + ((cnt & 255) != 0);
        np1 = units * c1;
        np2 = units * c2;
      } else if (cnt > 0 && cnt <= a.narrow_rows) {
        ns1 = (nI + kFc1NarrowCols - 1) / kFc1NarrowCols;
        ns2 = (a.H + kFc2NarrowCols - 1) / kFc2NarrowCols;
      } else {
        const int tiles = cnt / kTileRows + (cnt % kTileRows != 0);
        ns1 = tiles * c1;
        ns2 = tiles * c2;
      }
    }
    int t_p1 = 0, t_s1 = 0, t_p2 = 0, t_s2 = 0;
    const int o_p1 = block_exclusive_scan(np1, G, s_warp, &t_p1);
    const int o_s1 = block_exclusive_scan(ns1, G, s_warp, &t_s1);
    const int o_p2 = block_exclusive_scan(np2, G, s_warp, &t_p2);
    const int o_s2 = block_exclusive_scan(ns2, G, s_warp, &t_s2);
    if (tid < G) {
      a.tile_off1[tid] = o_p1;
      a.tile_off1[G + 1 + tid] = o_s1;
      a.tile_off2[tid] = o_p2;
      a.tile_off2[G + 1 + tid] = o_s2;
    }
    if (tid == 0) {
      a.tile_off1[G] = t_p1;
      a.tile_off1[2 * G + 1] = t_s1;
      a.tile_off2[G] = t_p2;
      a.tile_off2[2 * G + 1] = t_s2;
    }
    for (int i = tid; i < kSchedCounters + G; i += blockDim.x) a.sched[i] = 0;
  }
  __syncthreads();

  // Stable ranks inside the chunk, kPermThreads pairs at a time.
  const int lane = tid & 31, warp = tid >> 5;
  const int64_t f0 = static_cast<int64_t>(b) * kPermChunk;
  const int64_t f1 = (a.P < f0 + kPermChunk ? a.P : f0 + kPermChunk);
  for (int64_t base = f0; base < f1; base += kPermThreads) {
    const int64_t f = base + tid;
    int e = -1;
    if (f < f1) {
      e = a.ids[f];
      if (e < 0 || e >= E) {
        if (publish) {
          a.perm_inv[f] = -1;
          atomicOr(a.status, MOE_DEVICE_FLAG_BAD_ID);
        }
        e = -1;
      } else if (e < a.e_lo || e >= a.e_hi) {
        if (publish) a.perm_inv[f] = -1;   // another call's expert: this slot adds 0 here
        e = -1;
      }
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
    const bool leader = rank_in_warp == 0;
    if (e >= 0 && leader) s_wcnt[warp][e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int pos = s_run[e] + rank_in_warp;
      for (int w = 0; w < warp; ++w) pos += s_wcnt[w][e];
      if (publish) {
        a.perm_src[pos] = static_cast<int32_t>(f);
        a.perm_inv[f] = pos;
      }
      if (s_src) s_src[pos] = static_cast<int32_t>(f);
    }
    __syncthreads();
    if (tid < E) {
      int add = 0;
      for (int w = 0; w < kPermWarps; ++w) {
        add += s_wcnt[w][tid];
        s_wcnt[w][tid] = 0;
      }
      s_run[tid] += add;
    }
    __syncthreads();
  }
  return p_valid;
}

template <bool kSingleChunk>
__global__ void __launch_bounds__(kPermThreads) plan_kernel(PlanArgs a) {
  pdl_trigger();
  pdl_wait();
  plan_body<kSingleChunk>(a, blockIdx.x, true, nullptr);
}

// Plan and row copy in one launch, for a problem of one chunk copied row by row (decode
// batches): every block computes the (small) plan itself, block 0 also publishes it, and
// each block then copies its rows, x_perm[r] = x[perm_src[r] / k] (and x[t] for the shared
// rows), from its own copy of perm_src. One kernel boundary fewer on the way to the GEMM.
__global__ void __launch_bounds__(kPermThreads)
plan_gather_kernel(PlanArgs a, const __nv_bfloat16* __restrict__ x, int64_t rows, int H,
                   __nv_bfloat16* __restrict__ x_perm) {
  __shared__ int32_t s_src[kPermChunk];
  pdl_trigger();
  pdl_wait();
  const int p_valid = plan_body<true>(a, 0, blockIdx.x == 0, s_src);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int nvec = H / 8;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       r < rows; r += warps) {
    int64_t src;
    if (r < a.P) {
      if (r >= p_valid) continue;
      src = s_src[r] / a.k;
    } else {
      src = r - a.P;
    }
    const uint4* sp = reinterpret_cast<const uint4*>(x + src * H);
    uint4* d = reinterpret_cast<uint4*>(x_perm + r * H);
    int v = lane;
    for (; v + 224 < nvec; v += 256) {
      uint4 q8[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) q8[q] = __ldg(sp + v + 32 * q);
#pragma unroll
      for (int q = 0; q < 8; ++q) __stcs(d + v + 32 * q, q8[q]);
    }
    for (; v < nvec; v += 32) d[v] = __ldg(sp + v);
  }
}

__global__ void __launch_bounds__(256)
gather_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ perm_src,
              const int32_t* __restrict__ offsets, int64_t P, int E, int k, int64_t rows,
              int H, __nv_bfloat16* __restrict__ x_perm) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  pdl_trigger();
  pdl_wait();
  const int64_t p_valid = offsets[E];
  const int nvec = H / 8;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       r < rows; r += warps) {
    int64_t src;
    if (r < P) {
      if (r >= p_valid) continue;
      src = perm_src[r] / k;
    } else {
      src = r - P;
    }
    const uint4* s = reinterpret_cast<const uint4*>(x + src * H);
    uint4* d = reinterpret_cast<uint4*>(x_perm + r * H);
    // Four independent 16-byte loads in flight per lane before their stores.
    int v = lane;
    for (; v + 224 < nvec; v += 256) {
      uint4 a[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) a[q] = __ldg(s + v + 32 * q);
#pragma unroll
      for (int q = 0; q < 8; ++q) __stcs(d + v + 32 * q, a[q]);
    }
    for (; v + 96 < nvec; v += 128) {
      const uint4 a0 = __ldg(s + v), a1 = __ldg(s + v + 32), a2 = __ldg(s + v + 64),
                  a3 = __ldg(s + v + 96);
      d[v] = a0;
      d[v + 32] = a1;
      d[v + 64] = a2;
      d[v + 96] = a3;
    }
    for (; v < nvec; v += 32) d[v] = __ldg(s + v);
  }
}

// Token-major row copy (see the header): warp w takes tokens w, w + warps, ...; lane j < k
// reads perm_inv[t*k + j] and every lane gets all k destination rows by shuffles. Each
// 16-byte vector of x[t] is loaded once and stored to every destination (streaming
// stores). Slots whose id was invalid or belongs to another call (perm_inv = -1) write
// nothing.
__global__ void __launch_bounds__(256)
scatter_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ perm_inv,
               int64_t T, int k, int64_t P, int has_shared, int H,
               __nv_bfloat16* __restrict__ x_perm) {
  constexpr int kMaxDst = 9;   // up to 8 slots and the shared row
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  pdl_trigger();
  pdl_wait();
  const int nvec = H / 8;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       t < T; t += warps) {
    const int32_t mine = lane < k ? perm_inv[t * k + lane] : -1;
    int32_t dst[kMaxDst];   // permuted rows (< 2^31), -1 = none
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[j] = __shfl_sync(0xffffffffu, mine, j);
    dst[8] = has_shared ? static_cast<int32_t>(P + t) : -1;
    const uint4* s = reinterpret_cast<const uint4*>(x + t * H);
    int v = lane;
    for (; v + 224 < nvec; v += 256) {
      uint4 a[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) a[q] = __ldg(s + v + 32 * q);
#pragma unroll
      for (int j = 0; j < kMaxDst; ++j) {
        if (dst[j] < 0) continue;
        uint4* d = reinterpret_cast<uint4*>(x_perm + static_cast<int64_t>(dst[j]) * H);
#pragma unroll
        for (int q = 0; q < 8; ++q) __stcs(d + v + 32 * q, a[q]);
      }
    }
    for (; v < nvec; v += 32) {
      const uint4 a = __ldg(s + v);
#pragma unroll
      for (int j = 0; j < kMaxDst; ++j)
        if (dst[j] >= 0) __stcs(reinterpret_cast<uint4*>(x_perm + static_cast<int64_t>(dst[j]) * H) + v, a);
    }
  }
}

}  // namespace

moe_status launch_permute(const moe_problem& p, const moe_ws_layout& L, const void* x,
                          const int32_t* ids, int e_lo, int e_hi, char* ws, cudaStream_t s) {
  const int64_t P = p.T * p.k;
  const int nb = L.n_chunks;
  PlanArgs a;
  a.ids = ids;
  a.P = P;
  a.T = static_cast<int>(p.T);
  a.E = p.E;
  a.e_lo = e_lo;
  a.e_hi = e_hi;
  a.k = p.k;
  a.nb = nb;
  a.has_shared = p.shared_I > 0;
  a.I = p.I;
  a.shared_I = p.shared_I;
  a.H = p.H;
  a.pair_min_rows = pair_min_rows(p);
  a.narrow_rows = narrow_max_rows(p);
  a.block_hist = reinterpret_cast<const int32_t*>(ws + L.block_hist);
  a.counts = reinterpret_cast<int32_t*>(ws + L.counts);
  a.starts = reinterpret_cast<int32_t*>(ws + L.starts);
  a.offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  a.tile_off1 = reinterpret_cast<int32_t*>(ws + L.tile_off1);
  a.tile_off2 = reinterpret_cast<int32_t*>(ws + L.tile_off2);
  a.perm_src = reinterpret_cast<int32_t*>(ws + L.perm_src);
  a.perm_inv = reinterpret_cast<int32_t*>(ws + L.perm_inv);
  a.status = reinterpret_cast<int32_t*>(ws + L.status);
  a.sched = reinterpret_cast<int32_t*>(ws + L.sched);
  cudaError_t err;
  if (nb == 1 && p.T < kScatterMinTokens) {
    // One chunk, row-by-row copy: plan and copy in one launch (16 warps of rows per block).
    const int64_t rows = L.rows;
    int64_t blocks = (rows + kPermWarps - 1) / kPermWarps;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 4;
    if (blocks > cap) blocks = cap;
    err = launch_pdl(plan_gather_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kPermThreads),
                     0, s, a, static_cast<const __nv_bfloat16*>(x), rows, p.H,
                     reinterpret_cast<__nv_bfloat16*>(ws + L.x_perm));
    if (err != cudaSuccess)
      return set_error(MOE_ERR_CUDA, "permute launch: %s", cudaGetErrorString(err));
    return MOE_OK;
  }
  if (nb == 1) {
    err = launch_pdl(plan_kernel<true>, dim3(1), dim3(kPermThreads), 0, s, a);
  } else {
    err = launch_pdl(hist_kernel, dim3(nb), dim3(kPermThreads), 0, s, ids, P, p.E, e_lo, e_hi,
                     reinterpret_cast<int32_t*>(ws + L.block_hist), a.status);
    if (err == cudaSuccess) err = launch_pdl(plan_kernel<false>, dim3(nb), dim3(kPermThreads), 0, s, a);
  }
  if (err == cudaSuccess) {
    const int sms = device_sm_count();
    const int64_t cap = static_cast<int64_t>(sms) * 16;
    if (p.T >= kScatterMinTokens) {
      int64_t blocks = (p.T + 7) / 8;
      if (blocks > cap) blocks = cap;
      err = launch_pdl(scatter_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                       static_cast<const __nv_bfloat16*>(x), static_cast<const int32_t*>(a.perm_inv),
                       p.T, p.k, P, a.has_shared, p.H, reinterpret_cast<__nv_bfloat16*>(ws + L.x_perm));
    } else {
      const int64_t rows = L.rows;
      int64_t blocks = (rows + 7) / 8;
      if (blocks > cap) blocks = cap;
      err = launch_pdl(gather_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                       static_cast<const __nv_bfloat16*>(x), static_cast<const int32_t*>(a.perm_src),
                       static_cast<const int32_t*>(a.offsets), P, p.E, p.k, rows, p.H,
                       reinterpret_cast<__nv_bfloat16*>(ws + L.x_perm));
    }
  }
  if (err != cudaSuccess) return set_error(MOE_ERR_CUDA, "permute launch: %s", cudaGetErrorString(err));
  return MOE_OK;
}

}  // namespace moe
