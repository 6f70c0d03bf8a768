// Router gate (vLLM MoE page, section "Gate 计算与 FSE"): router_logits = x . wg^T, one
// GEMM for the routed experts' gate and, with the fused shared-expert gate (FSE), the
// shared expert's gate as one more row of wg ([E + n_shared, H]).
//
// The contraction is long in K (H) and small in M x N (T x (E + n_shared)), so a tile of
// 128 tokens x up to 256 gate rows is split along K over the S CTAs of a thread-block
// cluster: each CTA runs tcgen05 MMAs (operands staged by TMA, fp32 accumulator in TMEM)
// over its share of the K blocks, copies its partial tile into its own shared memory,
// and after a cluster barrier reduces 128 / S of the tile's rows over the S partials
// (read through distributed shared memory) in rank order, so the sums are deterministic.
// Rows past T and columns past E + n_shared are zero-filled by the tensor maps and not
// stored.
//
// Gate with routing (moe_gate_route): after the reduction each CTA holds its rows' complete
// routed logits (all E <= 256 routed columns lie in column tile 0) in shared memory, and
// its warps route those tokens there (one warp per token, the selection and weights of
// route_device.cuh), so the logits need not go through HBM to a second launch.
#include <atomic>
#include <cstdint>

#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"
#include "route_device.cuh"
#include "tmap.cuh"

namespace moe {
namespace {

constexpr int kGateBK = 64;                  // K elements per slot
constexpr int kGateRowBytes = kGateBK * 2;
// The ring holds up to 8 slots of one K block each (an X box and a W box); a pipeline
// stage is one slot, or two consecutive slots when at least six fit, so that the MMA
// thread, whose instruction latency (a try_wait, four tiny MMAs and a commit per stage)
// bounds the K loop, waits and commits once per eight MMAs.
constexpr int kGateMaxSlots = 8;
constexpr int kGateMaxStages = kGateMaxSlots;
constexpr int kGateXBytes = 128 * kGateRowBytes;       // 128 token rows
constexpr int kGateWMaxBytes = 256 * kGateRowBytes;    // up to 256 gate rows
constexpr int kGateRingBytes = 4 * (kGateXBytes + kGateWMaxBytes);   // 192 KB of stages
constexpr int kGateSmemBytes = 1024 + kGateRingBytes;
constexpr int kGateMaxSplit = 8;             // portable cluster size
// Routing scratch of the fused gate + route kernel, inside the (by then idle) stage ring,
// past the partial tile (at most 128 rows x 260 floats = 130 KB): per warp 256 keys, 256
// exact-key flags and a 256-entry list; then the per-token slot records of up to 128 rows.
constexpr int kGateRouteScratch = 136 * 1024;

// Routing done in the fused kernel's epilogue.
enum GateRoute { kGateNoRoute = 0, kGateRoutePlain = 1, kGateRouteKeyed = 2, kGateRouteGroupedTopk = 3 };

// Threads per CTA. Warps 0-3 run the GEMM (producer, MMA issuer) and read the accumulator
// out of TMEM (warp w reaches TMEM lanes 32w..32w+31). With routing fused in, 16 warps: the
// routing of one token is a long dependent chain (up to about 2,600 instructions for the
// grouped methods), so the CTA's tokens (128 / cluster size of them) are spread over as
// many warps as possible, ideally one token each.
constexpr int gate_threads(int route) { return route == kGateNoRoute ? 128 : 512; }
constexpr int kGateRouteWarps = 16;
static_assert(kGateRouteScratch >= 128 * (256 + 4) * 4, "routing scratch overlaps the partial tile");
constexpr int kGateWarpScratch = 256 * 4 + 256 + 256;            // keys, flags, list
constexpr int kGateSlotsOff = kGateRouteScratch + kGateRouteWarps * kGateWarpScratch;
constexpr int kGateSlots = 128 * 8;                                 // rows x kMaxTopK
constexpr int kGateSlotBytes = kGateSlots * (4 + 4 + 8 + 4) + 128 * 8;   // sel, l, e, ek; z
static_assert(kGateSlotsOff % 16 == 0, "slot records must stay aligned");
static_assert(kGateSlotsOff + kGateSlotBytes <= kGateRingBytes, "routing scratch past the ring");
static_assert(kGateBK == static_cast<int>(kMapBoxCols), "tensor-map boxes are one K block wide");

struct GateArgs {
  int64_t T;
  int H;
  int E;            // routed gate rows
  int E_out;        // E + n_shared
  int n_col;        // column tiles of 256
  int S;            // CTAs per cluster (K split)
  int box_rows;     // gate rows per tensor-map box (min(256, round_up(E_out, 16)))
  int stage_bytes;  // one slot: X box + W box, rounded up to 1024 (the swizzle atom)
  int per_stage;    // K blocks (slots) per pipeline stage: 1 or 2
  int stages;       // pipeline stages: as many slots as fit in the ring (at most 8) / per_stage
  uint32_t tmem_cols;
  float* logits;          // [T, E], or NULL (fused routing without the logits written)
  float* shared_logits;   // [T] or NULL
  int32_t* status;        // device status word or NULL
  // routing (fused kernel only)
  int method, k, n_group, topk_group;
  float rsf;
  const float* bias;      // [E] or NULL
  int32_t* ids;           // [T, k]
  float* scales;          // [T, k]
};

// kRoute: GateRoute; EPL: routed experts per lane of the routing warps (E <= 32 * EPL).
template <int EPL, int kRoute>
__global__ void __launch_bounds__(gate_threads(kRoute), 1)
gate_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
            GateArgs g) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kGateMaxStages], empty_bar[kGateMaxStages], acc_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int S = g.S;
  const uint32_t rank = cluster_ctarank();
  const int cluster = static_cast<int>(blockIdx.x) / S;
  const int col_tile = cluster % g.n_col;
  const int row_tile = cluster / g.n_col;
  const int col0 = col_tile * 256;
  const int n_cols = min(256, g.E_out - col0);
  const int n_mma = (n_cols + 15) & ~15;
  const int row0 = row_tile * 128;
  const int nkb = g.H / kGateBK;
  const int kb0 = static_cast<int>(rank) * nkb / S;
  const int kb1 = (static_cast<int>(rank) + 1) * nkb / S;

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  float* partial = reinterpret_cast<float*>(smem);   // [128][n_mma + 4], after the MMAs
  const int pstride = n_mma + 4;

  pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < g.stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&acc_bar, 1);
    s_abort = 0;
    fence_barrier_init();
    tma_prefetch_map(&map_x);
    tma_prefetch_map(&map_w);
  }
  if (warp == 0) {
    tmem_alloc(&s_tmem, g.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort = &s_abort;
  pdl_wait();   // x may be the previous kernel's output

  const int G = g.per_stage;
  if (warp == 0 && lane == 0) {
    // TMA producer over this CTA's K blocks, G per stage.
    const uint32_t bytes = static_cast<uint32_t>(kGateXBytes + g.box_rows * kGateRowBytes);
    int issued = 0, st = 0;
    uint32_t ph = 0;
    for (int kb = kb0; kb < kb1; kb += G, ++issued) {
      const int nk = kb1 - kb < G ? kb1 - kb : G;
      if (!mbar_wait(&empty_bar[st], ph ^ 1u, abort)) {
        *abort = 1;
        break;
      }
      mbar_arrive_expect_tx(&full_bar[st], static_cast<uint32_t>(nk) * bytes);
      for (int b = 0; b < nk; ++b) {
        uint8_t* xs = smem + (st * G + b) * g.stage_bytes;
        tma_load_2d(xs, &map_x, &full_bar[st], (kb + b) * kGateBK, row0);
        tma_load_2d(xs + kGateXBytes, &map_w, &full_bar[st], (kb + b) * kGateBK, col0);
      }
      if (++st == g.stages) {
        st = 0;
        ph ^= 1u;
      }
    }
    if (*abort) {
      // Let the copies in flight land before shared memory is reused (bounded waits).
      volatile int never = 0;
      const int first = issued > g.stages ? issued - g.stages : 0;
      for (int i = first; i < issued; ++i)
        mbar_wait(&full_bar[i % g.stages], (i / g.stages) & 1, &never);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer: D[128 tokens, n_mma gate rows] += X . W^T.
    const uint32_t idesc = idesc_bf16_f32(128, n_mma);
    // Descriptors of slot 0's X and W tiles; a slot's are these plus its offset / 16 (the
    // start-address field holds shared-address bits 4-17, and the ring lies below 228 KB).
    const uint64_t dx0 = sdesc_k_major(smem_u32(smem), kGateRowBytes);
    const uint64_t dw0 = sdesc_k_major(smem_u32(smem) + kGateXBytes, kGateRowBytes);
    const uint32_t slot_step = static_cast<uint32_t>(g.stage_bytes) >> 4;
    int st = 0;
    uint32_t ph = 0;
    for (int kb = kb0; kb < kb1; kb += G) {
      const int nk = kb1 - kb < G ? kb1 - kb : G;
      if (!mbar_wait(&full_bar[st], ph, abort)) {
        *abort = 1;
        break;
      }
      tc_fence_after();
      for (int b = 0; b < nk; ++b) {
        const uint64_t so = static_cast<uint64_t>((st * G + b) * slot_step);
#pragma unroll
        for (int kk = 0; kk < kGateBK / 16; ++kk)
          umma_bf16(tmem, dx0 + so + 2 * kk, dw0 + so + 2 * kk, idesc,
                    (kb != kb0 || b != 0 || kk != 0) ? 1u : 0u);
      }
      umma_commit(&empty_bar[st]);
      if (++st == g.stages) {
        st = 0;
        ph ^= 1u;
      }
    }
    umma_commit(&acc_bar);   // arrives once every MMA issued above has completed
  }
  __syncwarp();

  // Partial tile: TMEM lane (token row) 32 * warp + lane, columns 0..n_mma-1, read by
  // warps 0-3. Warps past them (routing) go straight to the cluster barrier instead of
  // polling the accumulator barrier beside the producer and the MMA issuer.
  if (warp < 4) {
    const bool done = mbar_wait(&acc_bar, 0, abort);
    if (!__all_sync(0xffffffffu, done)) *abort = 1;
    tc_fence_after();
    const int row = 32 * warp + lane;
    float v[16];
    for (int c0 = 0; c0 < n_mma; c0 += 16) {
      tmem_ld_x16(tmem + (static_cast<uint32_t>(32 * warp) << 16) + c0, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) partial[row * pstride + c0 + i] = v[i];
    }
  }
  tc_fence_before();
  cluster_sync();   // every CTA's partial tile is in its shared memory

  // This CTA's rows of the tile, summed over the S partials in rank order: four columns
  // per thread and step, the S partials' loads issued before the adds.
  const int r0 = static_cast<int>(rank) * 128 / S, r1 = (static_cast<int>(rank) + 1) * 128 / S;
  const uint32_t pbase = smem_u32(partial);
  const int nq = n_mma / 4;   // column quads of the partial tile
  for (int idx = tid; idx < (r1 - r0) * nq; idx += blockDim.x) {
    const int row = r0 + idx / nq;
    const int col = (idx - (row - r0) * nq) * 4;
    const uint32_t off = static_cast<uint32_t>((row * pstride + col) * 4);
    float4 part[kGateMaxSplit];
#pragma unroll
    for (int q = 0; q < kGateMaxSplit; ++q)
      if (q < S) part[q] = ld_shared_cluster_f32x4(mapa_shared(pbase + off, q));
    float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < kGateMaxSplit; ++q)
      if (q < S) {
        sum[0] += part[q].x;
        sum[1] += part[q].y;
        sum[2] += part[q].z;
        sum[3] += part[q].w;
      }
    const int64_t t = row0 + row;
    if (t < g.T) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = col0 + col + j;
        if (col + j >= n_cols) break;
        if (c < g.E) {
          if (kRoute == kGateNoRoute || g.logits) g.logits[t * g.E + c] = sum[j];
        } else if (g.shared_logits) {
          g.shared_logits[t] = sum[j];
        }
      }
    }
    if (kRoute != kGateNoRoute) {
      // The reduced row replaces this CTA's own partial in place: rows [r0, r1) of this
      // CTA's tile are read by this thread only (the other CTAs reduce other rows).
      float* dst = partial + row * pstride + col;
      dst[0] = sum[0];
      dst[1] = sum[1];
      dst[2] = sum[2];
      dst[3] = sum[3];
    }
  }
  if (kRoute != kGateNoRoute && col_tile == 0) {
    // Route this CTA's tokens on their reduced logits (columns 0..E-1 of the rows): one warp
    // selects each token's experts, then the block computes the weights of all the (token,
    // slot) pairs packed across its threads.
    __syncthreads();
    const int nwarps = gate_threads(kRoute) / 32;
    uint8_t* ws = smem + kGateRouteScratch + warp * kGateWarpScratch;
    float* skey = reinterpret_cast<float*>(ws);
    uint8_t* sexact = ws + 256 * 4;
    uint8_t* slist = ws + 256 * 4 + 256;
    uint8_t* so = smem + kGateSlotsOff;
    const PairSlots ps{reinterpret_cast<int*>(so),
                       reinterpret_cast<float*>(so + kGateSlots * 4),
                       reinterpret_cast<double*>(so + kGateSlots * 8),
                       reinterpret_cast<float*>(so + kGateSlots * 16),
                       reinterpret_cast<double*>(so + kGateSlots * 20)};
    for (int row = r0 + warp; row < r1; row += nwarps) {
      const int64_t t = row0 + row;
      if (t >= g.T) break;
      const float* lrow = partial + row * pstride;
      int sel[kMaxTopK];
      if (kRoute == kGateRouteGroupedTopk) {
        grouped_topk_select_token<EPL>(lrow, g.E, g.k, g.n_group, g.topk_group, lane, skey, sel);
      } else {
        double z = 0.0;
        select_token<EPL, kRoute == kGateRouteKeyed>(lrow, g.E, g.bias, g.method, g.k, g.n_group,
                                                     g.topk_group, lane, skey, sexact, slist, sel,
                                                     &z);
        if (kRoute == kGateRoutePlain && g.method == MOE_ROUTE_DEFAULT && lane == 0)
          ps.z[row - r0] = z;
      }
      record_selection(lrow, sel, g.k, lane, ps, row - r0);
      __syncwarp();
    }
    __syncthreads();
    block_pair_weights<kRoute == kGateRouteGroupedTopk ? 2 : kRoute == kGateRouteKeyed ? 1 : 0>(
        r1 - r0, row0 + r0, g.T, g.k, g.method, g.rsf, ps, g.ids, g.scales);
  }
  cluster_sync();   // no CTA leaves while another reads its shared memory
  if (tid == 0 && *abort && g.status) atomicOr(g.status, MOE_DEVICE_FLAG_TIMEOUT);
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, g.tmem_cols);
  }
}

// The dynamic shared-memory opt-in of one instantiation, once per device (published after
// it is set; a thread that finds it unset sets it again, which is harmless).
template <int EPL, int kRoute>
cudaError_t gate_smem_optin() {
  static std::atomic<bool> done[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(gate_kernel<EPL, kRoute>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kGateSmemBytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
  return e;
}

// How many clusters of S CTAs of one instantiation can be resident at once, once per device
// and S (0 if the query fails: then no limit is applied).
template <int EPL, int kRoute>
int gate_max_clusters(int S) {
  static std::atomic<int> known[64][4];   // value + 1; 0 = not yet queried
  int dev = 0;
  cudaGetDevice(&dev);
  const int si = S <= 1 ? 0 : S == 2 ? 1 : S == 4 ? 2 : 3;
  const bool cache = dev >= 0 && dev < 64;
  if (cache) {
    const int v = known[dev][si].load(std::memory_order_acquire);
    if (v) return v - 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(S));
  cfg.blockDim = dim3(gate_threads(kRoute));
  cfg.dynamicSmemBytes = kGateSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gate_kernel<EPL, kRoute>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (cache) known[dev][si].store(n + 1, std::memory_order_release);
  return n;
}

template <int EPL, int kRoute>
cudaError_t launch_gate_t(const cudaLaunchConfig_t& cfg0, const CUtensorMap& mx,
                          const CUtensorMap& mw, const GateArgs& g0) {
  const cudaError_t e = gate_smem_optin<EPL, kRoute>();
  if (e != cudaSuccess) return e;
  // All clusters resident at once: clusters that do not fit wait for a second wave (16
  // clusters of 8 CTAs started up to 9 us apart). Halve the K split until they fit.
  GateArgs g = g0;
  const int clusters = static_cast<int>(cfg0.gridDim.x) / g.S;
  while (g.S > 1) {
    const int fit = gate_max_clusters<EPL, kRoute>(g.S);
    if (fit == 0 || clusters <= fit) break;
    g.S >>= 1;
  }
  cudaLaunchConfig_t cfg = cfg0;
  cfg.blockDim = dim3(gate_threads(kRoute));
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * g.S));
  cudaLaunchAttribute attr[2];
  for (unsigned i = 0; i < cfg0.numAttrs && i < 2; ++i) {
    attr[i] = cfg0.attrs[i];
    if (attr[i].id == cudaLaunchAttributeClusterDimension)
      attr[i].val.clusterDim.x = static_cast<unsigned>(g.S);
  }
  cfg.attrs = attr;
  return cudaLaunchKernelEx(&cfg, gate_kernel<EPL, kRoute>, mx, mw, g);
}

template <int kRoute>
cudaError_t launch_gate_e(const cudaLaunchConfig_t& cfg, const CUtensorMap& mx,
                          const CUtensorMap& mw, const GateArgs& g) {
  if (g.E <= 32) return launch_gate_t<1, kRoute>(cfg, mx, mw, g);
  if (g.E <= 64) return launch_gate_t<2, kRoute>(cfg, mx, mw, g);
  if (g.E <= 128) return launch_gate_t<4, kRoute>(cfg, mx, mw, g);
  return launch_gate_t<8, kRoute>(cfg, mx, mw, g);
}

}  // namespace

moe_status launch_gate(const void* x, const void* wg, int64_t T, int H, int E, int n_shared,
                       float* logits, float* shared_logits, int32_t* status, cudaStream_t s,
                       const GateRouteArgs* route) {
  GateArgs g;
  g.T = T;
  g.H = H;
  g.E = E;
  g.E_out = E + n_shared;
  g.n_col = (g.E_out + 255) / 256;
  const int n_row = static_cast<int>((T + 127) / 128);
  const int nkb = H / kGateBK;
  // Enough CTAs to cover the SMs, at least two K blocks each, at most the portable cluster.
  const int clusters = n_row * g.n_col;
  const int want = (device_sm_count() + clusters - 1) / clusters;
  int S = 1;   // a power of two: 1, 2, 4 or 8 CTAs per cluster
  while (S * 2 <= want && S * 2 <= kGateMaxSplit && S * 2 <= nkb / 2) S *= 2;
  g.S = S;
  const int e16 = (g.E_out + 15) & ~15;
  g.box_rows = e16 < 256 ? e16 : 256;
  g.stage_bytes = (kGateXBytes + g.box_rows * kGateRowBytes + 1023) & ~1023;
  int slots = kGateRingBytes / g.stage_bytes;
  if (slots > kGateMaxSlots) slots = kGateMaxSlots;
  g.per_stage = slots >= 6 ? 2 : 1;
  g.stages = slots / g.per_stage;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(g.box_rows)) cols <<= 1;
  g.tmem_cols = cols;
  g.logits = logits;
  g.shared_logits = shared_logits;
  g.status = status;
  g.method = 0;
  g.k = 0;
  g.n_group = 1;
  g.topk_group = 1;
  g.rsf = 1.0f;
  g.bias = nullptr;
  g.ids = nullptr;
  g.scales = nullptr;
  int mode = kGateNoRoute;
  if (route) {
    const moe_route_params& p = route->params;
    const bool keyed = p.method == MOE_ROUTE_DEEPSEEKV3 || p.method == MOE_ROUTE_MINIMAX2;
    const bool dsv3 = p.method == MOE_ROUTE_DEEPSEEKV3;
    const bool vgrp = p.method == MOE_ROUTE_GROUPED_TOPK;
    mode = vgrp ? kGateRouteGroupedTopk : keyed ? kGateRouteKeyed : kGateRoutePlain;
    g.method = p.method;
    g.k = p.top_k;
    // as in moe_route: groups and the scaling factor belong to DeepSeekV3 and the grouped
    // top-k; MiniMax2 has one group and its bias is optional
    g.n_group = (dsv3 || vgrp) ? p.n_group : 1;
    g.topk_group = (dsv3 || vgrp) ? p.topk_group : 1;
    g.rsf = (dsv3 || vgrp) ? p.routed_scaling_factor : 1.0f;
    g.bias = keyed ? route->bias : nullptr;
    g.ids = route->ids;
    g.scales = route->scales;
  }
  CUtensorMap mx, mw;
  if (!encode_map2(&mx, x, static_cast<uint64_t>(T), static_cast<uint64_t>(H), 128) ||
      !encode_map2(&mw, wg, static_cast<uint64_t>(g.E_out), static_cast<uint64_t>(H),
                   static_cast<uint32_t>(g.box_rows)))
    return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (gate)");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * S));
  cfg.dynamicSmemBytes = kGateSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t err;
  switch (mode) {
    case kGateRoutePlain: err = launch_gate_e<kGateRoutePlain>(cfg, mx, mw, g); break;
    case kGateRouteKeyed: err = launch_gate_e<kGateRouteKeyed>(cfg, mx, mw, g); break;
    case kGateRouteGroupedTopk: err = launch_gate_e<kGateRouteGroupedTopk>(cfg, mx, mw, g); break;
    default: err = launch_gate_t<1, kGateNoRoute>(cfg, mx, mw, g); break;
  }
  if (err != cudaSuccess) return set_error(MOE_ERR_CUDA, "gate launch: %s", cudaGetErrorString(err));
  return MOE_OK;
}

}  // namespace moe
