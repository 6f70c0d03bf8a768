// Steps 3 and 4: grouped GEMM over all experts; the forward runs both as ONE persistent
// launch (FC1's work list, then FC2's; an FC2 tile of expert g waits on a counter for
// g's FC1 tiles), and moe_fc1 / moe_fc2 run one GEMM each with the same tiles.
// Scheduling (Dense GEMM -> GroupedGEMM article, section 2.2): tile scheduling over
// flattened global work lists rather than one block per expert. The permute step wrote,
// per group g (routed experts, then the optional shared expert), its row count m_g, its
// first permuted row and exclusive scans of its work. One kernel family takes every group
// of a launch: the CTA-pair kernel when T*k >= 256*E, else the single-SM kernel.
//  * CTA-pair kernel: 2-CTA clusters with pair MMAs (tcgen05.mma.cta_group::2, M = 256).
//    Each CTA holds 128 rows of the A operand and half of the B operand in its own shared
//    memory, so a stage is 32 KB per SM and six stages fit; each CTA's TMEM receives its
//    128 rows of the result. A group gives floor(m_g / 256) token-major units (two full
//    128-row tiles, one per CTA,
//        D[256 tokens, 256] = X[256, K] . W[256, K]^T,   A = X, B = W, N = 256)
//    and one unit for the rows left over: 129..255 rows run token-major with the
//    missing rows masked; 1..128 rows run weight-major (swap AB,
//        D[256 weights, n] = W[256, K] . X[n, K]^T,      A = W, B = X,
//    n = rows rounded up to 16, each CTA holding n/2 token rows), per channel tile.
//  * single-SM kernel (decode-sized experts), one SM per tile: a full 128-row tile
//    token-major (D[128, 256] = X . W^T, N = 256) and the partial tile weight-major
//    (D0[128 ch, n] = W[0:128] . X^T, D1 = W[128:256] . X^T, n = rows rounded up to 16);
//    48 KB stages keep 32 KB of weights per stage in flight, which is what a
//    weight-streaming (HBM-bound) tile needs.
//
// Weight rows (w13 = gate and up merged, vLLM MoE page, section "专家权重如何存储") are
// arranged so the SwiGLU epilogue (h = silu(gate) * up) finds gate and up of a channel in
// one thread: token-major tiles load gate rows [n0, n0+128) and up rows [I+n0, I+n0+128)
// as the two halves of N = 256 (columns c and 128+c); single-SM weight-major tiles load
// them as D0 and D1 (same TMEM lane); pair weight-major units load, in CTA r, gate rows
// [n0+64r, +64) and up rows [I+n0+64r, +64) (lanes c and 64+c, swapped through a 4 KB
// shared buffer). FC2 takes w2[e] rows [n0, n0+256) (output channels).
//
// Warp roles (192 threads per CTA): warp 0 = TMA producer (and work claims), warp 1 =
// TMEM allocator and MMA issuer (in a pair, the first CTA issues), warps 2-5 = epilogue
// (TMEM lanes 32*(warp%4) .. +31). Two 256-column TMEM accumulators let the epilogue of
// one unit overlap the next mainloop. Work is claimed dynamically from an atomic counter
// per list (in a pair, the first CTA claims and passes the index to both CTAs through
// DSMEM); claims move through the list in order and faster SMs take more work. The last
// CTA to finish resets the counter.
//
// Rows past a group's end inside a tile read the next group's rows (or zero fill past
// the tensor); they only reach accumulator rows/columns that the epilogue masks.
#include <atomic>
#include <cstdint>
#include <cstdio>

#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace moe {
namespace {

constexpr int kBK = 64;                              // K elements per stage
static_assert(kBK == static_cast<int>(kMapBoxCols), "tensor-map boxes are one K block wide");
constexpr int kRowBytes = kBK * 2;                   // one K row of a tile = the swizzle width
constexpr int kXStageBytes = 128 * kRowBytes;        // 128 rows of X
constexpr int kWStageBytes = 128 * kRowBytes;        // 128 rows of W
// Pair kernel: six 16 KB slots each of X and W rows, one K block per slot; a pipeline
// stage is two consecutive slots (two K blocks), so the MMA thread waits and commits once
// per eight MMAs. That thread's own instruction latency bounds the pair kernel: at one K
// block per stage (a try_wait, four MMAs and a commit, about 600 cycles) it issued more
// slowly than the tensor pipe ran the four 256 x 256 x 16 MMAs.
constexpr int kPairSlots = 6;
constexpr int kPairBlocksPerStage = 2;
constexpr int kStages = kPairSlots / kPairBlocksPerStage;
constexpr int kSingleStages = 4;                     // single kernel: X + 2 W halves, 48 KB
constexpr int kAccCols = 256;
constexpr int kTmemCols = 512;
constexpr int kThreads = 192;
constexpr int kMaxGroups = 257;
constexpr int kSchedDepth = 4;                       // work indices in flight inside a CTA
// Pair kernel: the first CTA claims its next unit this many K blocks before it has issued
// the current unit's loads, so the claim's atomic latency stays off the load stream; a
// whole unit ahead would lengthen the tail (faster pairs could no longer take more work).
// (In the single-SM kernel the same early claim measured no gain.)
constexpr int kClaimLead = 4;
// Epilogue staging of both kernels: per epilogue warp two 32 x 32 bf16 boxes for TMA
// stores, after the stage ring.
constexpr int kStoreBufBytes = static_cast<int>(kStoreBoxRows * kStoreBoxCols * 2);
constexpr int kStageAreaBytes = 4 * 2 * kStoreBufBytes;
constexpr int kSmemBytes =
    1024 /*alignment slack*/ + kPairSlots * (kXStageBytes + kWStageBytes) + kStageAreaBytes;
constexpr int kSingleSmemBytes =
    1024 + kSingleStages * (kXStageBytes + 2 * kWStageBytes) + kStageAreaBytes;
constexpr uint16_t kPairMask = 0x3;
// Consumers that return a scheduling slot to the first CTA: its MMA thread and 4
// epilogue warps, and the second CTA's producer and 4 epilogue warps.
constexpr uint32_t kSchedConsumers = 1 + 4 + 1 + 4;
constexpr int kXchgStride = 17;                      // padded row of the gate/up swap buffer
constexpr int64_t kPrefetchBytes = 48ll << 20;       // narrow FC1 L2 prefetch, whole grid

struct GemmArgs {
  const int32_t* counts;    // [G]
  const int32_t* starts;    // [G]
  const int32_t* tile_off;  // [G+1] offsets into this kernel's work list
  int32_t G;
  int32_t E;                // routed groups; group E (if G > E) uses the shared maps
  int32_t plane_off;        // routed expert g reads weight plane g - plane_off
  int32_t K_routed, K_shared;
  int32_t N_routed, N_shared;   // FC1: I / shared_I (channels); FC2: H
  __nv_bfloat16* out;
  int64_t out_ld;
  int32_t* status;
  int32_t* sched;           // [0] next unit to claim, [1] CTAs finished (both reset at exit)
  int32_t* dep;             // fused single-SM launch: [G] FC1 tiles finished per group
  int32_t planes;           // routed weight planes in the maps (experts of this call)
  int32_t prefetch_kb;      // narrow FC1: K blocks of its guessed first tile each CTA
                            // prefetches into L2 before the work lists exist (0: none)
};

struct Unit {
  int g;
  int token_major;   // 1: two full 128-row tiles; 0: the group's leftover rows, weight-major
  int row0;          // token-major: this CTA's first row; weight-major: the first leftover row
  int rows;          // valid rows (token-major 128; weight-major 1..255)
  int ntok;          // weight-major: rows rounded up to 16 (the MMA N)
  int narrow;        // single-SM only: a narrow weight-major tile (128 weight rows)
  int n0;            // first output channel of the unit
  int K;
  int N;             // channels of this group
};

// Largest g with off[g] <= idx (groups without work have equal offsets).
__device__ __forceinline__ int find_group(int idx, const int32_t* s_off, int G) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_off[mid] <= idx) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// FC2 work of group g in the fused launch reads the h rows its FC1 tiles stored: the
// producer waits (acquire, bounded) until the group's completion counter shows them all,
// then fences the async proxy for its TMA loads. A group's h rows never change after that,
// so each producer remembers the groups it has seen complete (one bit per group in shared
// memory, touched by the producer thread only) and skips the global load for them.
constexpr int kDepWords = (kMaxGroups + 31) / 32;
__device__ __forceinline__ bool wait_group_h(uint32_t* seen, const int32_t* dep, int g, int need,
                                             volatile int* abort) {
  const uint32_t bit = 1u << (g & 31);
  if (seen[g >> 5] & bit) return true;
  if (!wait_count(dep + g, need, abort)) return false;
  fence_proxy_async_global();
  seen[g >> 5] |= bit;
  return true;
}

__device__ __forceinline__ Unit decode_unit(int unit, const int32_t* s_off, const int32_t* s_cnt,
                                            const int32_t* s_start, const GemmArgs& a, bool fc1,
                                            uint32_t rank) {
  const int g = find_group(unit, s_off, a.G);
  const int m = s_cnt[g];
  const int pairs = m >> 8;
  const int left = m - (pairs << 8);
  const int nu = pairs + (left > 0);
  const int local = unit - s_off[g];
  const bool shared = g >= a.E;
  Unit t;
  t.g = g;
  t.K = shared ? a.K_shared : a.K_routed;
  t.N = shared ? a.N_shared : a.N_routed;
  // Order of the group's (row unit u, channel tile nt) grid. The pairs working at the
  // same time should share their operands in L2, so the smaller of the two panels is
  // kept resident: when the group's rows outnumber the expert's weight rows (FC1 2N,
  // FC2 N), the row units go outer and every channel tile of a row unit follows it (the
  // expert's weights stay in L2 and each A row block is read once); otherwise the
  // channel tiles go outer (each weight tile stays in L2 while the row units pass).
  const int cols = fc1 ? kFc1Cols : kFc2Cols;
  int nt, u;
  if (m >= (fc1 ? 2 : 1) * t.N) {
    const int nnt = (t.N + cols - 1) / cols;
    u = local / nnt;
    nt = local - u * nnt;
  } else {
    nt = local / nu;
    u = local - nt * nu;
  }
  t.n0 = nt * cols;
  t.narrow = 0;
  if (u < pairs || left > 128) {
    // Two row tiles, one per CTA; for the leftover unit (129..255 rows) the second tile
    // is partial and its missing rows are masked.
    t.token_major = 1;
    t.row0 = s_start[g] + 256 * u + 128 * static_cast<int>(rank);
    t.rows = u < pairs ? 128 : min(128, left - 128 * static_cast<int>(rank));
    t.ntok = 128;
  } else {
    t.token_major = 0;
    t.row0 = s_start[g] + 256 * pairs;
    t.rows = left;
    t.ntok = (left + 15) & ~15;
  }
  return t;
}

// Single-SM list: every row tile of a group (full 128-row tiles and/or the partial last
// tile), channel-tile major; in a narrow launch a group of at most kNarrowRows rows has one
// narrow weight-major tile per narrow channel tile instead.
__device__ __forceinline__ Unit decode_single(int tile, const int32_t* s_off, const int32_t* s_cnt,
                                              const int32_t* s_start, const GemmArgs& a, bool fc1,
                                              bool narrow_launch) {
  const int g = find_group(tile, s_off, a.G);
  const int m = s_cnt[g];
  if (narrow_launch && m <= kNarrowRows) {
    const bool shared = g >= a.E;
    Unit t;
    t.g = g;
    t.K = shared ? a.K_shared : a.K_routed;
    t.N = shared ? a.N_shared : a.N_routed;
    t.narrow = 1;
    t.token_major = 0;
    t.n0 = (tile - s_off[g]) * (fc1 ? kFc1NarrowCols : kFc2NarrowCols);
    t.row0 = s_start[g];
    t.rows = m;
    t.ntok = (m + 15) & ~15;
    return t;
  }
  const int nfull = m / 128;
  const int n_mt = nfull + (m % 128 != 0);
  const int local = tile - s_off[g];
  const int nt = local / n_mt;
  const int mt = local - nt * n_mt;
  const bool shared = g >= a.E;
  Unit t;
  t.g = g;
  t.K = shared ? a.K_shared : a.K_routed;
  t.N = shared ? a.N_shared : a.N_routed;
  t.n0 = nt * (fc1 ? kFc1Cols : kFc2Cols);
  t.narrow = 0;
  t.token_major = mt < nfull;
  t.row0 = s_start[g] + mt * 128;
  t.rows = min(128, m - mt * 128);
  t.ntok = (t.rows + 15) & ~15;
  return t;
}

__device__ __forceinline__ void flag_timeout(int32_t* status, volatile int* s_abort) {
  *s_abort = 1;
  atomicOr(status, MOE_DEVICE_FLAG_TIMEOUT);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

// Token-major epilogue: thread = token row lrow; TMEM columns = channels (FC1: 0..127
// gate and 128..255 up of channels n0..n0+127; FC2: channels n0..n0+255).
template <bool kFc1>
__device__ __forceinline__ void store_token_major(uint32_t tb, const Unit& t, int lrow,
                                                  const GemmArgs& a) {
  float va[16], vb[16];
  const bool valid = lrow < t.rows;
  __nv_bfloat16* orow = a.out + static_cast<int64_t>(t.row0 + lrow) * a.out_ld;
  if (kFc1) {
#pragma unroll 1
    for (int c0 = 0; c0 < 128; c0 += 16) {
      tmem_ld2_x16(tb + c0, tb + 128 + c0, va, vb);
      if (valid && t.n0 + c0 < t.N) {
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          pk[i] = pack_bf16x2(silu(va[2 * i]) * vb[2 * i], silu(va[2 * i + 1]) * vb[2 * i + 1]);
        uint4* dst = reinterpret_cast<uint4*>(orow + t.n0 + c0);
        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
  } else {
#pragma unroll 1
    for (int c0 = 0; c0 < 256; c0 += 32) {
      tmem_ld2_x16(tb + c0, tb + c0 + 16, va, vb);
      if (valid && t.n0 + c0 < t.N) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          pk[i] = pack_bf16x2(va[2 * i], va[2 * i + 1]);
          pk[8 + i] = pack_bf16x2(vb[2 * i], vb[2 * i + 1]);
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + t.n0 + c0);
        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        dst[2] = make_uint4(pk[8], pk[9], pk[10], pk[11]);
        dst[3] = make_uint4(pk[12], pk[13], pk[14], pk[15]);
      }
    }
  }
}

// Token-major epilogue of a full 128-row tile through shared memory: each epilogue warp
// converts its 32 rows, 32 columns at a time, into one of its two staging boxes (the
// store map's 64-byte swizzle) and its lane 0 writes the 32 x 32 box with one TMA store.
// Stored row by row from registers instead, each store instruction touches 32 rows; at
// short K those instructions keep the SM's load/store pipe busy for much of the next
// tile's mainloop and slow the producer's and MMA issuer's shared-memory traffic.
template <bool kFc1>
__device__ __forceinline__ void store_token_major_tma(uint32_t tb, const Unit& t, int q, int lane,
                                                      uint8_t* stage, int& sbuf,
                                                      const CUtensorMap* map_out) {
  const int sw = (lane >> 1) & 3;
  constexpr int kCols = kFc1 ? kFc1Cols : kFc2Cols;
#pragma unroll 1
  for (int c0 = 0; c0 < kCols; c0 += static_cast<int>(kStoreBoxCols)) {
    if (t.n0 + c0 >= t.N) break;   // N is a multiple of 64: whole boxes only
    uint4 v[4];
    if (kFc1) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float va[16], vb[16];
        tmem_ld2_x16(tb + c0 + 16 * h, tb + 128 + c0 + 16 * h, va, vb);
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          pk[i] = pack_bf16x2(silu(va[2 * i]) * vb[2 * i], silu(va[2 * i + 1]) * vb[2 * i + 1]);
        v[2 * h] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        v[2 * h + 1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    } else {
      float va[16], vb[16];
      tmem_ld2_x16(tb + c0, tb + c0 + 16, va, vb);
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        pk[i] = pack_bf16x2(va[2 * i], va[2 * i + 1]);
        pk[8 + i] = pack_bf16x2(vb[2 * i], vb[2 * i + 1]);
      }
      v[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      v[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      v[2] = make_uint4(pk[8], pk[9], pk[10], pk[11]);
      v[3] = make_uint4(pk[12], pk[13], pk[14], pk[15]);
    }
    uint8_t* buf = stage + sbuf * kStoreBufBytes;
    // The box stored from this buffer two boxes ago must have been read out of it.
    if (lane == 0) bulk_wait_group_read<1>();
    __syncwarp();
    uint4* row = reinterpret_cast<uint4*>(buf + lane * 64);
#pragma unroll
    for (int j = 0; j < 4; ++j) row[j ^ sw] = v[j];
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(map_out, buf, t.n0 + c0, t.row0 + 32 * q);
      bulk_commit_group();
    }
    sbuf ^= 1;
  }
}

// Weight-major epilogue: TMEM lane = one of this CTA's 128 weight rows, columns = tokens.
// FC2: lane L is output channel n0 + 128 * rank + L. FC1: lanes 0-63 are the gate and
// lanes 64-127 the up projection of channels n0 + 64 * rank + (L mod 64); the up half
// passes through `xchg` to the warps holding the gate half (named barrier 1 over the
// four epilogue warps).
template <bool kFc1>
__device__ __forceinline__ void store_weight_major(uint32_t tb, const Unit& t, int lrow,
                                                   uint32_t rank, float* xchg,
                                                   const GemmArgs& a) {
  float va[16];
  if (kFc1) {
    const bool gate_half = lrow < 64;
    const int c = lrow & 63;
    const int ch = t.n0 + 64 * static_cast<int>(rank) + c;
#pragma unroll 1
    for (int c0 = 0; c0 < t.ntok; c0 += 16) {
      tmem_ld_x16(tb + c0, va);
      if (!gate_half) {
#pragma unroll
        for (int i = 0; i < 16; ++i) xchg[c * kXchgStride + i] = va[i];
      }
      named_barrier_sync(1, 128);
      if (gate_half && ch < t.N) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = c0 + i;
          if (r < t.rows)
            a.out[static_cast<int64_t>(t.row0 + r) * a.out_ld + ch] =
                __float2bfloat16_rn(silu(va[i]) * xchg[c * kXchgStride + i]);
        }
      }
      named_barrier_sync(1, 128);
    }
  } else {
    const int ch = t.n0 + 128 * static_cast<int>(rank) + lrow;
#pragma unroll 1
    for (int c0 = 0; c0 < t.ntok; c0 += 16) {
      tmem_ld_x16(tb + c0, va);
      if (ch < t.N) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = c0 + i;
          if (r < t.rows)
            a.out[static_cast<int64_t>(t.row0 + r) * a.out_ld + ch] = __float2bfloat16_rn(va[i]);
        }
      }
    }
  }
}

// Both kernels: the last CTA to finish resets the work counter for the next launch.
__device__ __forceinline__ void finish_claims(const GemmArgs& a) {
  __threadfence();
  if (atomicAdd(a.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
    atomicExch(a.sched, 0);
    atomicExch(a.sched + 1, 0);
  }
}

// ============================================================== single-SM kernel

// Shared-memory descriptor of the tile `off` bytes past the one `desc` describes. The
// start-address field holds bits 4-17 of the shared address, and every operand here lies
// inside the CTA's shared memory (below 228 KB), so adding off / 16 to the base
// descriptor gives what sdesc_k_major would build from the shifted address. The MMA
// issuer's loops are bound by its own instruction latency (a try_wait, four to eight
// MMAs, a commit per stage), so they build no descriptor and divide nothing inside.
__device__ __forceinline__ uint64_t sdesc_at(uint64_t desc, uint32_t off) {
  return desc + (off >> 4);
}

// The K loop of one tile of the single-SM kernel. Token-major: A = 128 X rows, B = the
// 256 W rows of the stage (N = 256). Weight-major: two MMAs, A = each 128-row half of the
// W stage, B = the tile's X rows (N = ntok), into accumulator columns 0 and 128. One loop
// per form, as in the pair kernel. dx0 / dw0 describe stage 0's X and W tiles. Returns
// false if a stage did not arrive in time.
template <bool kTokenMajor>
__device__ __forceinline__ bool single_k_loop(uint32_t d, uint32_t idesc, int nkb, int& stage,
                                              uint32_t& phase, uint64_t dx0, uint64_t dw0,
                                              uint64_t* full_bar, uint64_t* empty_bar,
                                              volatile int* abort) {
  for (int kb = 0; kb < nkb; ++kb) {
    if (!mbar_wait(&full_bar[stage], phase, abort)) return false;
    tc_fence_after();
    const uint64_t xs = sdesc_at(dx0, stage * kXStageBytes);
    const uint64_t wst = sdesc_at(dw0, stage * (2 * kWStageBytes));
#pragma unroll
    for (int kk = 0; kk < kBK / 16; ++kk) {
      const uint32_t accum = (kb | kk) != 0;
      const uint64_t dx = sdesc_at(xs, kk * 32);
      if (kTokenMajor) {
        umma_bf16(d, dx, sdesc_at(wst, kk * 32), idesc, accum);
      } else {
        umma_bf16(d, sdesc_at(wst, kk * 32), dx, idesc, accum);
        umma_bf16(d + 128, sdesc_at(wst, kWStageBytes + kk * 32), dx, idesc, accum);
      }
    }
    umma_commit(&empty_bar[stage]);
    if (++stage == kSingleStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
  return true;
}

// The K loop of a narrow weight-major tile: each stage holds two K blocks (the last one
// may hold one), each a 128-row W block (FC1: 64 gate rows, then the 64 up rows of the
// same channels) and the tile's X rows; one MMA per 16 K, A = the W block, B = X (N = ntok).
__device__ __forceinline__ bool single_k_loop_narrow(uint32_t d, uint32_t idesc, int nkb,
                                                     int& stage, uint32_t& phase, uint64_t dx0,
                                                     uint64_t dw0, uint64_t* full_bar,
                                                     uint64_t* empty_bar, volatile int* abort) {
  for (int kb = 0; kb < nkb; kb += 2) {
    if (!mbar_wait(&full_bar[stage], phase, abort)) return false;
    tc_fence_after();
    const uint64_t xs = sdesc_at(dx0, stage * kXStageBytes);
    const uint64_t wst = sdesc_at(dw0, stage * (2 * kWStageBytes));
    const int nk = nkb - kb < 2 ? 1 : 2;
    for (int b = 0; b < nk; ++b) {
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        umma_bf16(d, sdesc_at(wst, b * kWStageBytes + kk * 32),
                  sdesc_at(xs, b * (kXStageBytes / 2) + kk * 32), idesc, (kb | b | kk) != 0);
      }
    }
    umma_commit(&empty_bar[stage]);
    if (++stage == kSingleStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
  return true;
}

// Tensor maps of one GEMM for the single-SM kernel: addresses of the kernel's
// __grid_constant__ parameters.
struct SingleMaps {
  const CUtensorMap* x128;   // A rows, box 64 x 128
  const CUtensorMap* x16;    // A rows, box 64 x 16
  const CUtensorMap* x64;    // A rows, box 64 x 64
  const CUtensorMap* w;      // routed weights [planes, R, K], box 64 x 128
  const CUtensorMap* ws;     // shared weights [1, R, K]
  const CUtensorMap* w64;    // routed, box 64 x 64 (narrow launches only)
  const CUtensorMap* ws64;   // shared, box 64 x 64 (narrow launches only)
  const CUtensorMap* out;    // output rows, store box 32 x 32
};

// What a single-SM launch runs: one GEMM, or both (FC1's work list, then FC2's).
constexpr int kModeFc2 = 0;
constexpr int kModeFc1 = 1;
constexpr int kModeFused = 2;

// Producer of the single-SM kernel: the TMA loads of one tile, stage by stage. Returns
// false if a stage did not come free in time.
template <bool kFc1, bool kNarrow>
__device__ __forceinline__ bool single_produce(const Unit& t, const SingleMaps& m,
                                               const GemmArgs& a, int& stage, uint32_t& phase,
                                               int& issued, uint8_t* sX, uint8_t* sW,
                                               uint64_t* full_bar, uint64_t* empty_bar,
                                               volatile int* abort) {
  const bool shared = t.g >= a.E;
  const CUtensorMap* mw = shared ? m.ws : m.w;
  const int ecoord = shared ? 0 : t.g - a.plane_off;
  const int wr0 = t.n0;
  const int wr1 = kFc1 ? (t.N + t.n0) : (t.n0 + 128);
  const uint32_t xbytes = static_cast<uint32_t>(t.ntok) * kRowBytes;
  // A wide weight-major tile (a group's last partial tile) loads its X rows as at most two
  // 16-row boxes, else as one 64- or 128-row box per stage (rows past ntok land in the
  // stage; the MMA, N = ntok, never reads them; rows past the tensor are zero-filled).
  const int xbox = t.ntok <= 32 ? 16 : (t.ntok <= 64 ? 64 : 128);
  const uint32_t xwide = xbox == 16 ? xbytes : static_cast<uint32_t>(xbox) * kRowBytes;
  const uint32_t bytes = (2 * kWStageBytes) + (t.token_major ? kXStageBytes : xwide);
  const int nkb = t.K / kBK;
  // Narrow tiles: two K blocks per stage; FC1 W blocks are 64 gate rows (64-row boxes)
  // then the 64 up rows, FC2 W blocks 128 channel rows.
  const CUtensorMap* mwn = kFc1 ? (shared ? m.ws64 : m.w64) : mw;
  const int nst = kNarrow && t.narrow ? (nkb + 1) >> 1 : nkb;
  for (int j = 0; j < nst; ++j) {
    if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort)) return false;
    uint8_t* xs = sX + stage * kXStageBytes;
    uint8_t* ws = sW + stage * (2 * kWStageBytes);
    if (kNarrow && t.narrow) {
      const int nk = nkb - 2 * j < 2 ? 1 : 2;
      mbar_arrive_expect_tx(&full_bar[stage], nk * (kWStageBytes + xbytes));
      for (int b = 0; b < nk; ++b) {
        const int kc = (2 * j + b) * kBK;
        uint8_t* xb = xs + b * (kXStageBytes / 2);
        uint8_t* wb = ws + b * kWStageBytes;
        for (int r = 0; r < t.ntok; r += 16)
          tma_load_2d(xb + r * kRowBytes, m.x16, &full_bar[stage], kc, t.row0 + r);
        if (kFc1) {
          tma_load_3d(wb, mwn, &full_bar[stage], kc, t.n0, ecoord);
          tma_load_3d(wb + kWStageBytes / 2, mwn, &full_bar[stage], kc, t.N + t.n0, ecoord);
        } else {
          tma_load_3d(wb, mwn, &full_bar[stage], kc, t.n0, ecoord);
        }
      }
    } else {
      mbar_arrive_expect_tx(&full_bar[stage], bytes);
      const int kc = j * kBK;
      if (t.token_major || xbox == 128) {
        tma_load_2d(xs, m.x128, &full_bar[stage], kc, t.row0);
      } else if (xbox == 64) {
        tma_load_2d(xs, m.x64, &full_bar[stage], kc, t.row0);
      } else {
        for (int r = 0; r < t.ntok; r += 16)
          tma_load_2d(xs + r * kRowBytes, m.x16, &full_bar[stage], kc, t.row0 + r);
      }
      tma_load_3d(ws, mw, &full_bar[stage], kc, wr0, ecoord);
      tma_load_3d(ws + kWStageBytes, mw, &full_bar[stage], kc, wr1, ecoord);
    }
    ++issued;
    if (++stage == kSingleStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
  return true;
}

// Epilogue of one single-SM tile, by the four epilogue warps (q = TMEM lane quarter).
template <bool kFc1, bool kNarrow>
__device__ __forceinline__ void single_epilogue(uint32_t tb, const Unit& t, int q, int lane,
                                                uint8_t* my_out, int& sbuf, float* s_xchg,
                                                const SingleMaps& m, const GemmArgs& a) {
  const int lrow = q * 32 + lane;
  if (kNarrow && t.narrow) {
    // Lane = weight row of the narrow tile (FC1: gate lanes 0-63, up lanes 64-127).
    store_weight_major<kFc1>(tb, t, lrow, 0u, s_xchg, a);
  } else if (t.token_major) {
    // Thread = token row lrow; columns = channels (a full 128-row tile).
    store_token_major_tma<kFc1>(tb, t, q, lane, my_out, sbuf, m.out);
  } else {
    // Thread = channel lrow (of the 128 in D0, and of D1); columns = tokens.
    float va[16], vb[16];
    const int ch0 = t.n0 + lrow;
    const int ch1 = kFc1 ? ch0 : (t.n0 + 128 + lrow);
    const bool v0 = ch0 < t.N, v1 = ch1 < t.N;
#pragma unroll 1
    for (int c0 = 0; c0 < t.ntok; c0 += 16) {
      tmem_ld2_x16(tb + c0, tb + 128 + c0, va, vb);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = c0 + i;
        if (r < t.rows) {
          __nv_bfloat16* orow = a.out + static_cast<int64_t>(t.row0 + r) * a.out_ld;
          if (kFc1) {
            if (v0) orow[ch0] = __float2bfloat16_rn(silu(va[i]) * vb[i]);
          } else {
            if (v0) orow[ch0] = __float2bfloat16_rn(va[i]);
            if (v1) orow[ch1] = __float2bfloat16_rn(vb[i]);
          }
        }
      }
    }
  }
}

// The single-SM kernel. kNarrow: a launch whose small groups get narrow weight-major
// tiles (see narrow_max_rows); only that form reads the 64-row weight maps. kMode: FC1
// alone (m1, a1), FC2 alone (m2, a2; the callers pass the same maps and arguments twice),
// or both GEMMs in one persistent launch: the work list is FC1's tiles, then FC2's, claimed
// from one counter. A fused FC2 tile of group g first waits (bounded) until every FC1 tile
// of group g has stored its h rows: each FC1 tile's epilogue adds 1 to the group's
// completion counter (a1.dep[g]) once its stores are visible. Tiles are claimed in list
// order and every claimed FC1 tile completes without waiting on FC2 work, so the waits
// end; FC2 starts on SMs that FC1's last round leaves idle, with no second launch.
template <int kMode, bool kNarrow>
__device__ __forceinline__ void single_kernel_body(const SingleMaps& m1, const SingleMaps& m2,
                                                   const GemmArgs& a1, const GemmArgs& a2) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kSingleStages], empty_bar[kSingleStages];
  __shared__ float s_xchg[kNarrow ? 64 * kXchgStride : 1];
  __shared__ uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ uint64_t sched_full[kSchedDepth], sched_empty[kSchedDepth];
  __shared__ int s_tile[kSchedDepth];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int32_t s_off1[kMode == kModeFc2 ? 1 : kMaxGroups + 1];
  __shared__ int32_t s_off2[kMode == kModeFc1 ? 1 : kMaxGroups + 1];
  __shared__ int32_t s_cnt[kMaxGroups], s_start[kMaxGroups];
  __shared__ uint32_t s_dep_seen[kDepWords];
  constexpr bool kFused = kMode == kModeFused;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // 1024-byte aligned stage buffers (the 128-byte swizzle repeats every 1024 bytes).
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sX = smem;                                   // kSingleStages x 16 KB
  uint8_t* sW = smem + kSingleStages * kXStageBytes;          // kSingleStages x 256 W rows
  uint8_t* sOut = sW + kSingleStages * 2 * kWStageBytes;      // epilogue staging boxes

  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSingleStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tfull_bar[s], 1);
      mbar_init(&tempty_bar[s], 128);
    }
    mbar_init(&drain_bar, 1);
    for (int s = 0; s < kSchedDepth; ++s) {
      mbar_init(&sched_full[s], 1);
      mbar_init(&sched_empty[s], 1 + 4);   // the MMA thread + one arrival per epilogue warp
    }
    for (int i = 0; i < kDepWords; ++i) s_dep_seen[i] = 0;
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    if (kMode != kModeFc2) {
      tma_prefetch_map(m1.x128);
      tma_prefetch_map(m1.x16);
      tma_prefetch_map(m1.x64);
      tma_prefetch_map(m1.w);
      tma_prefetch_map(m1.ws);
      tma_prefetch_map(m1.out);
    }
    if (kMode != kModeFc1) {
      tma_prefetch_map(m2.x128);
      tma_prefetch_map(m2.x16);
      tma_prefetch_map(m2.x64);
      tma_prefetch_map(m2.w);
      tma_prefetch_map(m2.ws);
      tma_prefetch_map(m2.out);
    }
    if (kNarrow && kMode != kModeFc1) tma_prefetch_map(m2.w64);
    if (kNarrow && kMode != kModeFc2) {
      tma_prefetch_map(m1.w64);
      tma_prefetch_map(m1.ws64);
      // The kernels before this one (routing and the permutation) leave HBM idle. Pull
      // this CTA's likely first tiles into L2 meanwhile: the claims of round r are list
      // entries r * gridDim.x .. (r + 1) * gridDim.x - 1, and with every expert active
      // entry b is expert b / tiles-per-expert, narrow tile b mod tiles-per-expert. A
      // wrong guess (an inactive expert) only costs idle bandwidth.
      const int tpe = (a1.N_routed + kFc1NarrowCols - 1) / kFc1NarrowCols;
      const int nkb = a1.K_routed / kBK;
      int left = a1.prefetch_kb;
      for (int b = static_cast<int>(blockIdx.x); left > 0; b += static_cast<int>(gridDim.x)) {
        const int g = b / tpe;
        if (g >= a1.planes) break;
        const int n0 = (b - g * tpe) * kFc1NarrowCols;
        const int n = left < nkb ? left : nkb;
        for (int kb = 0; kb < n; ++kb) {
          tma_prefetch_3d(m1.w64, kb * kBK, n0, g);
          tma_prefetch_3d(m1.w64, kb * kBK, a1.N_routed + n0, g);
        }
        left -= n;
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // Everything above overlaps the previous kernel; the work lists are its output.
  pdl_wait();
  if (kMode != kModeFc2)
    for (int i = threadIdx.x; i <= a1.G; i += blockDim.x) s_off1[i] = a1.tile_off[i];
  if (kMode != kModeFc1)
    for (int i = threadIdx.x; i <= a2.G; i += blockDim.x) s_off2[i] = a2.tile_off[i];
  for (int i = threadIdx.x; i < a1.G; i += blockDim.x) {
    s_cnt[i] = a1.counts[i];
    s_start[i] = a1.starts[i];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  volatile int* abort = &s_abort;
  const int total1 = kMode == kModeFc2 ? 0 : s_off1[a1.G];
  const int total = total1 + (kMode == kModeFc1 ? 0 : s_off2[a2.G]);
  // A claimed index -> (GEMM, tile). In the single-GEMM modes the branch is a constant.
  auto is_fc1 = [&](int tile) { return kFused ? tile < total1 : kMode == kModeFc1; };
  auto decode = [&](int tile, bool fc1) {
    return fc1 ? decode_single(tile, s_off1, s_cnt, s_start, a1, true, kNarrow)
               : decode_single(kFused ? tile - total1 : tile, s_off2, s_cnt, s_start, a2, false,
                               kNarrow);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int slot = it & (kSchedDepth - 1);
        if (!mbar_wait(&sched_empty[slot], ((it / kSchedDepth) & 1) ^ 1u, abort)) {
          flag_timeout(a1.status, abort);
          ok = false;
          break;
        }
        int tile = atomicAdd(a1.sched, 1);
        if (tile >= total) tile = -1;
        s_tile[slot] = tile;
        mbar_arrive(&sched_full[slot]);
        if (tile < 0) break;
        const bool fc1 = is_fc1(tile);
        const Unit t = decode(tile, fc1);
        if (fc1) {
          ok = single_produce<true, kNarrow>(t, m1, a1, stage, phase, issued, sX, sW, full_bar,
                                             empty_bar, abort);
        } else {
          if (kFused) {
            // h rows of group g are complete once all its FC1 tiles have signalled.
            ok = wait_group_h(s_dep_seen, a1.dep, t.g, s_off1[t.g + 1] - s_off1[t.g], abort);
          }
          if (ok)
            ok = single_produce<false, kNarrow>(t, m2, a2, stage, phase, issued, sX, sW,
                                                full_bar, empty_bar, abort);
        }
        if (!ok) flag_timeout(a1.status, abort);
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA exits: wait (bounded)
        // on the full barrier of each of the last kSingleStages issues.
        int s = stage;
        uint32_t ph = phase;
        const int n = issued < kSingleStages ? issued : kSingleStages;
        for (int i = 0; i < n; ++i) {
          if (--s < 0) {
            s = kSingleStages - 1;
            ph ^= 1u;
          }
          volatile int never = 0;
          mbar_wait(&full_bar[s], ph, &never);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      const uint64_t dx0 = sdesc_k_major(smem_u32(sX), kRowBytes);
      const uint64_t dw0 = sdesc_k_major(smem_u32(sW), kRowBytes);
      for (int it = 0; ok; ++it) {
        const int slot = it & (kSchedDepth - 1);
        if (!mbar_wait(&sched_full[slot], (it / kSchedDepth) & 1, abort)) {
          flag_timeout(a1.status, abort);
          ok = false;
          break;
        }
        const int tile = *reinterpret_cast<volatile int*>(&s_tile[slot]);
        mbar_arrive(&sched_empty[slot]);
        if (tile < 0) break;
        const Unit t = decode(tile, is_fc1(tile));
        if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort)) {
          flag_timeout(a1.status, abort);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kAccCols);
        const int nkb = t.K / kBK;
        if (kNarrow && t.narrow)
          ok = single_k_loop_narrow(d, idesc_bf16_f32(128, t.ntok), nkb, stage, phase, dx0, dw0,
                                    full_bar, empty_bar, abort);
        else if (t.token_major)
          ok = single_k_loop<true>(d, idesc_bf16_f32(128, 256), nkb, stage, phase, dx0, dw0,
                                   full_bar, empty_bar, abort);
        else
          ok = single_k_loop<false>(d, idesc_bf16_f32(128, t.ntok), nkb, stage, phase, dx0, dw0,
                                    full_bar, empty_bar, abort);
        if (!ok) {
          flag_timeout(a1.status, abort);
          break;
        }
        umma_commit(&tfull_bar[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        // Wait (bounded) for every MMA issued so far before TMEM is released.
        umma_commit(&drain_bar);
        volatile int never = 0;
        mbar_wait(&drain_bar, 0, &never);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    uint8_t* my_out = sOut + q * 2 * kStoreBufBytes;
    int sbuf = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = 0;; ++it) {
      const int slot = it & (kSchedDepth - 1);
      const bool have = mbar_wait(&sched_full[slot], (it / kSchedDepth) & 1, abort);
      if (!__all_sync(0xffffffffu, have)) {
        flag_timeout(a1.status, abort);
        break;
      }
      const int tile = *reinterpret_cast<volatile int*>(&s_tile[slot]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sched_empty[slot]);
      if (tile < 0) break;
      const bool fc1 = is_fc1(tile);
      const Unit t = decode(tile, fc1);
      const bool got = mbar_wait(&tfull_bar[acc], acc_phase, abort);
      // Lanes may leave the poll at different times; tcgen05.ld is warp-collective.
      if (!__all_sync(0xffffffffu, got)) {
        flag_timeout(a1.status, abort);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * kAccCols) +
                          (static_cast<uint32_t>(q * 32) << 16);
      if (fc1) single_epilogue<true, kNarrow>(tb, t, q, lane, my_out, sbuf, s_xchg, m1, a1);
      else single_epilogue<false, kNarrow>(tb, t, q, lane, my_out, sbuf, s_xchg, m2, a2);
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
      if (kFused && fc1) {
        // Publish this tile's h rows to the FC2 tiles of its group: every store of the
        // four warps complete and visible (TMA stores: waited for, then a proxy fence),
        // then one release add on the group's counter.
        if (lane == 0) {
          bulk_wait_group<0>();
          fence_proxy_async_global();
        }
        __threadfence();
        named_barrier_sync(2, 128);
        if (q == 0 && lane == 0) red_release_gpu_add(a1.dep + t.g, 1);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // Every TMA store of this warp has written its box before the CTA ends.
    if (lane == 0) bulk_wait_group<0>();
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0) finish_claims(a1);
}

template <bool kFc1>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_x128, const __grid_constant__ CUtensorMap map_x16,
                    const __grid_constant__ CUtensorMap map_x64, const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_ws,
                    const __grid_constant__ CUtensorMap map_out, GemmArgs a) {
  const SingleMaps m{&map_x128, &map_x16, &map_x64, &map_w, &map_ws, nullptr, nullptr, &map_out};
  single_kernel_body<kFc1 ? kModeFc1 : kModeFc2, false>(m, m, a, a);
}

template <bool kFc1>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_narrow_kernel(const __grid_constant__ CUtensorMap map_x128,
                           const __grid_constant__ CUtensorMap map_x16,
                           const __grid_constant__ CUtensorMap map_x64,
                           const __grid_constant__ CUtensorMap map_w,
                           const __grid_constant__ CUtensorMap map_ws,
                           const __grid_constant__ CUtensorMap map_w64,
                           const __grid_constant__ CUtensorMap map_ws64,
                           const __grid_constant__ CUtensorMap map_out, GemmArgs a) {
  const SingleMaps m{&map_x128, &map_x16, &map_x64, &map_w, &map_ws, &map_w64, &map_ws64, &map_out};
  single_kernel_body<kFc1 ? kModeFc1 : kModeFc2, true>(m, m, a, a);
}

// Both GEMMs in one launch (FC1's tiles, then FC2's): maps and arguments of FC1 (x_perm,
// w13, h) then of FC2 (h, w2, out_perm).
template <bool kNarrow>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_fused_kernel(const __grid_constant__ CUtensorMap f1_x128,
                          const __grid_constant__ CUtensorMap f1_x16,
                          const __grid_constant__ CUtensorMap f1_x64,
                          const __grid_constant__ CUtensorMap f1_w,
                          const __grid_constant__ CUtensorMap f1_ws,
                          const __grid_constant__ CUtensorMap f1_w64,
                          const __grid_constant__ CUtensorMap f1_ws64,
                          const __grid_constant__ CUtensorMap f1_out,
                          const __grid_constant__ CUtensorMap f2_x128,
                          const __grid_constant__ CUtensorMap f2_x16,
                          const __grid_constant__ CUtensorMap f2_x64,
                          const __grid_constant__ CUtensorMap f2_w,
                          const __grid_constant__ CUtensorMap f2_ws,
                          const __grid_constant__ CUtensorMap f2_w64,
                          const __grid_constant__ CUtensorMap f2_ws64,
                          const __grid_constant__ CUtensorMap f2_out, GemmArgs a1, GemmArgs a2) {
  const SingleMaps m1{&f1_x128, &f1_x16, &f1_x64, &f1_w, &f1_ws, &f1_w64, &f1_ws64, &f1_out};
  const SingleMaps m2{&f2_x128, &f2_x16, &f2_x64, &f2_w, &f2_ws, &f2_w64, &f2_ws64, &f2_out};
  single_kernel_body<kModeFused, kNarrow>(m1, m2, a1, a2);
}

// ============================================================== CTA-pair kernel

// The K loop of one unit, issued by the first CTA's MMA thread: token-major units
// multiply X rows (A, M = 256 over the pair) by W rows (B, N = 256); weight-major units
// swap the operands (A = W rows, B = the unit's X rows, N = ntok). A separate loop per
// form keeps the operand order and the instruction descriptor fixed inside the loop; a
// per-instruction choice between the two forms cost a quarter of the tensor throughput.
// Returns false if a stage did not arrive in time.
template <bool kTokenMajor>
__device__ __forceinline__ bool pair_k_loop(uint32_t d, uint32_t idesc, int nkb, int& stage,
                                            uint32_t& phase, uint64_t dx0, uint64_t dw0,
                                            uint64_t* full_bar, uint64_t* empty_bar,
                                            volatile int* abort) {
  for (int kb = 0; kb < nkb; kb += kPairBlocksPerStage) {
    if (!mbar_wait<true>(&full_bar[stage], phase, abort)) return false;
    tc_fence_after();
    const int slot0 = stage * kPairBlocksPerStage;
    const uint64_t xs = sdesc_at(dx0, slot0 * kXStageBytes);
    const uint64_t wst = sdesc_at(dw0, slot0 * kWStageBytes);
#pragma unroll
    for (int b = 0; b < kPairBlocksPerStage; ++b) {
      if (b > 0 && kb + b >= nkb) break;   // an odd block count: the last stage holds one
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint64_t dx = sdesc_at(xs, b * kXStageBytes + kk * 32);
        const uint64_t dw = sdesc_at(wst, b * kWStageBytes + kk * 32);
        if (kTokenMajor) umma_bf16_pair(d, dx, dw, idesc, (kb | b | kk) != 0);
        else umma_bf16_pair(d, dw, dx, idesc, (kb | b | kk) != 0);
      }
    }
    // The stage is free in both CTAs once these MMAs have read it.
    umma_commit_pair(&empty_bar[stage], kPairMask);
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
  return true;
}

// Tensor maps of one GEMM for the pair kernel: addresses of the kernel's __grid_constant__
// parameters.
struct PairMaps {
  const CUtensorMap* x128;   // A rows, box 64 x 128
  const CUtensorMap* x64;    // A rows, box 64 x 64
  const CUtensorMap* w128;   // routed weights, box 64 x 128
  const CUtensorMap* ws128;  // shared weights, box 64 x 128
  const CUtensorMap* w64;    // routed weights, box 64 x 64
  const CUtensorMap* ws64;   // shared weights, box 64 x 64
  const CUtensorMap* out;    // output rows, store box 32 x 32
};

// Producer of one CTA of the pair: the TMA loads of one unit, K block by K block. The
// first CTA also claims the pair's next unit kClaimLead K blocks before the end (from
// *sched, into claimed / have_claim). Returns false if a stage did not come free in time.
template <bool kFc1>
__device__ __forceinline__ bool pair_produce(const Unit& t, const PairMaps& m, const GemmArgs& a,
                                             uint32_t rank, bool lead, int32_t* sched,
                                             int& claimed, bool& have_claim, int& fills,
                                             uint8_t* sX, uint8_t* sW, uint32_t lead_full,
                                             uint64_t* full_bar, uint64_t* empty_bar,
                                             volatile int* abort) {
  const bool shared = t.g >= a.E;
  const CUtensorMap* mw128 = shared ? m.ws128 : m.w128;
  const CUtensorMap* mw64 = shared ? m.ws64 : m.w64;
  const int ecoord = shared ? 0 : t.g - a.plane_off;
  const int r = static_cast<int>(rank);
  // This CTA's token rows and its share of the weight rows.
  const int half = t.ntok >> 1;
  const int xrow = t.token_major ? t.row0 : t.row0 + r * half;
  // Weight-major units have at most 128 token rows: each CTA loads its <= 64 rows as one
  // 64-row box (rows past its share land in the stage but the MMA, N = ntok, never reads
  // them; rows past the tensor are zero-filled).
  const uint32_t xbytes = t.token_major ? kXStageBytes : 64u * kRowBytes;
  const uint32_t tx_bytes = 2u * (xbytes + kWStageBytes);
  const int nkb = t.K / kBK;
  const int claim_kb = nkb > kClaimLead ? nkb - kClaimLead : 0;
  for (int kb = 0; kb < nkb; kb += kPairBlocksPerStage) {
    const int nk = nkb - kb < kPairBlocksPerStage ? nkb - kb : kPairBlocksPerStage;
    if (lead && claim_kb >= kb && claim_kb < kb + nk) {
      claimed = atomicAdd(sched, 1);
      have_claim = true;
    }
    const int stage = fills % kStages;
    if (!mbar_wait<true>(&empty_bar[stage], ((fills / kStages) & 1) ^ 1u, abort)) return false;
    if (lead) mbar_arrive_expect_tx(&full_bar[stage], static_cast<uint32_t>(nk) * tx_bytes);
    const uint32_t fb = lead_full + 8u * stage;
    for (int b = 0; b < nk; ++b) {
      const int slot = stage * kPairBlocksPerStage + b;
      const int kc = (kb + b) * kBK;
      uint8_t* xs = sX + slot * kXStageBytes;
      uint8_t* wsm = sW + slot * kWStageBytes;
      if (t.token_major) {
        tma_load_2d_pair(xs, m.x128, fb, kc, xrow);
        const int wrow = kFc1 ? (lead ? t.n0 : t.N + t.n0) : (t.n0 + 128 * r);
        tma_load_3d_pair(wsm, mw128, fb, kc, wrow, ecoord);
      } else {
        tma_load_2d_pair(xs, m.x64, fb, kc, xrow);
        if (kFc1) {
          tma_load_3d_pair(wsm, mw64, fb, kc, t.n0 + 64 * r, ecoord);
          tma_load_3d_pair(wsm + 64 * kRowBytes, mw64, fb, kc, t.N + t.n0 + 64 * r, ecoord);
        } else {
          tma_load_3d_pair(wsm, mw128, fb, kc, t.n0 + 128 * r, ecoord);
        }
      }
    }
    ++fills;
  }
  return true;
}

// Epilogue of one pair unit in one CTA, by its four epilogue warps.
template <bool kFc1>
__device__ __forceinline__ void pair_epilogue(uint32_t tb, const Unit& t, int q, int lane,
                                              uint32_t rank, uint8_t* my_out, int& sbuf,
                                              float* s_xchg, const PairMaps& m,
                                              const GemmArgs& a) {
  const int lrow = q * 32 + lane;
  if (t.token_major && t.rows == kTileRows)
    store_token_major_tma<kFc1>(tb, t, q, lane, my_out, sbuf, m.out);
  else if (t.token_major)
    store_token_major<kFc1>(tb, t, lrow, a);
  else
    store_weight_major<kFc1>(tb, t, lrow, rank, s_xchg, a);
}

// The CTA-pair kernel body. kMode as in the single-SM kernel: FC1 alone (m1, a1), FC2
// alone (m2, a2; the callers pass the same maps and arguments twice), or both GEMMs in
// one launch, FC1's units then FC2's from one counter. In the fused form an FC2 unit of
// group g waits (bounded) until both CTAs of every FC1 unit of group g have signalled
// that their h rows are stored and visible; claims go in list order and FC1 units never
// wait, so every wait ends.
template <int kMode>
__device__ __forceinline__ void pair_kernel_body(const PairMaps& m1, const PairMaps& m2,
                                                 const GemmArgs& a1, const GemmArgs& a2) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages];
  __shared__ uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ uint64_t sched_full[kSchedDepth], sched_empty[kSchedDepth];
  __shared__ int s_tile[kSchedDepth];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int32_t s_off1[kMode == kModeFc2 ? 1 : kMaxGroups + 1];
  __shared__ int32_t s_off2[kMode == kModeFc1 ? 1 : kMaxGroups + 1];
  __shared__ int32_t s_cnt[kMaxGroups], s_start[kMaxGroups];
  __shared__ float s_xchg[64 * kXchgStride];
  __shared__ uint32_t s_dep_seen[kDepWords];
  constexpr bool kFused = kMode == kModeFused;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const bool lead = rank == 0;

  // 1024-byte aligned stage buffers (the 128-byte swizzle repeats every 1024 bytes), at
  // the same offsets in both CTAs: the pair MMA reads the second CTA's operands at the
  // first CTA's shared-memory addresses.
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sX = smem;                                   // kPairSlots x up to 128 X rows
  uint8_t* sW = smem + kPairSlots * kXStageBytes;       // kPairSlots x 128 W rows
  uint8_t* sOut = sW + kPairSlots * kWStageBytes;       // epilogue staging boxes

  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);    // first CTA: its producer's arrival + both CTAs' bytes
      mbar_init(&empty_bar[s], 1);   // the first CTA's pair commit, delivered to both CTAs
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&tfull_bar[s], 1);
      mbar_init(&tempty_bar[s], 8);  // first CTA: one arrival per epilogue warp of both CTAs
    }
    mbar_init(&drain_bar, 1);
    for (int s = 0; s < kSchedDepth; ++s) {
      mbar_init(&sched_full[s], 1);
      mbar_init(&sched_empty[s], kSchedConsumers);   // used in the first CTA only
    }
    for (int i = 0; i < kDepWords; ++i) s_dep_seen[i] = 0;
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    const PairMaps* ms[2] = {&m1, &m2};
    for (int i = (kMode == kModeFc2 ? 1 : 0); i < (kMode == kModeFc1 ? 1 : 2); ++i) {
      tma_prefetch_map(ms[i]->x128);
      tma_prefetch_map(ms[i]->x64);
      tma_prefetch_map(ms[i]->w128);
      tma_prefetch_map(ms[i]->ws128);
      tma_prefetch_map(ms[i]->w64);
      tma_prefetch_map(ms[i]->ws64);
      tma_prefetch_map(ms[i]->out);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(&s_tmem_base, kTmemCols);   // collective with the other CTA's warp 1
    tmem_relinquish_pair();
  }
  // Everything above overlaps the previous kernel; the work lists are its output.
  pdl_wait();
  if (kMode != kModeFc2)
    for (int i = threadIdx.x; i <= a1.G; i += blockDim.x) s_off1[i] = a1.tile_off[i];
  if (kMode != kModeFc1)
    for (int i = threadIdx.x; i <= a2.G; i += blockDim.x) s_off2[i] = a2.tile_off[i];
  for (int i = threadIdx.x; i < a1.G; i += blockDim.x) {
    s_cnt[i] = a1.counts[i];
    s_start[i] = a1.starts[i];
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers exist before any remote arrival or copy
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  volatile int* abort = &s_abort;
  const int total1 = kMode == kModeFc2 ? 0 : s_off1[a1.G];
  const int total = total1 + (kMode == kModeFc1 ? 0 : s_off2[a2.G]);
  // A claimed index -> (GEMM, unit). In the single-GEMM modes the branch is a constant.
  auto is_fc1 = [&](int unit) { return kFused ? unit < total1 : kMode == kModeFc1; };
  auto decode = [&](int unit, bool fc1, uint32_t r) {
    return fc1 ? decode_unit(unit, s_off1, s_cnt, s_start, a1, true, r)
               : decode_unit(kFused ? unit - total1 : unit, s_off2, s_cnt, s_start, a2, false, r);
  };

  const uint32_t lead_full = mapa_shared(smem_u32(&full_bar[0]), 0);
  const uint32_t lead_tempty = mapa_shared(smem_u32(&tempty_bar[0]), 0);
  const uint32_t lead_sched_empty = mapa_shared(smem_u32(&sched_empty[0]), 0);
  const uint32_t peer_s_tile = mapa_shared(smem_u32(&s_tile[0]), peer);
  const uint32_t peer_sched_full = mapa_shared(smem_u32(&sched_full[0]), peer);
  auto release_slot = [&](int slot) {
    if (lead) mbar_arrive(&sched_empty[slot]);
    else mbar_arrive_cluster(lead_sched_empty + 8u * slot);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int fills = 0;
      bool ok = true;
      // The first CTA claims each next unit kClaimLead K blocks before it has issued the
      // current unit's loads, so the atomic's latency is hidden; a whole unit ahead would
      // lengthen the tail.
      int claimed = 0;
      bool have_claim = false;
      for (int it = 0; ok; ++it) {
        const int slot = it & (kSchedDepth - 1);
        const uint32_t sph = (it / kSchedDepth) & 1;
        int unit;
        if (lead) {
          if (!mbar_wait<true>(&sched_empty[slot], sph ^ 1u, abort)) {
            flag_timeout(a1.status, abort);
            ok = false;
            break;
          }
          unit = have_claim ? claimed : atomicAdd(a1.sched, 1);
          have_claim = false;
          if (unit >= total) unit = -1;
          s_tile[slot] = unit;
          st_shared_cluster_u32(peer_s_tile + 4u * slot, static_cast<uint32_t>(unit));
          mbar_arrive(&sched_full[slot]);
          mbar_arrive_cluster(peer_sched_full + 8u * slot);
        } else {
          if (!mbar_wait<true>(&sched_full[slot], sph, abort)) {
            flag_timeout(a1.status, abort);
            ok = false;
            break;
          }
          unit = *reinterpret_cast<volatile int*>(&s_tile[slot]);
          release_slot(slot);
        }
        if (unit < 0) break;
        const bool fc1 = is_fc1(unit);
        const Unit t = decode(unit, fc1, rank);
        if (fc1) {
          ok = pair_produce<true>(t, m1, a1, rank, lead, a1.sched, claimed, have_claim, fills,
                                  sX, sW, lead_full, full_bar, empty_bar, abort);
        } else {
          if (kFused) {
            // Both CTAs of every FC1 unit of group g signal once their h rows are stored.
            ok = wait_group_h(s_dep_seen, a1.dep, t.g, 2 * (s_off1[t.g + 1] - s_off1[t.g]),
                              abort);
          }
          if (ok)
            ok = pair_produce<false>(t, m2, a2, rank, lead, a1.sched, claimed, have_claim,
                                     fills, sX, sW, lead_full, full_bar, empty_bar, abort);
        }
        if (!ok) flag_timeout(a1.status, abort);
      }
      // Before this CTA may exit, the first CTA's commits for every stage it filled must
      // have arrived (they target this CTA's barriers); bounded.
      volatile int never = 0;
      const int first = fills > kStages ? fills - kStages : 0;
      for (int f = first; f < fills; ++f)
        mbar_wait<true>(&empty_bar[f % kStages], (f / kStages) & 1, &never);
    }
  } else if (warp == 1) {
    if (lane == 0 && lead) {
      // ------------------------------------------------------------ MMA issuer (first CTA)
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      const uint64_t dx0 = sdesc_k_major(smem_u32(sX), kRowBytes);
      const uint64_t dw0 = sdesc_k_major(smem_u32(sW), kRowBytes);
      for (int it = 0; ok; ++it) {
        const int slot = it & (kSchedDepth - 1);
        if (!mbar_wait<true>(&sched_full[slot], (it / kSchedDepth) & 1, abort)) {
          flag_timeout(a1.status, abort);
          ok = false;
          break;
        }
        const int unit = *reinterpret_cast<volatile int*>(&s_tile[slot]);
        release_slot(slot);
        if (unit < 0) break;
        const Unit t = decode(unit, is_fc1(unit), 0u);
        if (!mbar_wait<true>(&tempty_bar[acc], acc_phase ^ 1u, abort)) {
          flag_timeout(a1.status, abort);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kAccCols);
        const int nkb = t.K / kBK;
        ok = t.token_major
                 ? pair_k_loop<true>(d, idesc_bf16_f32(256, 256), nkb, stage, phase, dx0, dw0,
                                     full_bar, empty_bar, abort)
                 : pair_k_loop<false>(d, idesc_bf16_f32(256, t.ntok), nkb, stage, phase, dx0,
                                      dw0, full_bar, empty_bar, abort);
        if (!ok) {
          flag_timeout(a1.status, abort);
          break;
        }
        umma_commit_pair(&tfull_bar[acc], kPairMask);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        // Wait (bounded) for every MMA issued so far before TMEM is released.
        umma_commit_pair(&drain_bar, 0x1);
        volatile int never = 0;
        mbar_wait(&drain_bar, 0, &never);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue (both CTAs)
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    uint8_t* my_out = sOut + q * 2 * kStoreBufBytes;
    int sbuf = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = 0;; ++it) {
      const int slot = it & (kSchedDepth - 1);
      const bool have = mbar_wait<true>(&sched_full[slot], (it / kSchedDepth) & 1, abort);
      if (!__all_sync(0xffffffffu, have)) {
        flag_timeout(a1.status, abort);
        break;
      }
      const int unit = *reinterpret_cast<volatile int*>(&s_tile[slot]);
      __syncwarp();
      if (lane == 0) release_slot(slot);
      if (unit < 0) break;
      const bool fc1 = is_fc1(unit);
      const Unit t = decode(unit, fc1, rank);
      const bool got = mbar_wait<true>(&tfull_bar[acc], acc_phase, abort);
      // Lanes may leave the poll at different times; tcgen05.ld is warp-collective.
      if (!__all_sync(0xffffffffu, got)) {
        flag_timeout(a1.status, abort);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * kAccCols) +
                          (static_cast<uint32_t>(q * 32) << 16);
      if (fc1) pair_epilogue<true>(tb, t, q, lane, rank, my_out, sbuf, s_xchg, m1, a1);
      else pair_epilogue<false>(tb, t, q, lane, rank, my_out, sbuf, s_xchg, m2, a2);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (lead) mbar_arrive(&tempty_bar[acc]);
        else mbar_arrive_cluster(lead_tempty + 8u * acc);
      }
      if (kFused && fc1) {
        // Publish this CTA's h rows of the unit to the FC2 units of its group: every
        // store of the four warps complete and visible (TMA stores: waited for, then a
        // proxy fence), then one release add on the group's counter.
        if (lane == 0) {
          bulk_wait_group<0>();
          fence_proxy_async_global();
        }
        __threadfence();
        named_barrier_sync(2, 128);
        if (q == 0 && lane == 0) red_release_gpu_add(a1.dep + t.g, 1);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // Every TMA store of this warp has written its box before the CTA ends.
    if (lane == 0) bulk_wait_group<0>();
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);   // collective with the other CTA's warp 1
  }
  // No CTA leaves while the other may still write into it or arrive on its barriers.
  cluster_sync();
  if (threadIdx.x == 0) finish_claims(a1);
}

template <bool kFc1>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_x128,
                         const __grid_constant__ CUtensorMap map_x64,
                         const __grid_constant__ CUtensorMap map_w128,
                         const __grid_constant__ CUtensorMap map_ws128,
                         const __grid_constant__ CUtensorMap map_w64,
                         const __grid_constant__ CUtensorMap map_ws64,
                         const __grid_constant__ CUtensorMap map_out, GemmArgs a) {
  const PairMaps m{&map_x128, &map_x64, &map_w128, &map_ws128, &map_w64, &map_ws64, &map_out};
  pair_kernel_body<kFc1 ? kModeFc1 : kModeFc2>(m, m, a, a);
}

// Both GEMMs in one launch (FC1's units, then FC2's): maps and arguments of FC1 (x_perm,
// w13, h) then of FC2 (h, w2, out_perm).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
grouped_gemm_pair_fused_kernel(const __grid_constant__ CUtensorMap f1_x128,
                               const __grid_constant__ CUtensorMap f1_x64,
                               const __grid_constant__ CUtensorMap f1_w128,
                               const __grid_constant__ CUtensorMap f1_ws128,
                               const __grid_constant__ CUtensorMap f1_w64,
                               const __grid_constant__ CUtensorMap f1_ws64,
                               const __grid_constant__ CUtensorMap f1_out,
                               const __grid_constant__ CUtensorMap f2_x128,
                               const __grid_constant__ CUtensorMap f2_x64,
                               const __grid_constant__ CUtensorMap f2_w128,
                               const __grid_constant__ CUtensorMap f2_ws128,
                               const __grid_constant__ CUtensorMap f2_w64,
                               const __grid_constant__ CUtensorMap f2_ws64,
                               const __grid_constant__ CUtensorMap f2_out, GemmArgs a1,
                               GemmArgs a2) {
  const PairMaps m1{&f1_x128, &f1_x64, &f1_w128, &f1_ws128, &f1_w64, &f1_ws64, &f1_out};
  const PairMaps m2{&f2_x128, &f2_x64, &f2_w128, &f2_ws128, &f2_w64, &f2_ws64, &f2_out};
  pair_kernel_body<kModeFused>(m1, m2, a1, a2);
}

// ---------------------------------------------------------------- host side


// Per device: the large dynamic shared memory opt-in of the kernels, and how many 2-CTA
// clusters of the pair kernel can be resident at once. The count is published (release)
// only after the attributes are set, so a thread that reads it (acquire) may launch; two
// threads that both find it unset both do the same idempotent work.
template <bool kFc1>
moe_status prepare_kernels(int* max_clusters) {
  static std::atomic<int> clusters_dev[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return set_error(MOE_ERR_CUDA, "cudaGetDevice failed");
  int have = clusters_dev[dev].load(std::memory_order_acquire);
  if (!have) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<kFc1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSingleSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(grouped_gemm_narrow_kernel<kFc1>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSingleSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(grouped_gemm_pair_kernel<kFc1>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess && kFc1)
      e = cudaFuncSetAttribute(grouped_gemm_pair_fused_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess && kFc1)
      e = cudaFuncSetAttribute(grouped_gemm_fused_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSingleSmemBytes);
    if (e == cudaSuccess && kFc1)
      e = cudaFuncSetAttribute(grouped_gemm_fused_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSingleSmemBytes);
    if (e != cudaSuccess)
      return set_error(MOE_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    const int sms = device_sm_count();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<kFc1>, &cfg) != cudaSuccess ||
        n < 1) {
      cudaGetLastError();   // clear the failed query; fall back to one cluster per SM pair
      n = sms / 2;
    }
    clusters_dev[dev].store(n, std::memory_order_release);
    have = n;
  }
  *max_clusters = have;
  return MOE_OK;
}

// The tensor maps, arguments and work bounds of one GEMM.
struct GemmSetup {
  CUtensorMap mx128, mx64, mx16, mw128, mws128, mw64, mws64, mout;
  GemmArgs pair, single;        // arguments of the pair and single-SM launches
  int64_t pair_bound, single_bound;
  bool narrow;
  int max_clusters;
};

template <bool kFc1>
moe_status setup_gemm(const moe_problem& p, const moe_ws_layout& L, const void* w,
                      const void* w_s, int e_lo, int e_hi, char* ws, GemmSetup* g) {
  g->max_clusters = 1;
  moe_status st = prepare_kernels<kFc1>(&g->max_clusters);
  if (st != MOE_OK) return st;
  const int64_t R = L.rows;
  const int has_shared = p.shared_I > 0;
  const void* A = kFc1 ? static_cast<const void*>(ws + L.x_perm) : static_cast<const void*>(ws + L.h);
  const uint64_t a_cols = kFc1 ? static_cast<uint64_t>(p.H) : static_cast<uint64_t>(L.h_ld);
  bool ok = encode_map2(&g->mx128, A, R, a_cols, 128) && encode_map2(&g->mx64, A, R, a_cols, 64) &&
            encode_map2(&g->mx16, A, R, a_cols, 16);
  // Weights [planes, rows, K]: FC1 w13 [E, 2I, H] (shared [1, 2Is, H]); FC2 w2 [E, H, I]
  // (shared [1, H, Is]).
  const uint64_t wr = kFc1 ? 2ull * p.I : static_cast<uint64_t>(p.H);
  const uint64_t wk = kFc1 ? static_cast<uint64_t>(p.H) : static_cast<uint64_t>(p.I);
  const uint64_t sr = kFc1 ? 2ull * p.shared_I : static_cast<uint64_t>(p.H);
  const uint64_t sk = kFc1 ? static_cast<uint64_t>(p.H) : static_cast<uint64_t>(p.shared_I);
  // Routed weights hold the experts [e_lo, e_hi) of this call only.
  const uint64_t planes = static_cast<uint64_t>(e_hi - e_lo);
  ok = ok && encode_map3(&g->mw128, w, planes, wr, wk, 128) &&
       encode_map3(&g->mw64, w, planes, wr, wk, 64);
  if (has_shared)
    ok = ok && encode_map3(&g->mws128, w_s, 1, sr, sk, 128) &&
         encode_map3(&g->mws64, w_s, 1, sr, sk, 64);
  else
    ok = ok && encode_map3(&g->mws128, w, planes, wr, wk, 128) &&
         encode_map3(&g->mws64, w, planes, wr, wk, 64);
  // Output rows: FC1 h [R, h_ld], FC2 out_perm [R, H].
  const uint64_t out_cols = kFc1 ? static_cast<uint64_t>(L.h_ld) : static_cast<uint64_t>(p.H);
  ok = ok && encode_store_map2(&g->mout, ws + (kFc1 ? L.h : L.out_perm), R, out_cols);
  if (!ok) return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed");

  GemmArgs a;
  a.counts = reinterpret_cast<const int32_t*>(ws + L.counts);
  a.starts = reinterpret_cast<const int32_t*>(ws + L.starts);
  a.G = L.groups;
  a.E = p.E;
  a.plane_off = e_lo;
  if (kFc1) {
    a.K_routed = p.H;
    a.K_shared = p.H;
    a.N_routed = p.I;
    a.N_shared = has_shared ? p.shared_I : p.I;
    a.out = reinterpret_cast<__nv_bfloat16*>(ws + L.h);
    a.out_ld = L.h_ld;
  } else {
    a.K_routed = p.I;
    a.K_shared = has_shared ? p.shared_I : p.I;
    a.N_routed = p.H;
    a.N_shared = p.H;
    a.out = reinterpret_cast<__nv_bfloat16*>(ws + L.out_perm);
    a.out_ld = p.H;
  }
  a.status = reinterpret_cast<int32_t*>(ws + L.status);
  a.dep = nullptr;
  a.planes = e_hi - e_lo;
  a.prefetch_kb = 0;
  // Work lists [pair units | single-SM tiles], each G+1 offsets; counters [pair | single].
  const int32_t* lists = reinterpret_cast<const int32_t*>(ws + (kFc1 ? L.tile_off1 : L.tile_off2));
  int32_t* sched = reinterpret_cast<int32_t*>(ws + L.sched) + (kFc1 ? 0 : 4);
  g->pair = a;
  g->pair.tile_off = lists;
  g->pair.sched = sched;
  g->single = a;
  g->single.tile_off = lists + (L.groups + 1);
  g->single.sched = sched + 2;

  // One of the two kernels takes every group (see pair_min_rows). Upper bounds on its
  // work per channel tile: pair units at most R/256 + G, single-SM tiles at most
  // R/128 + G.
  const int nI = has_shared && p.shared_I > p.I ? p.shared_I : p.I;
  const int64_t n_nt = kFc1 ? (nI + kFc1Cols - 1) / kFc1Cols : (p.H + kFc2Cols - 1) / kFc2Cols;
  const bool use_pairs = pair_min_rows(p) <= 2 * kTileRows;
  g->pair_bound = use_pairs ? (R / 256 + L.groups) * n_nt : 0;
  // (A narrow tile is half a channel tile wide: at most twice as many tiles.)
  g->narrow = narrow_max_rows(p) > 0;
  g->single_bound = use_pairs ? 0 : (g->narrow ? 2 : 1) * (R / kTileRows + L.groups) * n_nt;
  return MOE_OK;
}

// Narrow FC1: L2 prefetch of each CTA's guessed first tiles (see the kernel),
// kPrefetchBytes over the grid: two 64-row boxes (16 KB) per K block.
int32_t narrow_prefetch_kb(int64_t grid) {
  const int64_t per_kb = 2 * 64 * kRowBytes;
  const int64_t kb = kPrefetchBytes / (grid * per_kb);
  return static_cast<int32_t>(kb < (1 << 20) ? kb : (1 << 20));
}

template <bool kFc1>
moe_status launch_gemm(const moe_problem& p, const moe_ws_layout& L, const void* w,
                       const void* w_s, int e_lo, int e_hi, char* ws, cudaStream_t s) {
  GemmSetup g;
  moe_status st = setup_gemm<kFc1>(p, L, w, w_s, e_lo, e_hi, ws, &g);
  if (st != MOE_OK) return st;
  cudaError_t err = cudaSuccess;
  if (g.single_bound > 0) {
    GemmArgs as = g.single;
    int64_t grid = device_sm_count();
    if (grid > g.single_bound) grid = g.single_bound;
    if (grid < 1) grid = 1;
    if (kFc1 && g.narrow) as.prefetch_kb = narrow_prefetch_kb(grid);
    if (g.narrow)
      err = launch_pdl(grouped_gemm_narrow_kernel<kFc1>, dim3(static_cast<unsigned>(grid)),
                       dim3(kThreads), kSingleSmemBytes, s, g.mx128, g.mx16, g.mx64, g.mw128,
                       g.mws128, g.mw64, g.mws64, g.mout, as);
    else
      err = launch_pdl(grouped_gemm_kernel<kFc1>, dim3(static_cast<unsigned>(grid)), dim3(kThreads),
                       kSingleSmemBytes, s, g.mx128, g.mx16, g.mx64, g.mw128, g.mws128, g.mout, as);
  }
  if (err == cudaSuccess && g.pair_bound > 0) {
    int64_t clusters = g.max_clusters;
    if (clusters > g.pair_bound) clusters = g.pair_bound;
    err = launch_pdl(grouped_gemm_pair_kernel<kFc1>, dim3(static_cast<unsigned>(2 * clusters)),
                     dim3(kThreads), kSmemBytes, s, g.mx128, g.mx64, g.mw128, g.mws128, g.mw64,
                     g.mws64, g.mout, g.pair);
  }
  if (err != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "grouped_gemm launch: %s", cudaGetErrorString(err));
  return MOE_OK;
}

}  // namespace

moe_status launch_fc1(const moe_problem& p, const moe_ws_layout& L, const void* w13,
                      const void* w13_s, int e_lo, int e_hi, char* ws, cudaStream_t s) {
  return launch_gemm<true>(p, L, w13, w13_s, e_lo, e_hi, ws, s);
}

moe_status launch_fc2(const moe_problem& p, const moe_ws_layout& L, const void* w2,
                      const void* w2_s, int e_lo, int e_hi, char* ws, cudaStream_t s) {
  return launch_gemm<false>(p, L, w2, w2_s, e_lo, e_hi, ws, s);
}

moe_status launch_fc12(const moe_problem& p, const moe_ws_layout& L, const void* w13,
                       const void* w13_s, const void* w2, const void* w2_s, int e_lo, int e_hi,
                       char* ws, cudaStream_t s) {
  GemmSetup g1, g2;
  moe_status st = setup_gemm<true>(p, L, w13, w13_s, e_lo, e_hi, ws, &g1);
  if (st == MOE_OK) st = setup_gemm<false>(p, L, w2, w2_s, e_lo, e_hi, ws, &g2);
  if (st != MOE_OK) return st;
  if (g1.pair_bound > 0 && g2.pair_bound > 0) {
    // CTA-pair sizes: one launch of the pair kernel for both GEMMs, as below.
    GemmArgs a1 = g1.pair, a2 = g2.pair;
    a1.dep = reinterpret_cast<int32_t*>(ws + L.sched) + kSchedCounters;
    a2.dep = a1.dep;
    a2.sched = a1.sched;
    int64_t clusters = g1.max_clusters;
    if (clusters > g1.pair_bound + g2.pair_bound) clusters = g1.pair_bound + g2.pair_bound;
    const cudaError_t err = launch_pdl(
        grouped_gemm_pair_fused_kernel, dim3(static_cast<unsigned>(2 * clusters)), dim3(kThreads),
        kSmemBytes, s, g1.mx128, g1.mx64, g1.mw128, g1.mws128, g1.mw64, g1.mws64, g1.mout, g2.mx128,
        g2.mx64, g2.mw128, g2.mws128, g2.mw64, g2.mws64, g2.mout, a1, a2);
    if (err != cudaSuccess)
      return set_error(MOE_ERR_CUDA, "grouped_gemm launch: %s", cudaGetErrorString(err));
    return MOE_OK;
  }
  if (g1.single_bound == 0 || g2.single_bound == 0)
    return set_error(MOE_ERR_CUDA, "grouped_gemm: inconsistent launch bounds");
  // One persistent single-SM launch for both GEMMs: FC1's counter serves the joint list
  // and the per-group completion counters follow the work counters.
  GemmArgs a1 = g1.single, a2 = g2.single;
  a1.dep = reinterpret_cast<int32_t*>(ws + L.sched) + kSchedCounters;
  a2.dep = a1.dep;
  a2.sched = a1.sched;
  int64_t grid = device_sm_count();
  if (grid > g1.single_bound + g2.single_bound) grid = g1.single_bound + g2.single_bound;
  if (grid < 1) grid = 1;
  if (g1.narrow) a1.prefetch_kb = narrow_prefetch_kb(grid);
  cudaError_t err;
  if (g1.narrow)
    err = launch_pdl(grouped_gemm_fused_kernel<true>, dim3(static_cast<unsigned>(grid)),
                     dim3(kThreads), kSingleSmemBytes, s, g1.mx128, g1.mx16, g1.mx64, g1.mw128,
                     g1.mws128, g1.mw64, g1.mws64, g1.mout, g2.mx128, g2.mx16, g2.mx64, g2.mw128,
                     g2.mws128, g2.mw64, g2.mws64, g2.mout, a1, a2);
  else
    err = launch_pdl(grouped_gemm_fused_kernel<false>, dim3(static_cast<unsigned>(grid)),
                     dim3(kThreads), kSingleSmemBytes, s, g1.mx128, g1.mx16, g1.mx64, g1.mw128,
                     g1.mws128, g1.mw64, g1.mws64, g1.mout, g2.mx128, g2.mx16, g2.mx64, g2.mw128,
                     g2.mws128, g2.mw64, g2.mws64, g2.mout, a1, a2);
  if (err != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "grouped_gemm launch: %s", cudaGetErrorString(err));
  return MOE_OK;
}

}  // namespace moe
