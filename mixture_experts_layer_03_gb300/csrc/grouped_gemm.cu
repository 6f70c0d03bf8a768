// Steps 3 and 4: grouped GEMM over all experts in one persistent launch.
//
// Scheduling (Dense GEMM -> GroupedGEMM article, section 2.2): tile scheduling over a
// flattened global tile list rather than one block per expert. The permute step wrote,
// per group g (routed experts, then the optional shared expert), its row count m_g, its
// first permuted row, and an exclusive scan of its tile counts. Group g contributes
//     n_mt(g) = floor(m_g / 128) + (m_g % 128 != 0)  row tiles  x  n_nt(g) channel tiles.
// Row tile mt < floor(m_g/128) is a full 128-row tile computed "token-major":
//     D[128 tokens, 256] = X[128, K] . W[256, K]^T                  (one UMMA, N = 256)
// The last, partial row tile (1..127 rows) is computed "weight-major" (swap AB), so a
// few tokens do not waste a 128-row MMA:
//     D0[128 ch, n] = W[0:128, K] . X[n, K]^T,  D1[128 ch, n] = W[128:256, K] . X[n, K]^T
// with n = rows rounded up to 16. Small experts (decode) therefore stream their weights
// once through MMAs of M = 128 and N = 16..128.
//
// W rows per tile: FC1 loads gate rows [n0, n0+128) and up rows [I+n0, I+n0+128) of
// w13[e] (w13 = gate and up merged, vLLM MoE page, section "专家权重如何存储"), so gate
// channel c and up channel c land in the same TMEM lane (weight-major) or the same
// thread's columns c and 128+c (token-major); the SwiGLU epilogue h = silu(gate) * up
// needs no exchange. FC2 loads w2[e] rows [n0, n0+256) (output channels).
//
// Warp roles (192 threads): warp 0 = TMA producer and tile scheduler, warp 1 = TMEM
// allocator + MMA issuer, warps 2-5 = epilogue (TMEM lanes 32*(warp%4) .. +31). A 4-stage
// smem ring (16 KB X + 32 KB W per stage) feeds the MMAs; two 256-column TMEM
// accumulators let the epilogue of one tile overlap the mainloop of the next.
//
// Tiles are claimed dynamically: the producer takes the next index from a global atomic
// counter and passes it to the MMA and epilogue warps through a small smem ring, so CTAs
// that run faster (L2 hits, lighter tiles, the nearer die) take more tiles. Claims move
// through the flattened list in order, so the tiles in flight at any time are neighbours
// that share weight panels in L2. The last CTA to finish resets the counter.
//
// Rows past a group's end inside a tile read the next group's rows (or zero fill past
// the tensor); they only reach accumulator rows/columns that the epilogue masks.
#include <cstdint>
#include <cstdio>

#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kBK = 64;                              // K elements per stage
constexpr int kRowBytes = kBK * 2;                   // one K row of a tile = the swizzle width
constexpr int kStages = 4;
constexpr int kXStageBytes = 128 * kRowBytes;        // 128 rows of X
constexpr int kWHalfBytes = 128 * kRowBytes;         // 128 rows of W
constexpr int kWStageBytes = 2 * kWHalfBytes;
constexpr int kAccCols = 256;
constexpr int kTmemCols = 512;
constexpr int kThreads = 192;
constexpr int kMaxGroups = 257;
constexpr int kSchedDepth = 4;                       // tile indices in flight inside a CTA
constexpr int kSmemBytes = 1024 /*alignment slack*/ + kStages * (kXStageBytes + kWStageBytes);

struct GemmArgs {
  const int32_t* counts;    // [G]
  const int32_t* starts;    // [G]
  const int32_t* tile_off;  // [G+1]
  int32_t G;
  int32_t E;                // routed groups; group E (if G > E) uses the shared maps
  int32_t K_routed, K_shared;
  int32_t N_routed, N_shared;   // FC1: I / shared_I (channels); FC2: H
  __nv_bfloat16* out;
  int64_t out_ld;
  int32_t* status;
  int32_t* sched;           // [0] next tile to claim, [1] CTAs finished (both reset to 0 at exit)
};

struct Tile {
  int g;
  int token_major;   // 1: 128-row tile, 0: weight-major remainder tile
  int row0;          // first permuted row
  int rows;          // valid rows (<= 128)
  int ntok;          // weight-major: rows rounded up to 16
  int n0;            // first output channel
  int K;
  int N;             // channels of this group
};

__device__ __forceinline__ Tile decode_tile(int tile, const int32_t* s_off, const int32_t* s_cnt,
                                            const int32_t* s_start, const GemmArgs& a,
                                            bool fc1) {
  // Largest g with tile_off[g] <= tile (groups with no tiles have equal offsets).
  int lo = 0, hi = a.G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_off[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  Tile t;
  t.g = lo;
  const int m = s_cnt[lo];
  const int nfull = m / 128;
  const int n_mt = nfull + (m % 128 != 0);
  const int local = tile - s_off[lo];
  const int nt = local / n_mt;
  const int mt = local - nt * n_mt;
  t.token_major = mt < nfull;
  t.row0 = s_start[lo] + mt * 128;
  t.rows = min(128, m - mt * 128);
  t.ntok = (t.rows + 15) & ~15;
  const bool shared = lo >= a.E;
  t.K = shared ? a.K_shared : a.K_routed;
  t.N = shared ? a.N_shared : a.N_routed;
  t.n0 = nt * (fc1 ? kFc1Cols : kFc2Cols);
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

template <bool kFc1>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_x128,   // A rows, box 64 x 128
                    const __grid_constant__ CUtensorMap map_x16,    // A rows, box 64 x 16
                    const __grid_constant__ CUtensorMap map_w,      // routed weights [E, R, K]
                    const __grid_constant__ CUtensorMap map_ws,     // shared weights [1, R, K]
                    GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages];
  __shared__ uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ uint64_t sched_full[kSchedDepth], sched_empty[kSchedDepth];
  __shared__ int s_tile[kSchedDepth];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int32_t s_off[kMaxGroups + 1], s_cnt[kMaxGroups], s_start[kMaxGroups];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // 1024-byte aligned stage buffers (the 128-byte swizzle repeats every 1024 bytes).
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sX = smem;                                   // kStages x 16 KB
  uint8_t* sW = smem + kStages * kXStageBytes;          // kStages x 256 W rows

  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
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
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&map_x128);
    tma_prefetch_map(&map_x16);
    tma_prefetch_map(&map_w);
    tma_prefetch_map(&map_ws);
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // Everything above overlaps the previous kernel; the work lists are its output.
  pdl_wait();
  for (int i = threadIdx.x; i <= a.G; i += blockDim.x) s_off[i] = a.tile_off[i];
  for (int i = threadIdx.x; i < a.G; i += blockDim.x) {
    s_cnt[i] = a.counts[i];
    s_start[i] = a.starts[i];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  volatile int* abort = &s_abort;
  const int total = s_off[a.G];

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
          flag_timeout(a.status, abort);
          ok = false;
          break;
        }
        int tile = atomicAdd(a.sched, 1);
        if (tile >= total) tile = -1;
        s_tile[slot] = tile;
        mbar_arrive(&sched_full[slot]);
        if (tile < 0) break;
        const Tile t = decode_tile(tile, s_off, s_cnt, s_start, a, kFc1);
        const bool shared = t.g >= a.E;
        const CUtensorMap* mw = shared ? &map_ws : &map_w;
        const int ecoord = shared ? 0 : t.g;
        const int wr0 = t.n0;
        const int wr1 = kFc1 ? (t.N + t.n0) : (t.n0 + 128);
        const uint32_t bytes =
            kWStageBytes + (t.token_major ? kXStageBytes : static_cast<uint32_t>(t.ntok) * kRowBytes);
        const int nkb = t.K / kBK;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort)) {
            flag_timeout(a.status, abort);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[stage], bytes);
          const int kc = kb * kBK;
          uint8_t* xs = sX + stage * kXStageBytes;
          uint8_t* ws = sW + stage * kWStageBytes;
          if (t.token_major) {
            tma_load_2d(xs, &map_x128, &full_bar[stage], kc, t.row0);
          } else {
            for (int r = 0; r < t.ntok; r += 16)
              tma_load_2d(xs + r * kRowBytes, &map_x16, &full_bar[stage], kc, t.row0 + r);
          }
          tma_load_3d(ws, mw, &full_bar[stage], kc, wr0, ecoord);
          tma_load_3d(ws + kWHalfBytes, mw, &full_bar[stage], kc, wr1, ecoord);
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA exits: wait (bounded)
        // on the full barrier of each of the last kStages issues.
        int s = stage;
        uint32_t ph = phase;
        const int n = issued < kStages ? issued : kStages;
        for (int i = 0; i < n; ++i) {
          if (--s < 0) {
            s = kStages - 1;
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
      const uint32_t sx0 = smem_u32(sX), sw0 = smem_u32(sW);
      for (int it = 0; ok; ++it) {
        const int slot = it & (kSchedDepth - 1);
        if (!mbar_wait(&sched_full[slot], (it / kSchedDepth) & 1, abort)) {
          flag_timeout(a.status, abort);
          ok = false;
          break;
        }
        const int tile = *reinterpret_cast<volatile int*>(&s_tile[slot]);
        mbar_arrive(&sched_empty[slot]);
        if (tile < 0) break;
        const Tile t = decode_tile(tile, s_off, s_cnt, s_start, a, kFc1);
        if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort)) {
          flag_timeout(a.status, abort);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kAccCols);
        const uint32_t idesc = t.token_major ? idesc_bf16_f32(128, 256) : idesc_bf16_f32(128, t.ntok);
        const int nkb = t.K / kBK;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abort)) {
            flag_timeout(a.status, abort);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t xa = sx0 + stage * kXStageBytes;
          const uint32_t wa = sw0 + stage * kWStageBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t accum = (kb | kk) != 0;
            const uint64_t dx = sdesc_k_major(xa + kk * 32, kRowBytes);
            if (t.token_major) {
              umma_bf16(d, dx, sdesc_k_major(wa + kk * 32, kRowBytes), idesc, accum);
            } else {
              umma_bf16(d, sdesc_k_major(wa + kk * 32, kRowBytes), dx, idesc, accum);
              umma_bf16(d + 128, sdesc_k_major(wa + kWHalfBytes + kk * 32, kRowBytes), dx, idesc,
                        accum);
            }
          }
          umma_commit(&empty_bar[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
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
    const int lrow = q * 32 + lane;         // accumulator row (lane) of this thread
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = 0;; ++it) {
      const int slot = it & (kSchedDepth - 1);
      const bool have = mbar_wait(&sched_full[slot], (it / kSchedDepth) & 1, abort);
      if (!__all_sync(0xffffffffu, have)) {
        flag_timeout(a.status, abort);
        break;
      }
      const int tile = *reinterpret_cast<volatile int*>(&s_tile[slot]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sched_empty[slot]);
      if (tile < 0) break;
      const Tile t = decode_tile(tile, s_off, s_cnt, s_start, a, kFc1);
      const bool got = mbar_wait(&tfull_bar[acc], acc_phase, abort);
      // Lanes may leave the poll at different times; tcgen05.ld is warp-collective.
      if (!__all_sync(0xffffffffu, got)) {
        flag_timeout(a.status, abort);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * kAccCols) +
                          (static_cast<uint32_t>(q * 32) << 16);
      float va[16], vb[16];
      if (t.token_major) {
        // Thread = token row lrow; columns = channels.
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
      } else {
        // Thread = channel lrow (of the 128 in D0, and of D1); columns = tokens.
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
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0) {
    // Every CTA has claimed its last tile before it gets here; the last one to arrive
    // resets the counters for the next launch on this workspace.
    __threadfence();
    if (atomicAdd(a.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(a.sched, 0);
      atomicExch(a.sched + 1, 0);
    }
  }
}

// ---------------------------------------------------------------- host side

constexpr CUtensorMapSwizzle kSwizzle =
    kRowBytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// bf16 matrix [rows, cols] (cols contiguous), box = 64 cols x box_rows rows.
bool encode_map2(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {kBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, kSwizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 tensor [planes, rows, cols] (cols contiguous), box = 64 cols x box_rows rows x 1.
bool encode_map3(CUtensorMap* m, const void* base, uint64_t planes, uint64_t rows, uint64_t cols,
                 uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {cols, rows, planes};
  cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  cuuint32_t box[3] = {kBK, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, kSwizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool kFc1>
moe_status prepare_kernel() {
  static int done_dev[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return set_error(MOE_ERR_CUDA, "cudaGetDevice failed");
  if (!done_dev[dev]) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<kFc1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess)
      return set_error(MOE_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    done_dev[dev] = 1;
  }
  return MOE_OK;
}

template <bool kFc1>
moe_status launch_gemm(const moe_problem& p, const moe_ws_layout& L, const void* w,
                       const void* w_s, char* ws, cudaStream_t s) {
  moe_status st = prepare_kernel<kFc1>();
  if (st != MOE_OK) return st;
  const int64_t R = L.rows;
  const int has_shared = p.shared_I > 0;
  CUtensorMap mx128, mx16, mw, mws;
  const void* A = kFc1 ? static_cast<const void*>(ws + L.x_perm) : static_cast<const void*>(ws + L.h);
  const uint64_t a_cols = kFc1 ? static_cast<uint64_t>(p.H) : static_cast<uint64_t>(L.h_ld);
  bool ok = encode_map2(&mx128, A, R, a_cols, 128) && encode_map2(&mx16, A, R, a_cols, 16);
  if (kFc1) {
    ok = ok && encode_map3(&mw, w, p.E, 2ull * p.I, p.H, 128);
    ok = ok && (has_shared ? encode_map3(&mws, w_s, 1, 2ull * p.shared_I, p.H, 128)
                           : encode_map3(&mws, w, p.E, 2ull * p.I, p.H, 128));
  } else {
    ok = ok && encode_map3(&mw, w, p.E, p.H, p.I, 128);
    ok = ok && (has_shared ? encode_map3(&mws, w_s, 1, p.H, p.shared_I, 128)
                           : encode_map3(&mws, w, p.E, p.H, p.I, 128));
  }
  if (!ok) return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed");

  GemmArgs a;
  a.counts = reinterpret_cast<const int32_t*>(ws + L.counts);
  a.starts = reinterpret_cast<const int32_t*>(ws + L.starts);
  a.tile_off = reinterpret_cast<const int32_t*>(ws + (kFc1 ? L.tile_off1 : L.tile_off2));
  a.G = L.groups;
  a.E = p.E;
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
  a.sched = reinterpret_cast<int32_t*>(ws + L.sched) + (kFc1 ? 0 : 2);

  // Upper bound on the device-side tile count: each group has at most
  // floor(m/128) + 1 row tiles.
  const int nI = has_shared && p.shared_I > p.I ? p.shared_I : p.I;
  const int64_t n_nt = kFc1 ? (nI + kFc1Cols - 1) / kFc1Cols : (p.H + kFc2Cols - 1) / kFc2Cols;
  const int64_t bound = ((R + 127) / 128 + L.groups) * n_nt;
  int64_t grid = device_sm_count();
  if (grid > bound) grid = bound;
  if (grid < 1) grid = 1;
  cudaError_t err = launch_pdl(grouped_gemm_kernel<kFc1>, dim3(static_cast<unsigned>(grid)),
                               dim3(kThreads), kSmemBytes, s, mx128, mx16, mw, mws, a);
  if (err != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "grouped_gemm launch: %s", cudaGetErrorString(err));
  return MOE_OK;
}

}  // namespace

moe_status launch_fc1(const moe_problem& p, const moe_ws_layout& L, const void* w13,
                      const void* w13_s, char* ws, cudaStream_t s) {
  return launch_gemm<true>(p, L, w13, w13_s, ws, s);
}

moe_status launch_fc2(const moe_problem& p, const moe_ws_layout& L, const void* w2,
                      const void* w2_s, char* ws, cudaStream_t s) {
  return launch_gemm<false>(p, L, w2, w2_s, ws, s);
}

}  // namespace moe
