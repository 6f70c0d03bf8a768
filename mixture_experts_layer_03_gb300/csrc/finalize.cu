// Step 5: finalize (TensorRT-LLM MoE page: the top-k weighted row sum, routing weights
// applied after FC2; layer-structure figure: routed and shared outputs are summed).
//   y[t] = sum_{j<k} scales[t, j] * out_perm[perm_inv[t*k + j]]  (+ out_perm[P + t])
// fp32 accumulation in fixed slot order (deterministic); 16-byte vector loads of bf16
// rows; one rounding to bf16 at the store.
#include <cstdint>

#include <cuda_bf16.h>

#include "internal.h"
#include "launch.cuh"

namespace moe {
namespace {

constexpr int kFinThreads = 256;

__device__ __forceinline__ void acc_row(float (&acc)[8], uint4 v, float s) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    acc[2 * i] = fmaf(s, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(s, f.y, acc[2 * i + 1]);
  }
}

// One thread per 16-byte vector (8 channels) of one token: its K row loads are issued
// together, then accumulated in slot order j = 0..K-1 (then the shared row).
template <int K>
__global__ void __launch_bounds__(kFinThreads)
finalize_kernel(const __nv_bfloat16* __restrict__ out_perm, const int32_t* __restrict__ perm_inv,
                const float* __restrict__ scales, const float* __restrict__ shared_gate, int64_t T,
                int H, int64_t shared_row0, __nv_bfloat16* __restrict__ y) {
  constexpr int k = K;
  constexpr int kMaxK = K;
  pdl_trigger();
  pdl_wait();
  const int nvec = H / 8;
  const int64_t total = T * nvec;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int64_t t = i / nvec;
    const int v = static_cast<int>(i - t * nvec);
    int32_t row[kMaxK];
    float sc[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      row[j] = __ldg(perm_inv + t * k + j);
      sc[j] = __ldg(scales + t * k + j);
    }
    uint4 val[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (row[j] >= 0)   // rows of ids outside [0, E) were skipped
        val[j] = __ldg(reinterpret_cast<const uint4*>(out_perm + static_cast<int64_t>(row[j]) * H) + v);
    uint4 shv;
    if (shared_row0 >= 0)
      shv = __ldg(reinterpret_cast<const uint4*>(out_perm + (shared_row0 + t) * H) + v);
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (row[j] >= 0) acc_row(acc, val[j], sc[j]);
    if (shared_row0 >= 0) {
      // Fused shared-expert gate (vLLM MoE page, "Gate 计算与 FSE"): sigmoid of its logit.
      const float gs = shared_gate ? 1.0f / (1.0f + expf(-__ldg(shared_gate + t))) : 1.0f;
      acc_row(acc, shv, gs);
    }
    uint4 o;
    uint32_t* po = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * c], acc[2 * c + 1]);
      po[c] = *reinterpret_cast<uint32_t*>(&b);
    }
    reinterpret_cast<uint4*>(y + t * H)[v] = o;
  }
}

__global__ void cast_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out,
                            int64_t n) {
  pdl_trigger();
  pdl_wait();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = __float2bfloat16_rn(in[i]);
}

template <int K>
cudaError_t launch_finalize_k(const moe_problem& p, const moe_ws_layout& L, const float* scales,
                              const float* shared_gate, void* y, const char* ws, cudaStream_t s) {
  const int64_t P = p.T * p.k;
  const int64_t total = p.T * (p.H / 8);
  int64_t grid = (total + kFinThreads - 1) / kFinThreads;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 32;
  if (grid > cap) grid = cap;
  return launch_pdl(finalize_kernel<K>, dim3(static_cast<unsigned>(grid)), dim3(kFinThreads), 0, s,
                    reinterpret_cast<const __nv_bfloat16*>(ws + L.out_perm),
                    reinterpret_cast<const int32_t*>(ws + L.perm_inv), scales, shared_gate, p.T, p.H,
                    static_cast<int64_t>(p.shared_I > 0 ? P : -1), static_cast<__nv_bfloat16*>(y));
}

}  // namespace

moe_status launch_finalize(const moe_problem& p, const moe_ws_layout& L, const float* scales,
                           const float* shared_gate, void* y, const char* ws, cudaStream_t s) {
  cudaError_t err;
  switch (p.k) {
    case 1: err = launch_finalize_k<1>(p, L, scales, shared_gate, y, ws, s); break;
    case 2: err = launch_finalize_k<2>(p, L, scales, shared_gate, y, ws, s); break;
    case 3: err = launch_finalize_k<3>(p, L, scales, shared_gate, y, ws, s); break;
    case 4: err = launch_finalize_k<4>(p, L, scales, shared_gate, y, ws, s); break;
    case 5: err = launch_finalize_k<5>(p, L, scales, shared_gate, y, ws, s); break;
    case 6: err = launch_finalize_k<6>(p, L, scales, shared_gate, y, ws, s); break;
    case 7: err = launch_finalize_k<7>(p, L, scales, shared_gate, y, ws, s); break;
    default: err = launch_finalize_k<8>(p, L, scales, shared_gate, y, ws, s); break;
  }
  if (err != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "finalize launch: %s", cudaGetErrorString(err));
  return MOE_OK;
}

moe_status launch_cast_f32_bf16(const float* in, void* out, int64_t n, cudaStream_t s) {
  if (n == 0) return MOE_OK;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  cudaError_t err = launch_pdl(cast_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, in,
                               static_cast<__nv_bfloat16*>(out), n);
  if (err != cudaSuccess) return set_error(MOE_ERR_CUDA, "cast launch: %s", cudaGetErrorString(err));
  return MOE_OK;
}

}  // namespace moe
