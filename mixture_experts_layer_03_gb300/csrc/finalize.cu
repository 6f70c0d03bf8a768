// Step 5: finalize (TensorRT-LLM MoE page: the top-k weighted row sum, routing weights
// applied after FC2; layer-structure figure: routed and shared outputs are summed).
//   y[t] = sum_{j<k} scales[t, j] * out_perm[perm_inv[t*k + j]]  (+ out_perm[P + t])
// One block per token; fp32 accumulation in fixed slot order (deterministic); 16-byte
// vector loads of bf16 rows; one rounding to bf16 at the store.
#include <cstdint>

#include <cuda_bf16.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kFinThreads = 128;

__device__ __forceinline__ void acc_row(float (&acc)[8], uint4 v, float s) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    acc[2 * i] = fmaf(s, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(s, f.y, acc[2 * i + 1]);
  }
}

__global__ void __launch_bounds__(kFinThreads)
finalize_kernel(const __nv_bfloat16* __restrict__ out_perm, const int32_t* __restrict__ perm_inv,
                const float* __restrict__ scales, int64_t T, int k, int H, int64_t shared_row0,
                __nv_bfloat16* __restrict__ y) {
  __shared__ int64_t s_row[8];
  __shared__ float s_scale[8];
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    if (threadIdx.x < k) {
      const int32_t pos = perm_inv[t * k + threadIdx.x];
      s_row[threadIdx.x] = pos;
      s_scale[threadIdx.x] = scales[t * k + threadIdx.x];
    }
    __syncthreads();
    const int nvec = H / 8;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      for (int j = 0; j < k; ++j) {
        const int64_t r = s_row[j];
        if (r < 0) continue;   // id outside [0, E): the row was skipped
        const uint4 val = __ldg(reinterpret_cast<const uint4*>(out_perm + r * H) + v);
        acc_row(acc, val, s_scale[j]);
      }
      if (shared_row0 >= 0) {
        const uint4 val =
            __ldg(reinterpret_cast<const uint4*>(out_perm + (shared_row0 + t) * H) + v);
        acc_row(acc, val, 1.0f);
      }
      uint4 o;
      uint32_t* po = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        po[i] = *reinterpret_cast<uint32_t*>(&b);
      }
      reinterpret_cast<uint4*>(y + t * H)[v] = o;
    }
    __syncthreads();
  }
}

__global__ void cast_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out,
                            int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = __float2bfloat16_rn(in[i]);
}

}  // namespace

moe_status launch_finalize(const moe_problem& p, const moe_ws_layout& L, const float* scales,
                           void* y, const char* ws, cudaStream_t s) {
  const int64_t P = p.T * p.k;
  int64_t grid = p.T;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 32;
  if (grid > cap) grid = cap;
  finalize_kernel<<<static_cast<unsigned>(grid), kFinThreads, 0, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(ws + L.out_perm),
      reinterpret_cast<const int32_t*>(ws + L.perm_inv), scales, p.T, p.k, p.H,
      p.shared_I > 0 ? P : -1, static_cast<__nv_bfloat16*>(y));
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess)
    return set_error(MOE_ERR_CUDA, "finalize launch: %s", cudaGetErrorString(err));
  return MOE_OK;
}

moe_status launch_cast_f32_bf16(const float* in, void* out, int64_t n, cudaStream_t s) {
  if (n == 0) return MOE_OK;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  cast_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(in, static_cast<__nv_bfloat16*>(out), n);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return set_error(MOE_ERR_CUDA, "cast launch: %s", cudaGetErrorString(err));
  return MOE_OK;
}

}  // namespace moe
