// Folded router weights: W_eff = W_head W_lat (fp32, [E, d]) stored as a bf16
// hi/lo pair w_router[e] = [bf16(W_eff[e]) | bf16(W_eff[e] - hi)], so that
// s = x W_eff^T + b runs as one bf16 tensor-core GEMM with K = 2d
// (A = [x | x], B = w_router).  The summed head scores are linear in x, so
// this is the same function as latent projection followed by head scores.
// One-time preparation per weight load: a plain fp32 SIMT GEMM.
// The routing it computes is the multi-head latent routing of "MAGI-2 Preview" (heyaiwiki),
// Architecture table, "Routing" row.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"
#include "moe.h"

namespace moe {

constexpr int kFoldTile = 64;  // output tile 64 (experts) x 64 (hidden)
constexpr int kFoldK = 32;     // latent columns per step

// W_eff[e, i] = sum_l W_head[e, l] * W_lat[l, i]; 256 threads, 4x4 outputs each.
__global__ void __launch_bounds__(256) fold_router_kernel(const __nv_bfloat16* __restrict__ w_head,
                                                          const __nv_bfloat16* __restrict__ w_lat, int E, int L,
                                                          int d, __nv_bfloat16* __restrict__ w_router) {
  __shared__ float sh[kFoldK][kFoldTile + 1];  // W_head tile, transposed: [l][e]
  __shared__ float sl[kFoldK][kFoldTile];      // W_lat tile: [l][i]
  const int e0 = blockIdx.y * kFoldTile, i0 = blockIdx.x * kFoldTile;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 x 16 threads
  float acc[4][4] = {};
  for (int l0 = 0; l0 < L; l0 += kFoldK) {
    for (int t = threadIdx.x; t < kFoldK * kFoldTile; t += 256) {
      const int r = t / kFoldK, c = t % kFoldK;  // W_head[e0 + r, l0 + c]
      const int e = e0 + r;
      sh[c][r] = (e < E) ? __bfloat162float(w_head[static_cast<int64_t>(e) * L + l0 + c]) : 0.f;
      const int rr = t / kFoldTile, cc = t % kFoldTile;  // W_lat[l0 + rr, i0 + cc]
      sl[rr][cc] = __bfloat162float(w_lat[static_cast<int64_t>(l0 + rr) * d + i0 + cc]);
    }
    __syncthreads();
#pragma unroll 8
    for (int l = 0; l < kFoldK; ++l) {
      float a[4], b[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a[q] = sh[l][ty * 4 + q];
        b[q] = sl[l][tx * 4 + q];
      }
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[p][q] = fmaf(a[p], b[q], acc[p][q]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int e = e0 + ty * 4 + p;
    if (e >= E) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = i0 + tx * 4 + q;
      const float w = acc[p][q];
      const __nv_bfloat16 hi = __float2bfloat16_rn(w);
      const __nv_bfloat16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
      w_router[static_cast<int64_t>(e) * 2 * d + i] = hi;
      w_router[static_cast<int64_t>(e) * 2 * d + d + i] = lo;
    }
  }
}

int launch_fold_router(const uint16_t* w_head, const uint16_t* w_lat, int E, int L, int d, uint16_t* w_router,
                       cudaStream_t stream) {
  dim3 grid(d / kFoldTile, (E + kFoldTile - 1) / kFoldTile);
  fold_router_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const __nv_bfloat16*>(w_head),
                                              reinterpret_cast<const __nv_bfloat16*>(w_lat), E, L, d,
                                              reinterpret_cast<__nv_bfloat16*>(w_router));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
