// Gate-weighted combine: out[t] = sum_s gate[t,s] * y_perm[row_of[t,s]]
// (gate == nullptr: the rows already carry their gates, weight 1 each).
// One warp per (head, token) unit, grid-stride, scatter-free (each output row
// has one writer), fp32 accumulation in slot order, one bf16 rounding.
// 16-byte vector loads.
// Follows the last step of the MagiMoE operator library's routing -> sorting ->
// calculation chain ("Sand.ai: The world's first 100-billion-parameter open-source MoE video generation model MAGI Preview" (36kr), section "02. Two Key Technical Decision Points"):
// the routed experts' outputs are brought back to token order and summed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"
#include "moe.h"

namespace moe {

__device__ __forceinline__ void acc8(float (&a)[8], const uint4& v, float g) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(p[i]);
    a[2 * i] = fmaf(g, f.x, a[2 * i]);
    a[2 * i + 1] = fmaf(g, f.y, a[2 * i + 1]);
  }
}

template <int KMAX>
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ row_of,
                                                      const float* __restrict__ gate, uint4* __restrict__ out,
                                                      int64_t T, int d_vec, int64_t out_ld_vec, int k,
                                                      int64_t rows, int heads) {
  const int lane = threadIdx.x & 31;
  const int64_t wg = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const uint4* y0 = y;
  uint4* out0 = out;
  const int32_t* row_of0 = row_of;
  const float* gate0 = gate;
  const int64_t units = T * heads;
  // (head, token) unit ht: head h's outputs go to its d columns.  The next
  // unit's rows and gates are loaded while this one is summed (with short
  // rows, e.g. one 512-byte head slice per lane group, that load chain would
  // otherwise be exposed on every unit).
  int r_n = -1;
  float g_n = 0.f;
  if (wg < units && lane < k) {
    const int64_t h = wg / T, t = wg - h * T;
    r_n = __ldg(row_of0 + h * T * k + t * k + lane);
    g_n = gate0 != nullptr ? __ldg(gate0 + h * T * k + t * k + lane) : 1.0f;
  }
  for (int64_t ht = wg; ht < units; ht += nw) {
    const int64_t h = ht / T, t = ht - h * T;
    y = y0 + h * rows * d_vec;
    out = out0 + h * d_vec;
    int r_l = r_n;
    const float g_l = g_n;
    if (lane < k && (r_l < 0 || r_l >= rows)) r_l = -1;
    const int64_t nx = ht + nw;
    if (nx < units && lane < k) {
      const int64_t h2 = nx / T, t2 = nx - h2 * T;
      r_n = __ldg(row_of0 + h2 * T * k + t2 * k + lane);
      g_n = gate0 != nullptr ? __ldg(gate0 + h2 * T * k + t2 * k + lane) : 1.0f;
    }
    int r[KMAX];
    float g[KMAX];
#pragma unroll
    for (int s = 0; s < KMAX; ++s) {
      r[s] = __shfl_sync(0xffffffffu, r_l, s);
      g[s] = __shfl_sync(0xffffffffu, g_l, s);
    }
    for (int c = lane; c < d_vec; c += 32) {
      uint4 v[KMAX];
#pragma unroll
      for (int s = 0; s < KMAX; ++s)
        if (s < k && r[s] >= 0) v[s] = __ldcs(y + static_cast<int64_t>(r[s]) * d_vec + c);
      float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < KMAX; ++s)
        if (s < k && r[s] >= 0) acc8(a, v[s], g[s]);
      uint4 o;
      __nv_bfloat162 b0 = __floats2bfloat162_rn(a[0], a[1]);
      __nv_bfloat162 b1 = __floats2bfloat162_rn(a[2], a[3]);
      __nv_bfloat162 b2 = __floats2bfloat162_rn(a[4], a[5]);
      __nv_bfloat162 b3 = __floats2bfloat162_rn(a[6], a[7]);
      o.x = *reinterpret_cast<uint32_t*>(&b0);
      o.y = *reinterpret_cast<uint32_t*>(&b1);
      o.z = *reinterpret_cast<uint32_t*>(&b2);
      o.w = *reinterpret_cast<uint32_t*>(&b3);
      out[t * out_ld_vec + c] = o;
    }
  }
}

int launch_combine(const CombineArgs& a, cudaStream_t stream) {
  const int d_vec = a.d / 8;
  const int64_t want = (a.T * (a.heads > 1 ? a.heads : 1) + 7) / 8;
  const int grid = static_cast<int>(want < a.sm_count * 8LL ? want : a.sm_count * 8LL);
  const auto* y = reinterpret_cast<const uint4*>(a.y_perm);
  auto* o = reinterpret_cast<uint4*>(a.out);
  const int64_t rows = a.T * a.k;
  const int64_t out_ld_vec = (a.out_ld ? a.out_ld : a.d) / 8;
  const int heads = a.heads > 1 ? a.heads : 1;
  if (a.k <= 6)
    combine_kernel<6><<<grid, 256, 0, stream>>>(y, a.row_of, a.gate, o, a.T, d_vec, out_ld_vec, a.k, rows, heads);
  else
    combine_kernel<8><<<grid, 256, 0, stream>>>(y, a.row_of, a.gate, o, a.T, d_vec, out_ld_vec, a.k, rows, heads);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
