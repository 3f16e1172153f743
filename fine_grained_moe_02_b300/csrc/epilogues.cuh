// Epilogues of the tcgen05 GEMM engine.  Each thread owns one accumulator
// row (its TMEM lane) and walks the tile's columns 16 at a time.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "gemm_tc.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void store16_bf16(uint16_t* dst, const float (&v)[16]) {
  uint4 a, b;
  a.x = pack_bf16x2(v[0], v[1]);   a.y = pack_bf16x2(v[2], v[3]);
  a.z = pack_bf16x2(v[4], v[5]);   a.w = pack_bf16x2(v[6], v[7]);
  b.x = pack_bf16x2(v[8], v[9]);   b.y = pack_bf16x2(v[10], v[11]);
  b.z = pack_bf16x2(v[12], v[13]); b.w = pack_bf16x2(v[14], v[15]);
  reinterpret_cast<uint4*>(dst)[0] = a;
  reinterpret_cast<uint4*>(dst)[1] = b;
}

// out[row, n_blk*BN + j] = bf16(acc[j])  (expert GEMM-2: y_perm)
struct EpiStoreBf16 {
  struct Params {
    uint16_t* out;
    int64_t ld;
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const TileCoord& c, uint32_t taddr, int r, int) {
    const int row = c.row0 + r;
    const bool valid = row < c.row_end;
    uint16_t* dst = p.out + static_cast<int64_t>(row) * p.ld + c.n_blk * BN;
#pragma unroll 4
    for (int col = 0; col < BN; col += 16) {
      uint32_t u[16];
      __syncwarp();
      ptx::tmem_ld16(taddr + col, u);
      ptx::tmem_ld_wait();
      if (valid) {
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(u[j]);
        store16_bf16(dst + col, v);
      }
    }
  }
};

// Expert GEMM-1 with fused SwiGLU.  The B operand is the interleaved w13:
// within every 128 output columns, 64 gate rows then the matching 64 up rows.
// act[row, n_blk*BN/2 + 64*j + i] = bf16(silu(g) * u).
struct EpiSwiGLU {
  struct Params {
    uint16_t* act;
    int64_t ld;
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const TileCoord& c, uint32_t taddr, int r, int) {
    static_assert(BN % 128 == 0, "SwiGLU tiles hold whole 64+64 gate/up blocks");
    const int row = c.row0 + r;
    const bool valid = row < c.row_end;
    uint16_t* dst = p.act + static_cast<int64_t>(row) * p.ld + c.n_blk * (BN / 2);
#pragma unroll 1
    for (int j = 0; j < BN / 128; ++j) {
#pragma unroll
      for (int cc = 0; cc < 64; cc += 16) {
        uint32_t g[16], u[16];
        __syncwarp();
        ptx::tmem_ld16(taddr + j * 128 + cc, g);
        ptx::tmem_ld16(taddr + j * 128 + 64 + cc, u);
        ptx::tmem_ld_wait();
        if (valid) {
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float gv = __uint_as_float(g[i]);
            const float uv = __uint_as_float(u[i]);
            v[i] = gv / (1.0f + __expf(-gv)) * uv;
          }
          store16_bf16(dst + j * 64 + cc, v);
        }
      }
    }
  }
};

// Router stage 1: latent h (fp32 accumulator) -> bf16 hi + lo pair.
// hl[row, col] = hi, hl[row, L + col] = lo, with hi = bf16(h), lo = bf16(h - hi).
struct EpiHiLo {
  struct Params {
    uint16_t* hl;
    int64_t ld;  // 2L
    int L;
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const TileCoord& c, uint32_t taddr, int r, int) {
    const int row = c.row0 + r;
    const bool valid = row < c.row_end;
    uint16_t* dst = p.hl + static_cast<int64_t>(row) * p.ld + c.n_blk * BN;
#pragma unroll 2
    for (int col = 0; col < BN; col += 16) {
      uint32_t u[16];
      __syncwarp();
      ptx::tmem_ld16(taddr + col, u);
      ptx::tmem_ld_wait();
      if (valid) {
        float hi[16], lo[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float h = __uint_as_float(u[j]);
          const float hb = __bfloat162float(__float2bfloat16_rn(h));
          hi[j] = hb;
          lo[j] = h - hb;  // exact in fp32; rounded to bf16 by the store
        }
        store16_bf16(dst + col, hi);
        store16_bf16(dst + p.L + col, lo);
      }
    }
  }
};

// Router stage 2: summed head scores (fp32 accumulator, all E experts in one
// tile) -> + bias -> optional logits store -> top-k (value descending, ties
// to the lower expert index) -> softmax over the chosen k.
struct EpiTopK {
  struct Params {
    const float* bias;  // [E] or nullptr
    float* logits;      // [T, E] or nullptr
    int32_t* idx;       // [T, k]
    float* gate;        // [T, k]
    int E;
    int k;
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const TileCoord& c, uint32_t taddr, int r, int) {
    const int row = c.row0 + r;
    const bool valid = row < c.row_end;
    float bv[kMaxTopK];
    int bi[kMaxTopK];
#pragma unroll
    for (int i = 0; i < kMaxTopK; ++i) { bv[i] = -INFINITY; bi[i] = -1; }
    float* lrow = (p.logits != nullptr && valid) ? p.logits + static_cast<int64_t>(row) * p.E : nullptr;
#pragma unroll 1
    for (int col = 0; col < BN; col += 16) {
      uint32_t u[16];
      __syncwarp();
      ptx::tmem_ld16(taddr + col, u);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int e = col + j;
        if (e < p.E) {
          float s = __uint_as_float(u[j]);
          if (p.bias != nullptr) s += __ldg(p.bias + e);
          if (lrow != nullptr) lrow[e] = s;
          if (s > bv[kMaxTopK - 1]) {
            float cv = s;
            int ci = e;
#pragma unroll
            for (int q = 0; q < kMaxTopK; ++q) {
              const bool gt = cv > bv[q];
              const float tv = gt ? bv[q] : cv;
              const int ti = gt ? bi[q] : ci;
              bv[q] = gt ? cv : bv[q];
              bi[q] = gt ? ci : bi[q];
              cv = tv;
              ci = ti;
            }
          }
        }
      }
    }
    if (!valid) return;
    const float m = bv[0];
    float w[kMaxTopK];
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxTopK; ++i) {
      w[i] = (i < p.k) ? expf(bv[i] - m) : 0.f;
      sum += w[i];
    }
    const float inv = 1.0f / sum;
    int32_t* io = p.idx + static_cast<int64_t>(row) * p.k;
    float* go = p.gate + static_cast<int64_t>(row) * p.k;
#pragma unroll
    for (int i = 0; i < kMaxTopK; ++i) {
      if (i < p.k) {
        io[i] = bi[i];
        go[i] = w[i] * inv;
      }
    }
  }
};

}  // namespace moe
