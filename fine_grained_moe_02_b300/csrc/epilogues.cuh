// Epilogues of the tcgen05 GEMM engine: the router's hi/lo split and top-6
// selection ("MAGI-2 Preview" (heyaiwiki), Architecture table, "Routing" row), the
// experts' SwiGLU and the plain bf16 store.  Each thread owns one accumulator
// row (its TMEM lane); a warp owns 32 consecutive rows of the tile.  Results
// leave through a per-warp 32-row x 64-column staging chunk in shared memory
// (128-byte swizzled, the layout the output tensor map uses) and one TMA bulk
// store, so HBM sees whole 128-byte lines.  A warp whose 32 rows are cut by
// the end of an expert group stores its valid rows with plain 16-byte stores
// instead (the rows after the cut belong to the next group's tile).
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

// Loads 32 consecutive accumulator columns of this thread's row (one wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t a[16], b[16];
  ptx::tmem_ld16(taddr, a);
  ptx::tmem_ld16(taddr + 16, b);
  ptx::tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[i] = __uint_as_float(a[i]);
    v[16 + i] = __uint_as_float(b[i]);
  }
}

// Writes this warp's 32 rows x 64 bf16 columns (p[j] = columns 2j, 2j+1 of
// this thread's row) to the output at (row0w, col0).  nvalid = rows of the 32
// that may be written; row_ptr = this thread's row at col0 (fallback path).
__device__ __forceinline__ void store_rows64(EpiCtx& ctx, int row0w, int col0, int nvalid, const uint32_t* p,
                                             uint16_t* row_ptr) {
  if (nvalid >= 32) {
    if (ctx.pending) {  // the previous bulk store must be done reading the chunk
      if (ctx.lane == 0) ptx::bulk_wait_read_all();
      __syncwarp();
    }
    const uint32_t row_base = ctx.stage + static_cast<uint32_t>(ctx.lane) * 128u;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = make_uint4(p[4 * c], p[4 * c + 1], p[4 * c + 2], p[4 * c + 3]);
      ptx::st_shared_v4(row_base + ((static_cast<uint32_t>(c) ^ (ctx.lane & 7u)) << 4), v);
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (ctx.lane == 0) {
      ptx::tma_store_2d(ctx.tmap, ctx.stage, col0, row0w);
      ptx::bulk_commit();
    }
    ctx.pending = true;
  } else if (ctx.lane < nvalid) {
    uint4* dst = reinterpret_cast<uint4*>(row_ptr);
#pragma unroll
    for (int c = 0; c < 8; ++c) dst[c] = make_uint4(p[4 * c], p[4 * c + 1], p[4 * c + 2], p[4 * c + 3]);
  }
}

// Waits ctx.store_delay cycles (see EpiCtx) before a store-heavy epilogue's
// first store.  Expert GEMM-2 writes 64 KB per 128 x 256 tile against eight
// times less for GEMM-1; storing right when a tile's MMAs finish collides
// with the next tile's first operand loads.  On the clip workload, waiting
// half a tile's MMA time took GEMM-2 from 0.83 to 0.875 TFLOP/s per SM MHz,
// spreading the four warps' waits over 0.25-0.7 of it to 0.89.
__device__ __forceinline__ void store_delay_wait(const EpiCtx& ctx) {
  if (ctx.store_delay == 0) return;
  const long long t0 = clock64();
  while (clock64() - t0 < static_cast<long long>(ctx.store_delay)) __nanosleep(128);
}

// Hands the accumulator back to the MMA warp.  The caller's tcgen05.ld's have
// completed (tmem_ld32 waits on them), so the next tile's MMAs may overwrite
// the columns while this warp's stores of the tile are still under way.
__device__ __forceinline__ void release_accumulator(EpiCtx& ctx) {
  ptx::tc_fence_before();
  ptx::mbar_arrive(ctx.tempty);
  ctx.released = true;
}

// silu(g) = g * sigmoid(g) = g / (1 + e^-g): one ex2.approx for e^-g and one
// rcp.approx for the reciprocal (relative errors about 2^-22 and 1 ulp), so
// silu keeps fp32-level relative accuracy over the whole range, the negative
// side included, where the form h + h tanh(h) (h = g / 2) loses it: there
// 1 + tanh(h) cancels and tanh.approx's absolute error of ~2^-11 becomes a
// large relative one.  Two special-function ops and three other ops per
// value; a Newton-Raphson division in FMAs instead of the rcp (one
// special-function op, nine others) measured slower in the short-K SwiGLU
// epilogue of the head-local layer, which is bound by instruction issue.
// Far below -88, e^-g overflows to inf and the result is -0 (true value
// below 1e-36 in magnitude).
__device__ __forceinline__ float silu(float g) {
  float z, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(z) : "f"(-1.4426950408889634f * g));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + z));
  return g * r;
}

__device__ __forceinline__ int warp_valid_rows(const TileCoord& c, const EpiCtx& ctx) {
  const int first = c.row0 + ctx.quad * 32;
  const int n = c.row_end - first;
  return n < 0 ? 0 : (n > 32 ? 32 : n);
}

// out[row, n_blk*BN + j] = bf16(acc[j])  (expert GEMM-2: y_perm)
// The row's BN/2 packed bf16 pairs are read out of TMEM first and the
// accumulator released, so the MMAs of a later tile do not wait for the
// bulk stores of this one.
struct EpiStoreBf16 {
  static constexpr int kWarps = 4;
  struct Params {
    uint16_t* out;
    int64_t ld;
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const TileCoord& c, uint32_t taddr, int r,
                                             EpiCtx& ctx) {
    const int nvalid = warp_valid_rows(c, ctx);
    const int row = c.row0 + r;
    uint16_t* row_ptr = p.out + static_cast<int64_t>(row) * p.ld + c.n_blk * BN;
    uint32_t pk[BN / 2];
#pragma unroll
    for (int col = 0; col < BN; col += 32) {
      float v[32];
      __syncwarp();
      tmem_ld32(taddr + col, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) pk[col / 2 + j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
    }
    release_accumulator(ctx);
    store_delay_wait(ctx);
    if (nvalid > 0) {
#pragma unroll
      for (int col = 0; col < BN; col += 64)
        store_rows64(ctx, c.row0 + ctx.quad * 32, c.n_blk * BN + col, nvalid, pk + col / 2, row_ptr + col);
    }
  }
};

// Expert GEMM-2 with the gate multiply folded in:
//   y_perm[r] = bf16(gate[t, s] * acc),  t = src_token[r], row_of[t, s] = r,
// so the combine only sums a token's k rows.  Each thread finds its row's
// gate before it reads the accumulator (src_token, then the k row_of / gate
// entries of that token: L2-resident, their latency hidden behind the
// accumulator loads).  A row outside the group, or whose token does not list
// it, gets gate 0.
struct EpiStoreGated {
  static constexpr int kWarps = 4;
  struct Params {
    uint16_t* out;
    int64_t ld;
    const int32_t* src_token;  // [rows]
    const int32_t* row_of;     // [T, k]
    const float* gate;         // [T, k]
    int64_t T;
    int k;
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const TileCoord& c, uint32_t taddr, int r,
                                             EpiCtx& ctx) {
    const int nvalid = warp_valid_rows(c, ctx);
    const int row = c.row0 + r;
    float gw = 0.0f;
    if (row < c.row_end) {
      const int t = __ldg(p.src_token + row);
      if (t >= 0 && t < p.T) {
        const int64_t base = static_cast<int64_t>(t) * p.k;
#pragma unroll
        for (int s = 0; s < kMaxTopK; ++s)
          if (s < p.k && __ldg(p.row_of + base + s) == row) gw = __ldg(p.gate + base + s);
      }
    }
    uint16_t* row_ptr = p.out + static_cast<int64_t>(row) * p.ld + c.n_blk * BN;
    uint32_t pk[BN / 2];
#pragma unroll
    for (int col = 0; col < BN; col += 32) {
      float v[32];
      __syncwarp();
      tmem_ld32(taddr + col, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) pk[col / 2 + j] = pack_bf16x2(gw * v[2 * j], gw * v[2 * j + 1]);
    }
    release_accumulator(ctx);
    store_delay_wait(ctx);
    if (nvalid > 0) {
#pragma unroll
      for (int col = 0; col < BN; col += 64)
        store_rows64(ctx, c.row0 + ctx.quad * 32, c.n_blk * BN + col, nvalid, pk + col / 2, row_ptr + col);
    }
  }
};

// Expert GEMM-1 with fused SwiGLU.  The B operand is the interleaved w13:
// within every 128 output columns, 64 gate rows then the matching 64 up rows.
// act[row, n_blk*BN/2 + 64*j + i] = bf16(silu(g) * u).  All of the row's
// activations are formed in registers before the accumulator is released.
struct EpiSwiGLU {
  static constexpr int kWarps = 4;
  struct Params {
    uint16_t* act;
    int64_t ld;
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const TileCoord& c, uint32_t taddr, int r,
                                             EpiCtx& ctx) {
    static_assert(BN % 128 == 0, "SwiGLU tiles hold whole 64+64 gate/up blocks");
    const int nvalid = warp_valid_rows(c, ctx);
    const int row = c.row0 + r;
    uint16_t* row_ptr = p.act + static_cast<int64_t>(row) * p.ld + c.n_blk * (BN / 2);
    uint32_t pk[BN / 4];
#pragma unroll
    for (int j = 0; j < BN / 128; ++j) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float g[32], u[32];
        __syncwarp();
        tmem_ld32(taddr + j * 128 + h * 32, g);
        tmem_ld32(taddr + j * 128 + 64 + h * 32, u);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a0 = silu(g[2 * i]) * u[2 * i];
          const float a1 = silu(g[2 * i + 1]) * u[2 * i + 1];
          pk[j * 32 + h * 16 + i] = pack_bf16x2(a0, a1);
        }
      }
    }
    release_accumulator(ctx);
    if (nvalid > 0) {
#pragma unroll
      for (int j = 0; j < BN / 128; ++j)
        store_rows64(ctx, c.row0 + ctx.quad * 32, c.n_blk * (BN / 2) + j * 64, nvalid, pk + j * 32,
                     row_ptr + j * 64);
    }
  }
};

// Router stage 1: latent h (fp32 accumulator) -> bf16 hi + lo pair.
// hl[row, col] = hi, hl[row, L + col] = lo, with hi = bf16(h), lo = bf16(h - hi).
struct EpiHiLo {
  static constexpr int kWarps = 4;
  struct Params {
    uint16_t* hl;
    int64_t ld;  // 2L
    int L;
  };
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p, const TileCoord& c, uint32_t taddr, int r,
                                             EpiCtx& ctx) {
    const int nvalid = warp_valid_rows(c, ctx);
    const int row = c.row0 + r;
    uint16_t* row_ptr = p.hl + static_cast<int64_t>(row) * p.ld + c.n_blk * BN;
#pragma unroll 1
    for (int col = 0; col < BN; col += 64) {
      uint32_t hi[32], lo[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float v[32];
        __syncwarp();
        tmem_ld32(taddr + col + h * 32, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float h0 = v[2 * i], h1 = v[2 * i + 1];
          const float b0 = __bfloat162float(__float2bfloat16_rn(h0));
          const float b1 = __bfloat162float(__float2bfloat16_rn(h1));
          hi[h * 16 + i] = pack_bf16x2(b0, b1);
          lo[h * 16 + i] = pack_bf16x2(h0 - b0, h1 - b1);  // differences exact in fp32
        }
      }
      if (nvalid > 0) {
        const int r0 = c.row0 + ctx.quad * 32, c0 = c.n_blk * BN + col;
        store_rows64(ctx, r0, c0, nvalid, hi, row_ptr + col);
        store_rows64(ctx, r0, p.L + c0, nvalid, lo, row_ptr + p.L + col);
      }
    }
  }
};

// Summed head scores of one token (its TMEM lane, columns 0 .. E-1 from taddr)
// -> + bias -> optional logits row -> top-k (value descending, ties to the
// lower expert index) -> softmax over the chosen k -> idx/gate rows.  All 32
// lanes of the warp must call it (the TMEM loads are warp-collective).
constexpr int kMaxModalities = 8;

struct TopKParams {
  const float* bias;  // [E] or nullptr
  float* logits;      // [T, E] or nullptr
  int32_t* idx;       // [T, k_out]
  float* gate;        // [T, k_out]
  int E;
  int k;
  // Modality-specific routing and shared experts (all zero/null: plain layer).
  int k_out;                     // row stride of idx/gate: k + n_shared (0 means k)
  int n_shared;                  // slots k .. k_out-1 get experts E .. E+n_shared-1, gate 1
  const int32_t* modality;       // [T] modality id, or nullptr: every expert competes
  int n_mod;
  int ebeg[kMaxModalities], eend[kMaxModalities];
  int* status;                   // MOE_DEV_BAD_MODALITY for an id outside [0, n_mod)
  // Batched problems (one per GEMM group, rows g*T .. g*T+T-1 of the tile
  // space): outputs of group g start at idx + g*T*k_out, logits + g*T*E, bias + g*E.
  int T;                         // rows per group (0: not batched)
};

inline TopKParams make_topk_params(const RouteArgs& a) {
  TopKParams p{};
  p.bias = a.bias;
  p.logits = a.logits;
  p.idx = a.topk_idx;
  p.gate = a.topk_gate;
  p.E = a.E;
  p.k = a.k;
  p.k_out = a.k + a.ext.n_shared;
  p.n_shared = a.ext.n_shared;
  p.modality = a.ext.n_mod > 0 ? a.ext.modality : nullptr;
  p.n_mod = a.ext.n_mod;
  for (int m = 0; m < kMaxModalities; ++m) {
    p.ebeg[m] = a.ext.ebeg[m];
    p.eend[m] = a.ext.eend[m];
  }
  p.status = a.status;
  return p;
}

// The routed experts token `row` may choose: [*lo, *hi).
__device__ __forceinline__ void expert_range(const TopKParams& p, int row, bool valid, int* lo, int* hi) {
  *lo = 0;
  *hi = p.E;
  if (p.modality != nullptr && valid) {
    const int m = __ldg(p.modality + row);
    if (m >= 0 && m < p.n_mod) {
      *lo = p.ebeg[m];
      *hi = p.eend[m];
    } else {
      *hi = 0;  // no candidates: the row's routed slots get id -1
      if (p.status != nullptr) atomicOr(p.status, MOE_DEV_BAD_MODALITY);
    }
  }
}

// Writes the k chosen experts (bi, bv; value-ordered) and the shared slots.
__device__ __forceinline__ void write_topk(const TopKParams& p, int row, const float (&bv)[kMaxTopK],
                                           const int (&bi)[kMaxTopK]) {
  const float m = bv[0];
  float w[kMaxTopK];
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxTopK; ++i) {
    w[i] = (i < p.k && bi[i] >= 0) ? expf(bv[i] - m) : 0.f;
    sum += w[i];
  }
  const float inv = sum > 0.f ? 1.0f / sum : 0.f;
  const int ko = p.k_out > 0 ? p.k_out : p.k;
  int32_t* io = p.idx + static_cast<int64_t>(row) * ko;
  float* go = p.gate + static_cast<int64_t>(row) * ko;
#pragma unroll
  for (int i = 0; i < kMaxTopK; ++i) {
    if (i < p.k) {
      io[i] = bi[i];
      go[i] = w[i] * inv;
    }
  }
  for (int j = 0; j < p.n_shared; ++j) {
    io[p.k + j] = p.E + j;
    go[p.k + j] = 1.0f;
  }
}

// Inserts (s, e) into the descending list bv/bi (kMaxTopK slots) when s beats
// its last entry.  The list is sorted, so slot q keeps its entry when it is
// >= s, takes s when slot q-1 is >= s (or q = 0), and otherwise takes slot
// q-1's entry: every slot is decided from two comparisons, no chain of
// swaps.  Entries equal to s stay ahead of it (e grows along the row, so ties
// go to the lower expert index).
__device__ __forceinline__ void topk_insert(float (&bv)[kMaxTopK], int (&bi)[kMaxTopK], float s, int e) {
  bool ge[kMaxTopK];
#pragma unroll
  for (int q = 0; q < kMaxTopK; ++q) ge[q] = bv[q] >= s;
#pragma unroll
  for (int q = kMaxTopK - 1; q >= 0; --q) {
    const bool put = (q == 0) || ge[q - 1];
    const float shifted_v = q > 0 ? bv[q - 1] : s;
    const int shifted_i = q > 0 ? bi[q - 1] : e;
    bv[q] = ge[q] ? bv[q] : (put ? s : shifted_v);
    bi[q] = ge[q] ? bi[q] : (put ? e : shifted_i);
  }
}

// Columns [col, col + 32) of the row's score accumulator (only the first 16
// when !two), bias added; the missing half reads as -inf.
__device__ __forceinline__ void topk_load(const TopKParams& p, uint32_t taddr, int col, bool two, float (&s)[32]) {
  uint32_t u[32];
  __syncwarp();
  ptx::tmem_ld16(taddr + col, *reinterpret_cast<uint32_t(*)[16]>(&u[0]));
  if (two) ptx::tmem_ld16(taddr + col + 16, *reinterpret_cast<uint32_t(*)[16]>(&u[16]));
  ptx::tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    s[j] = (j < 16 || two) ? __uint_as_float(u[j]) : -INFINITY;
    if (p.bias != nullptr && (j < 16 || two) && col + j < p.E) s[j] += __ldg(p.bias + col + j);
  }
}

// v[j] for a j that differs between lanes, from registers: a 5-level select
// tree on the bits of j (a dynamic register index would go through local
// memory).
__device__ __forceinline__ float topk_pick(const float (&v)[32], int j) {
  float a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = (j & 1) ? v[2 * i + 1] : v[2 * i];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = (j & 2) ? a[2 * i + 1] : a[2 * i];
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = (j & 4) ? a[2 * i + 1] : a[2 * i];
#pragma unroll
  for (int i = 0; i < 2; ++i) a[i] = (j & 8) ? a[2 * i + 1] : a[2 * i];
  return (j & 16) ? a[1] : a[0];
}

// Scans the row's columns [c0, c1) (multiples of 16) of the score
// accumulator: bias, optional logits output, and the running top list for
// experts in [e_lo, e_hi).
//
// Each thread owns one row, and with k winners in every row nearly every
// column holds a winner of some lane of the warp, so inserting column by
// column makes the whole warp run an insertion at almost every column.  The
// scan therefore runs twice.  The first pass takes the maximum of each of
// kTauGroups column groups (column j of a 32-column batch is in group
// j % kTauGroups) and sets tau to the k-th largest of those maxima: k
// different groups hold a score >= tau, so the k-th best score of the range
// is >= tau and no member of the top k (ties included) is below it.  The
// second pass marks each lane's columns with s >= tau, a few per batch, and
// inserts only those, in column order, one per lane per step: the list then
// ends with the same first k entries as a scan of every column would.  Only
// the first k entries are used (written out or merged); later slots may
// differ from a full scan's.  NaN scores are never inserted, as before.
__device__ __forceinline__ void topk_scan(const TopKParams& p, uint32_t taddr, int c0, int c1, int e_lo, int e_hi,
                                          float* lrow, float (&bv)[kMaxTopK], int (&bi)[kMaxTopK]) {
  constexpr int kTauGroups = 16;
  static_assert(kTauGroups >= kMaxTopK, "tau needs at least k groups");
  if (e_hi > p.E) e_hi = p.E;
  float gm[kTauGroups];
#pragma unroll
  for (int g = 0; g < kTauGroups; ++g) gm[g] = -INFINITY;
#pragma unroll 1
  for (int col = c0; col < c1; col += 32) {
    const bool two = col + 16 < c1;
    float s[32];
    topk_load(p, taddr, col, two, s);
    const int lo = e_lo - col, hi = e_hi - col;
    if (__all_sync(0xffffffffu, lo <= 0 && hi >= (two ? 32 : 16))) {
#pragma unroll
      for (int j = 0; j < 32; ++j) gm[j % kTauGroups] = fmaxf(gm[j % kTauGroups], s[j]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j >= lo && j < hi) gm[j % kTauGroups] = fmaxf(gm[j % kTauGroups], s[j]);
    }
    if (lrow != nullptr) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if ((j < 16 || two) && col + j < p.E) lrow[col + j] = s[j];
    }
  }
  // descending bitonic sort of the group maxima; tau = the k-th largest
  constexpr int kLog = 4;
  static_assert(kTauGroups == 1 << kLog, "bitonic network size");
#pragma unroll
  for (int lg = 1; lg <= kLog; ++lg) {  // merged run length 2^lg
#pragma unroll
    for (int ls = kLog - 1; ls >= 0; --ls) {  // compare distance 2^ls, for ls < lg
#pragma unroll
      for (int i = 0; i < kTauGroups; ++i) {
        const int l = i ^ (1 << ls);
        if (ls < lg && l > i) {
          const float x = gm[i], y = gm[l];
          const bool desc = (i & (1 << lg)) == 0;
          gm[i] = desc ? fmaxf(x, y) : fminf(x, y);
          gm[l] = desc ? fminf(x, y) : fmaxf(x, y);
        }
      }
    }
  }
  // a select chain, not gm[p.k - 1]: an indexed read would put gm in local memory
  float tau = gm[kMaxTopK - 1];
#pragma unroll
  for (int q = kMaxTopK - 2; q >= 0; --q) tau = (p.k - 1 <= q) ? gm[q] : tau;
#pragma unroll 1
  for (int col = c0; col < c1; col += 32) {
    const bool two = col + 16 < c1;
    float s[32];
    topk_load(p, taddr, col, two, s);
    const int lo = e_lo - col, hi = e_hi - col;
    uint32_t mask = 0;
    if (__all_sync(0xffffffffu, lo <= 0 && hi >= (two ? 32 : 16))) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (s[j] >= tau) mask |= 1u << j;
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j >= lo && j < hi && s[j] >= tau) mask |= 1u << j;
    }
    const int steps = __reduce_max_sync(0xffffffffu, __popc(mask));
    // unrolled by two: the next candidate's lookup does not depend on the
    // list and overlaps the current insertion
#pragma unroll 2
    for (int it = 0; it < steps; ++it) {
      const int j = __ffs(mask) - 1;  // -1 once this lane has no candidate left
      mask &= mask - 1;
      const float v = topk_pick(s, j & 31);
      // -inf leaves the list unchanged: every entry is >= it
      topk_insert(bv, bi, (j >= 0 && v > bv[kMaxTopK - 1]) ? v : -INFINITY, col + j);
    }
  }
}

// The whole row by one thread: scan all BN columns, then write the top k.
template <int BN>
__device__ __forceinline__ void topk_row(const TopKParams& p, uint32_t taddr, int row, bool valid) {
  float bv[kMaxTopK];
  int bi[kMaxTopK];
#pragma unroll
  for (int i = 0; i < kMaxTopK; ++i) { bv[i] = -INFINITY; bi[i] = -1; }
  int e_lo, e_hi;
  expert_range(p, row, valid, &e_lo, &e_hi);
  float* lrow = (p.logits != nullptr && valid) ? p.logits + static_cast<int64_t>(row) * p.E : nullptr;
  topk_scan(p, taddr, 0, BN, e_lo, e_hi, lrow, bv, bi);
  if (!valid) return;
  write_topk(p, row, bv, bi);
}

// Router stage 2: summed head scores (fp32 accumulator, all E experts in one
// tile) -> top-k epilogue.  One TMEM lane is one token.  Eight epilogue
// warps: the two warps of a lane quadrant scan one half of the experts each;
// the upper half's warp hands its list (through the staging area) to the
// lower half's warp, which merges it in and writes the result.  Every
// candidate of the upper half has a higher expert index than the lower
// half's, so inserting them after it keeps ties with the lower index.
struct EpiTopK {
  using Params = TopKParams;
  static constexpr int kWarps = 8;
  template <int BN>
  static __device__ __forceinline__ void run(const Params& p0, const TileCoord& c, uint32_t taddr, int r,
                                             EpiCtx& ctx) {
    const int row0 = c.row0 + r;
    const bool valid = row0 < c.row_end;
    TopKParams p = p0;
    int row = row0;
    if (p0.T > 0) {  // batched: group c.group owns its own outputs
      const int64_t g = c.group;
      const int ko = p0.k_out > 0 ? p0.k_out : p0.k;
      p.idx = p0.idx + g * p0.T * ko;
      p.gate = p0.gate + g * p0.T * ko;
      if (p0.logits != nullptr) p.logits = p0.logits + g * p0.T * p0.E;
      if (p0.bias != nullptr) p.bias = p0.bias + g * p0.E;
      row = row0 - static_cast<int>(g) * p0.T;
    }
    float bv[kMaxTopK];
    int bi[kMaxTopK];
#pragma unroll
    for (int i = 0; i < kMaxTopK; ++i) { bv[i] = -INFINITY; bi[i] = -1; }
    int e_lo, e_hi;
    expert_range(p, row, valid, &e_lo, &e_hi);
    float* lrow = (p.logits != nullptr && valid) ? p.logits + static_cast<int64_t>(row) * p.E : nullptr;
    if constexpr (BN < 32) {  // one warp per quadrant is enough
      if (ctx.part == 1) return;
      topk_scan(p, taddr, 0, BN, e_lo, e_hi, lrow, bv, bi);
    } else {
      constexpr int kHalf = BN / 2;
      const uint32_t vbuf = ctx.scratch, ibuf = ctx.scratch + kMaxTopK * kBM * 4;  // [slot][tile row]
      const uint32_t parity = ctx.hand_uses & 1u;
      ++ctx.hand_uses;
      if (ctx.part == 1) {
        topk_scan(p, taddr, kHalf, BN, e_lo, e_hi, lrow, bv, bi);
        if (!ptx::mbar_wait(ctx.hand_free, parity ^ 1u, ctx.abort, ctx.wait_ns)) {
          ctx.failed = true;
          return;
        }
#pragma unroll
        for (int q = 0; q < kMaxTopK; ++q) {
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(vbuf + static_cast<uint32_t>((q * kBM + r) * 4)), "f"(bv[q])
                       : "memory");
          asm volatile("st.shared.s32 [%0], %1;" ::"r"(ibuf + static_cast<uint32_t>((q * kBM + r) * 4)), "r"(bi[q])
                       : "memory");
        }
        ptx::mbar_arrive(ctx.hand_full);
        return;
      }
      topk_scan(p, taddr, 0, kHalf, e_lo, e_hi, lrow, bv, bi);
      if (!ptx::mbar_wait(ctx.hand_full, parity, ctx.abort, ctx.wait_ns)) {
        ctx.failed = true;
        return;
      }
      float cv[kMaxTopK];
      int ci[kMaxTopK];
#pragma unroll
      for (int q = 0; q < kMaxTopK; ++q) {
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(cv[q]) : "r"(vbuf + static_cast<uint32_t>((q * kBM + r) * 4))
                     : "memory");
        asm volatile("ld.shared.s32 %0, [%1];" : "=r"(ci[q]) : "r"(ibuf + static_cast<uint32_t>((q * kBM + r) * 4))
                     : "memory");
      }
      ptx::mbar_arrive(ctx.hand_free);
#pragma unroll
      for (int q = 0; q < kMaxTopK; ++q)
        if (ci[q] >= 0 && cv[q] > bv[kMaxTopK - 1]) topk_insert(bv, bi, cv[q], ci[q]);
    }
    if (!valid) return;
    write_topk(p, row, bv, bi);
  }
};

}  // namespace moe
