// Sorting stage: counting-sort permutation of the (token, slot) pairs into
// expert-contiguous order, and the row gather x -> x_perm.
// This is the "sorting" step of the MagiMoE operator library ("Sand.ai: The world's first 100-billion-parameter open-source MoE video generation model MAGI Preview" (36kr), section "02. Two Key Technical Decision Points").
//
//   1. hist    : per token block, per-expert counts            (blocks of kTokBlock tokens)
//   2. assign  : each block first forms its own bases from all blocks' counts
//                (per expert, the counts of earlier blocks plus the exclusive
//                prefix over experts of the totals = offsets; block 0 writes
//                offsets), then row of (t, e) = offsets[e] + #{t' < t : t' chose e};
//                within a block the rank comes from per-warp bitmasks, so the
//                order is fixed by the token index and never by the order of atomics
//   3. gather  : one warp per token reads x[t] once and writes it to its k rows
// The three are chained with programmatic dependent launch: each kernel lets
// the next one be scheduled as soon as all of its blocks are running, and
// waits (griddepcontrol.wait) for its predecessor's completion and memory
// before touching anything the predecessor writes or reads, so a kernel's
// launch and ramp overlap the previous kernel's tail.
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"
#include "moe.h"
#include "ptx.cuh"

namespace moe {

constexpr int kTokBlock = 2048;   // tokens per hist/assign block
constexpr int kAssignWarps = 16;  // warps per assign block; each owns kTokBlock/16 tokens

// Loads token t's k expert ids.  An id outside [0, E), or a repeat of an
// earlier slot's id, becomes -1 (left out of the permutation) and sets *bad.
__device__ __forceinline__ void load_slots(const int32_t* __restrict__ row, int k, int E, int (&ex)[kMaxTopK],
                                           bool& bad) {
#pragma unroll
  for (int s = 0; s < kMaxTopK; ++s) {
    ex[s] = -1;
    if (s < k) {
      const int e = __ldg(row + s);
      bool ok = (e >= 0 && e < E);
#pragma unroll
      for (int q = 0; q < s; ++q) ok = ok && (ex[q] != e);
      if (ok) ex[s] = e;
      else bad = true;
    }
  }
}

__global__ void __launch_bounds__(256) dispatch_hist_kernel(const int32_t* __restrict__ topk_idx, int64_t T, int k,
                                                            int E, int32_t* __restrict__ block_counts,
                                                            int* status) {
  ptx::griddep_wait();
  ptx::griddep_launch();
  // head blockIdx.y of a batch of independent sorts
  topk_idx += static_cast<int64_t>(blockIdx.y) * T * k;
  block_counts += static_cast<int64_t>(blockIdx.y) * gridDim.x * E;
  __shared__ int hist[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTokBlock;
  const int64_t t1 = min(T, t0 + kTokBlock);
  bool bad = false;
  for (int64_t t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
    int ex[kMaxTopK];
    load_slots(topk_idx + t * k, k, E, ex, bad);
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s)
      if (ex[s] >= 0) atomicAdd(&hist[ex[s]], 1);
  }
  if (bad) atomicOr(status, MOE_DEV_BAD_EXPERT_ID);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    block_counts[static_cast<int64_t>(blockIdx.x) * E + e] = hist[e];
}

// kAssignWarps warps; warp w owns tokens [t0 + w*span, t0 + (w+1)*span) of the block.
__global__ void __launch_bounds__(kAssignWarps * 32) dispatch_assign_kernel(
    const int32_t* __restrict__ topk_idx, int64_t T, int k, int E, const int32_t* __restrict__ block_counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ row_of, int32_t* __restrict__ src_token) {
  ptx::griddep_wait();
  ptx::griddep_launch();
  // head blockIdx.y of a batch of independent sorts
  topk_idx += static_cast<int64_t>(blockIdx.y) * T * k;
  block_counts += static_cast<int64_t>(blockIdx.y) * gridDim.x * E;
  offsets += static_cast<int64_t>(blockIdx.y) * (E + 1);
  row_of += static_cast<int64_t>(blockIdx.y) * T * k;
  src_token += static_cast<int64_t>(blockIdx.y) * T * k;
  __shared__ int wcnt[kAssignWarps][kMaxExperts];   // per-warp counts, then per-warp cursors
  __shared__ unsigned mask[kAssignWarps][kMaxExperts];
  __shared__ int s_base[kMaxExperts];                // this block's first row of each expert
  __shared__ int s_off[kMaxExperts + 1];             // offsets (exclusive prefix of the totals)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = static_cast<int>(gridDim.x);

  // this block's bases: per expert the counts of the blocks before it, and
  // the totals over all blocks (every block forms the same totals)
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int pre = 0, tot = 0;
#pragma unroll 4
    for (int b = 0; b < nblk; ++b) {
      const int c = __ldg(block_counts + static_cast<int64_t>(b) * E + e);
      tot += c;
      pre += (b < static_cast<int>(blockIdx.x)) ? c : 0;
    }
    s_base[e] = pre;
    s_off[e] = tot;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive prefix over experts of the totals
    int carry = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = (e < E) ? s_off[e] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < E) s_off[e] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_off[E] = carry;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    if (e < E) s_base[e] += s_off[e];
    if (blockIdx.x == 0) offsets[e] = s_off[e];
  }
  constexpr int span = kTokBlock / kAssignWarps;
  const int64_t tb = static_cast<int64_t>(blockIdx.x) * kTokBlock;
  const int64_t w0 = tb + warp * span;
  const int64_t w1 = min(T, w0 + span);

  for (int e = lane; e < E; e += 32) { wcnt[warp][e] = 0; mask[warp][e] = 0u; }
  __syncwarp();
  bool bad = false;
  for (int64_t t = w0 + lane; t < w1; t += 32) {
    int ex[kMaxTopK];
    load_slots(topk_idx + t * k, k, E, ex, bad);
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s)
      if (ex[s] >= 0) atomicAdd(&wcnt[warp][ex[s]], 1);
  }
  __syncthreads();
  // exclusive prefix over warps, seeded with the block's global base
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = s_base[e];
    for (int w = 0; w < kAssignWarps; ++w) {
      const int c = wcnt[w][e];
      wcnt[w][e] = run;
      run += c;
    }
  }
  __syncthreads();

  // 32 tokens at a time, one per lane, in token order.  For each expert the
  // warp builds a bitmask of the lanes that chose it; a pair's row is the
  // expert's cursor plus the number of lower lanes in that mask.  Only the
  // lowest lane holding an expert advances its cursor and clears its mask.
  const unsigned lt = (1u << lane) - 1u;
  for (int64_t tb0 = w0; tb0 < w1; tb0 += 32) {
    const int64_t t = tb0 + lane;
    const bool live = t < w1;
    int ex[kMaxTopK];
    if (live) {
      load_slots(topk_idx + t * k, k, E, ex, bad);
    } else {
#pragma unroll
      for (int s = 0; s < kMaxTopK; ++s) ex[s] = -1;
    }
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s)
      if (ex[s] >= 0) atomicOr(&mask[warp][ex[s]], 1u << lane);
    __syncwarp();
    int rank[kMaxTopK];
    unsigned msk[kMaxTopK];
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
      msk[s] = (ex[s] >= 0) ? mask[warp][ex[s]] : 0u;
      rank[s] = (ex[s] >= 0) ? wcnt[warp][ex[s]] + __popc(msk[s] & lt) : -1;
    }
    __syncwarp();
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
      if (ex[s] >= 0 && (msk[s] & lt) == 0u) {
        wcnt[warp][ex[s]] += __popc(msk[s]);
        mask[warp][ex[s]] = 0u;
      }
    }
    __syncwarp();
    if (live) {
#pragma unroll
      for (int s = 0; s < kMaxTopK; ++s) {
        if (s < k) {
          row_of[t * k + s] = rank[s];
          if (rank[s] >= 0) src_token[rank[s]] = static_cast<int32_t>(t);
        }
      }
    }
  }
  (void)bad;  // already reported by the histogram pass
}

// One warp per token (grid-stride): read the row once into registers, write it
// to each of its k destination rows.  16-byte vectors; d % 8 == 0.
__global__ void __launch_bounds__(256) dispatch_gather_kernel(const uint4* __restrict__ x, int64_t T, int d_vec,
                                                              int64_t x_ld_vec, int64_t x_head_vec, int heads, int k,
                                                              const int32_t* __restrict__ row_of, int64_t rows,
                                                              uint4* __restrict__ x_perm) {
  ptx::griddep_wait();
  ptx::griddep_launch();
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  constexpr int kVec = 8;  // uint4 per lane per pass (4 KB per warp)
  for (int64_t ht = warp_global; ht < T * heads; ht += nwarps) {
    const int64_t h = ht / T, t = ht - h * T;  // (head, token)
    int dst = -1;
    if (lane < k) dst = __ldg(row_of + (h * T + t) * k + lane);
    const uint4* src = x + h * x_head_vec + t * x_ld_vec;
    uint4* x_perm_h = x_perm + h * rows * d_vec;
    for (int c0 = 0; c0 < d_vec; c0 += 32 * kVec) {
      uint4 v[kVec];
#pragma unroll
      for (int j = 0; j < kVec; ++j) {
        const int c = c0 + j * 32 + lane;
        if (c < d_vec) v[j] = __ldg(src + c);
      }
      for (int s = 0; s < k; ++s) {
        const int r = __shfl_sync(0xffffffffu, dst, s);
        if (r < 0 || r >= rows) continue;
        uint4* o = x_perm_h + static_cast<int64_t>(r) * d_vec;
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
          const int c = c0 + j * 32 + lane;
          if (c < d_vec) o[c] = v[j];
        }
      }
    }
  }
}

int launch_dispatch(const DispatchArgs& a, cudaStream_t stream) {
  const int nblk = static_cast<int>((a.T + kTokBlock - 1) / kTokBlock);
  const int heads = a.heads > 1 ? a.heads : 1;
  if (launch_pdl(dispatch_hist_kernel, dim3(nblk, heads), dim3(256), 0, stream, a.topk_idx, a.T, a.k, a.E,
                 a.block_counts, a.status) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_pdl(dispatch_assign_kernel, dim3(nblk, heads), dim3(kAssignWarps * 32), 0, stream, a.topk_idx, a.T, a.k,
                 a.E, a.block_counts, a.offsets, a.row_of, a.src_token) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (a.x_perm != nullptr) {
    const int d_vec = a.d / 8;
    const int64_t want = (a.T * heads + 7) / 8;  // 8 warps (tokens) per CTA
    const int grid = static_cast<int>(want < a.sm_count * 8LL ? want : a.sm_count * 8LL);
    const int64_t x_ld_vec = (a.x_ld ? a.x_ld : a.d) / 8;
    if (launch_pdl(dispatch_gather_kernel, dim3(grid), dim3(256), 0, stream, reinterpret_cast<const uint4*>(a.x), a.T,
                   d_vec, x_ld_vec, a.x_head_off / 8, heads, a.k, a.row_of, a.T * a.k,
                   reinterpret_cast<uint4*>(a.x_perm)) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t dispatch_scratch_bytes(int64_t T, int E) {
  const int64_t nblk = (T + kTokBlock - 1) / kTokBlock;
  return static_cast<size_t>(nblk * E) * sizeof(int32_t);
}

size_t dispatch_counter_cells(int64_t T, int E) { return static_cast<size_t>((T + kTokBlock - 1) / kTokBlock) * E; }

}  // namespace moe
