// Internal interface between the C-ABI layer (moe_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>

namespace moe {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kMaxGemmGroups = 3072;  // row groups of one grouped-GEMM launch

// Raises a kernel's dynamic shared-memory limit on the current device the
// first time it is launched there; `done` (one per kernel) holds one bit per
// device.  Later launches, stream captures included, skip the call.
template <class Kern>
inline bool smem_attr_ready(Kern kern, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t{1} << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  done.fetch_or(bit, std::memory_order_release);
  return true;
}

// Launches `kern` with programmatic stream serialization: the grid may be
// scheduled while the previous kernel on the stream is still running, and
// waits for it with griddepcontrol.wait before it touches that kernel's data.
template <class... P, class... A>
inline cudaError_t launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<P>(args)...);
}

struct DispatchArgs {
  const uint16_t* x;
  const int32_t* topk_idx;
  int64_t T;
  int d, k, E;
  int32_t* offsets;
  int32_t* row_of;
  int32_t* src_token;
  uint16_t* x_perm;        // nullptr: permutation only
  int64_t x_ld;            // row stride of x in elements (0: d)
  // Independent sorts side by side (head-local layer): head h reads x's
  // columns from h * x_head_off and topk_idx[h], writes offsets[h], row_of[h],
  // src_token[h], x_perm[h] (each the single-sort size) and uses its own
  // block counters.  heads <= 1: one sort.
  int heads;
  int64_t x_head_off;
  int32_t* block_counts;   // scratch [nblk * E]: per-block expert counts
  int* status;
  int sm_count;
};

// Modality-specific routing and shared experts (zero-initialised: plain layer).
struct RouteExt {
  int n_shared;
  int n_mod;
  int ebeg[8], eend[8];
  const int32_t* modality;
};

struct RouteArgs {
  const uint16_t* x;
  const uint16_t* w_lat;
  const uint16_t* w_head;
  const float* bias;
  int32_t* topk_idx;
  float* topk_gate;
  float* logits;
  uint16_t* hl;            // scratch [T, 2L] bf16: latent hi | lo (two-stage router)
  float* partial;          // scratch for the fused router's head-group partial scores (aliases hl)
  int64_t T;
  int d, L, E, k;
  int head_dim;
  RouteExt ext;
  int* status;
  int sm_count;
};

struct FfnArgs {
  const uint16_t* x;         // [T, d], gathered GEMM-1 only
  const int32_t* src_token;  // [rows], gathered GEMM-1 only
  int64_t T;
  const uint16_t* x_perm;
  const int32_t* offsets;
  const uint16_t* w13;
  const uint16_t* w_down;
  uint16_t* act;
  uint16_t* y_perm;
  int64_t rows;            // T * k
  int d, I, E;
  int* status;
  int sm_count;
  // gate folded into expert GEMM-2 (launch_gemm2_gated): y_perm[r] is scaled by
  // gate[t, s] for the pair (t, s) with row_of[t, s] = r, t = src_token[r]
  const int32_t* row_of;     // [T, k]
  const float* gate;         // [T, k]
  int k;
  int32_t* tiles;            // scratch [E + 1] (the fused expert kernel's tile table)
  // fused expert kernel: row r of group g is x[src_token[r], (g / head_groups) * d + (0 .. d)),
  // x with x_ld elements per row
  int64_t x_ld;
  int head_groups;
};

struct CombineArgs {
  const uint16_t* y_perm;
  const int32_t* row_of;
  const float* gate;       // nullptr: rows already carry their gates (summed with weight 1)
  uint16_t* out;
  int64_t T;
  int d, k;
  int64_t out_ld;          // row stride of out in elements (0: d)
  // Independent combines side by side: head h reads y_perm[h], row_of[h],
  // gate[h] and writes out's columns from h * d (heads <= 1: one combine).
  int heads;
  int sm_count;
};

int launch_dispatch(const DispatchArgs& a, cudaStream_t stream);
size_t dispatch_scratch_bytes(int64_t T, int E);
size_t dispatch_counter_cells(int64_t T, int E);  // ceil(T / block) * E: the per-block counters
int launch_route(const RouteArgs& a, cudaStream_t stream);
int launch_route_two_stage(const RouteArgs& a, cudaStream_t stream);
bool route_fused_supported(int head_dim);
int launch_route_fused(const RouteArgs& a, int head_dim, cudaStream_t stream);
int launch_route_folded(const RouteArgs& a, const uint16_t* w_router, cudaStream_t stream);
int launch_fold_router(const uint16_t* w_head, const uint16_t* w_lat, int E, int L, int d, uint16_t* w_router,
                       cudaStream_t stream);
int launch_gemm1(const FfnArgs& a, cudaStream_t stream);
int launch_gemm2(const FfnArgs& a, cudaStream_t stream);
int launch_gemm2_gated(const FfnArgs& a, cudaStream_t stream);
int launch_gemm1_gather(const FfnArgs& a, cudaStream_t stream);
// Both expert GEMMs of narrow experts (d <= 256) in one kernel, act kept on chip:
// y_perm = (silu(x_perm W_gate^T) * (x_perm W_up^T)) W_down^T; reads x_perm, offsets,
// w13, w_down, rows, d, I, E (groups); no group limit.
bool ffn_fused_supported(int D, int I);
int launch_ffn_fused(const FfnArgs& a, cudaStream_t stream);
int launch_combine(const CombineArgs& a, cudaStream_t stream);
int launch_selftest_timeout(uint16_t* scratch, int* status, uint64_t limit_ns, cudaStream_t stream);
int launch_ffn_fused_selftest(uint8_t* scratch, int* status, uint64_t limit_ns, cudaStream_t stream);
int launch_prepare_w13(const uint16_t* w_gate, const uint16_t* w_up, uint16_t* w13, int E, int I, int d,
                       cudaStream_t stream);

// cuTensorMapEncodeTiled, resolved once through the runtime (no -lcuda).
bool make_tmap_bf16_2d(void* tmap /* CUtensorMap* */, const void* base, uint64_t cols, uint64_t rows,
                       uint32_t box_cols, uint32_t box_rows, uint64_t row_stride_elems = 0);

int launch_router_headlocal(const uint16_t* x, int64_t T, int d, int H, int Dh, const uint16_t* w_router, int E,
                            int k, const float* bias, int32_t* idx, float* gate, float* logits, int* status,
                            int sm_count, cudaStream_t stream);



}  // namespace moe
