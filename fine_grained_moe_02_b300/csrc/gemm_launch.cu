// Host launchers for the tcgen05 GEMM engine: the two router GEMMs and the
// two grouped expert GEMMs, plus the tensor-map encoder and the w13 builder.
// The router is the multi-head latent routing of "MAGI-2 Preview" (heyaiwiki), Architecture
// table ("Architecture" and "Routing" rows: 12 latent heads x 256, top-6);
// the expert GEMMs are the "calculation" step over many small matrices of
// "Sand.ai: The world's first 100-billion-parameter open-source MoE video generation model MAGI Preview" (36kr), section "02. Two Key Technical Decision Points".
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "epilogues.cuh"
#include "gemm_tc.cuh"
#include "internal.h"
#include "moe.h"

namespace moe {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

template <int BN, class Epi, int GW = 0>
int run_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td, const GemmShape& shape,
             const typename Epi::Params& ep, int grid, cudaStream_t stream, int b_box_rows) {
  using S = GemmSmem<BN>;
  // the B tensor map must deliver exactly this kernel's per-CTA B slice, or
  // the stage byte count and the shared-memory ring would disagree
  if (b_box_rows != BN) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (shape.groups < 1 || shape.groups > kMaxGroups) return MOE_ERR_UNSUPPORTED_SHAPE;  // shared tile table
  {  // the kernel counts tiles in 32-bit ints: at most (rows / tile rows + groups) m-tiles per n-tile
    const int64_t rows_all = shape.batched ? static_cast<int64_t>(shape.groups) * shape.M : shape.M;
    const int64_t m_tiles = rows_all / kBM + shape.groups;
    if (shape.N % BN != 0 || m_tiles * (shape.N / BN) >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  }
  if ((GW > 0) != (shape.a_gather != nullptr)) return MOE_ERR_UNSUPPORTED_SHAPE;  // gathered A needs gather warps
  auto kern = gemm_tc_kernel<BN, Epi, GW>;
  constexpr int kThreads = gemm_threads<Epi, GW>();
  // once per device: later calls (and stream captures) launch without it
  static std::atomic<uint64_t> smem_set{0};
  if (!smem_attr_ready(kern, S::kDynBytes, smem_set)) return MOE_ERR_CUDA;
  if (grid < 1) grid = 1;
  // a plain launch: chaining the GEMMs and the combine by programmatic
  // dependent launch measured 3% slower on the clip workload
  kern<<<grid, kThreads, S::kDynBytes, stream>>>(ta, tb, td, shape, ep);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <class Epi>
int run_gemm_bn(int bn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td,
                const GemmShape& shape, const typename Epi::Params& ep, int grid, cudaStream_t stream,
                int b_box_rows) {
  switch (bn) {
    case 256: return run_gemm<256, Epi>(ta, tb, td, shape, ep, grid, stream, b_box_rows);
    case 128: return run_gemm<128, Epi>(ta, tb, td, shape, ep, grid, stream, b_box_rows);
    case 64: return run_gemm<64, Epi>(ta, tb, td, shape, ep, grid, stream, b_box_rows);
    case 32: return run_gemm<32, Epi>(ta, tb, td, shape, ep, grid, stream, b_box_rows);
    case 16: return run_gemm<16, Epi>(ta, tb, td, shape, ep, grid, stream, b_box_rows);
    default: return MOE_ERR_UNSUPPORTED_SHAPE;
  }
}


int pick_bn(int n) {
  if (n % 256 == 0) return 256;
  if (n % 128 == 0) return 128;
  return 64;
}

}  // namespace

bool make_tmap_bf16_2d(void* tmap, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                       uint32_t box_rows, uint64_t row_stride_elems) {
  auto enc = encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {(row_stride_elems ? row_stride_elems : cols) * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(static_cast<CUtensorMap*>(tmap), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Router, default path: two tensor-core GEMMs with h in HBM as a bf16 hi/lo
// pair.  On B300 it beats the on-chip kernel (router_fused.cu, moe_route_fused)
// because that kernel's per-head conversion of h serialises with its MMAs.
int launch_route(const RouteArgs& a, cudaStream_t stream) { return launch_route_two_stage(a, stream); }

// Two-stage router (h through HBM as a bf16 hi/lo pair):
//         stage 1  hl = [hi | lo](x W_lat^T)            dense GEMM, N = L, fused hi/lo split
//         stage 2  s  = hl [W_head | W_head]^T + bias   dense GEMM, K = 2L, N = E, fused top-k
int launch_route_two_stage(const RouteArgs& a, cudaStream_t stream) {
  const int64_t m_tiles = (a.T + kBM - 1) / kBM;
  CUtensorMap ta, tb, td;
  {
    const int bn = pick_bn(a.L);
    if (!make_tmap_bf16_2d(&ta, a.x, a.d, a.T, kBK, kBM)) return MOE_ERR_CUDA;
    if (!make_tmap_bf16_2d(&tb, a.w_lat, a.d, a.L, kBK, bn)) return MOE_ERR_CUDA;
    if (!make_tmap_bf16_2d(&td, a.hl, 2ULL * a.L, a.T, kBK, 32)) return MOE_ERR_CUDA;
    GemmShape sh{a.d, a.d, a.L, 1, nullptr, static_cast<int>(a.T), a.status};
    EpiHiLo::Params ep{a.hl, 2LL * a.L, a.L};
    const int64_t tiles = m_tiles * (a.L / bn);
    const int grid = static_cast<int>(tiles < a.sm_count ? tiles : a.sm_count);
    const int rc = run_gemm_bn<EpiHiLo>(bn, ta, tb, td, sh, ep, grid, stream, bn);
    if (rc != MOE_OK) return rc;
  }
  {
    const int bn = a.E <= 16 ? 16 : a.E <= 32 ? 32 : a.E <= 64 ? 64 : a.E <= 128 ? 128 : 256;
    if (!make_tmap_bf16_2d(&ta, a.hl, 2ULL * a.L, a.T, kBK, kBM)) return MOE_ERR_CUDA;
    if (!make_tmap_bf16_2d(&tb, a.w_head, a.L, a.E, kBK, bn)) return MOE_ERR_CUDA;
    GemmShape sh{2 * a.L, a.L, bn, 1, nullptr, static_cast<int>(a.T), a.status};
    EpiTopK::Params ep = make_topk_params(a);
    const int grid = static_cast<int>(m_tiles < a.sm_count ? m_tiles : a.sm_count);
    return run_gemm_bn<EpiTopK>(bn, ta, tb, ta /* no bulk output */, sh, ep, grid, stream, bn);
  }
}

// Folded router: s = [x | x] w_router^T + bias (K = 2d; w_router = [W_eff hi | lo])
// with the top-k epilogue.
int launch_route_folded(const RouteArgs& a, const uint16_t* w_router, cudaStream_t stream) {
  const int64_t m_tiles = (a.T + kBM - 1) / kBM;
  const int bn = a.E <= 16 ? 16 : a.E <= 32 ? 32 : a.E <= 64 ? 64 : a.E <= 128 ? 128 : 256;
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_2d(&ta, a.x, a.d, a.T, kBK, kBM)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&tb, w_router, 2ULL * a.d, a.E, kBK, bn)) return MOE_ERR_CUDA;
  GemmShape sh{2 * a.d, 2 * a.d, bn, 1, nullptr, static_cast<int>(a.T), a.status, nullptr, a.d};
  EpiTopK::Params ep = make_topk_params(a);
  const int grid = static_cast<int>(m_tiles < a.sm_count ? m_tiles : a.sm_count);
  return run_gemm_bn<EpiTopK>(bn, ta, tb, ta, sh, ep, grid, stream, bn);
}

// All heads' routers of the head-local layer in one launch: problem h is
// s_h = x[:, h*Dh : (h+1)*Dh] W_router[h]^T (+ bias[h]) with the top-k epilogue,
// outputs idx/gate [H, T, k], logits [H, T, E].
int launch_router_headlocal(const uint16_t* x, int64_t T, int d, int H, int Dh, const uint16_t* w_router, int E,
                            int k, const float* bias, int32_t* idx, float* gate, float* logits, int* status,
                            int sm_count, cudaStream_t stream) {
  const int64_t m_tiles = (T + kBM - 1) / kBM;
  const int bn = E <= 16 ? 16 : E <= 32 ? 32 : E <= 64 ? 64 : E <= 128 ? 128 : 256;
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_2d(&ta, x, d, T, kBK, kBM)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&tb, w_router, Dh, static_cast<uint64_t>(H) * E, kBK, bn)) return MOE_ERR_CUDA;
  GemmShape sh{Dh, Dh, bn, H, nullptr, static_cast<int>(T), status, nullptr, 0, 0, 0, 1, Dh, E};
  TopKParams ep{};
  ep.bias = bias;
  ep.logits = logits;
  ep.idx = idx;
  ep.gate = gate;
  ep.E = E;
  ep.k = k;
  ep.status = status;
  ep.T = static_cast<int>(T);
  const int64_t tiles = m_tiles * H;
  const int grid = static_cast<int>(tiles < sm_count ? tiles : sm_count);
  return run_gemm_bn<EpiTopK>(bn, ta, tb, ta, sh, ep, grid, stream, bn);
}

// Expert GEMM-1 over ragged groups (device offsets), SwiGLU fused: act = silu(x Wg^T) * (x Wu^T).
int launch_gemm1(const FfnArgs& a, cudaStream_t stream) {
  CUtensorMap ta, tb, td;
  const int rows = static_cast<int>(a.rows);
  const int n = 2 * a.I;
  const int bn = (n % 256 == 0) ? 256 : 128;
  if (!make_tmap_bf16_2d(&ta, a.x_perm, a.d, a.rows, kBK, kBM)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&tb, a.w13, a.d, static_cast<uint64_t>(a.E) * n, kBK, bn)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&td, a.act, a.I, a.rows, kBK, 32)) return MOE_ERR_CUDA;
  GemmShape sh{a.d, a.d, n, a.E, a.offsets, rows, a.status};
  EpiSwiGLU::Params ep{a.act, a.I};
  return (bn == 256) ? run_gemm<256, EpiSwiGLU>(ta, tb, td, sh, ep, a.sm_count, stream, bn)
                     : run_gemm<128, EpiSwiGLU>(ta, tb, td, sh, ep, a.sm_count, stream, bn);
}

// Expert GEMM-1 with the row gather fused into the A loads: A row r is
// x[src_token[r]], copied by kGatherWarps warps with 16-byte cp.async, so the
// permuted copy x_perm never exists.  Four warps: on the clip workload the
// gathered GEMM-1 takes 1.28x the time of GEMM-1 on x_perm with two, 1.12x
// with four, 1.20x with eight (the gather count must stay even: the rows one
// warp instruction covers must keep the 128-byte swizzle phase).
constexpr int kGatherWarps = 4;

int launch_gemm1_gather(const FfnArgs& a, cudaStream_t stream) {
  // A rows come from x through src_token (cp.async gather warps); tmap_a is unused
  CUtensorMap tb, td;
  const int rows = static_cast<int>(a.rows);
  const int n = 2 * a.I;
  const int bn = (n % 256 == 0) ? 256 : 128;
  if (!make_tmap_bf16_2d(&tb, a.w13, a.d, static_cast<uint64_t>(a.E) * n, kBK, bn)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&td, a.act, a.I, a.rows, kBK, 32)) return MOE_ERR_CUDA;
  GemmShape sh{a.d, a.d, n, a.E, a.offsets, rows, a.status, a.src_token};
  sh.a_src = a.x;
  sh.a_ld = a.d;
  sh.a_src_rows = static_cast<int>(a.T);
  EpiSwiGLU::Params ep{a.act, a.I};
  return (bn == 256) ? run_gemm<256, EpiSwiGLU, kGatherWarps>(tb, tb, td, sh, ep, a.sm_count, stream, bn)
                     : run_gemm<128, EpiSwiGLU, kGatherWarps>(tb, tb, td, sh, ep, a.sm_count, stream, bn);
}

// Expert GEMM-2 over ragged groups: y_perm = act Wd^T.
int launch_gemm2(const FfnArgs& a, cudaStream_t stream) {
  CUtensorMap ta, tb, td;
  const int rows = static_cast<int>(a.rows);
  const int bn = pick_bn(a.d);
  if (!make_tmap_bf16_2d(&ta, a.act, a.I, a.rows, kBK, kBM)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&tb, a.w_down, a.I, static_cast<uint64_t>(a.E) * a.d, kBK, bn)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&td, a.y_perm, a.d, a.rows, kBK, 32)) return MOE_ERR_CUDA;
  GemmShape sh{a.I, a.I, a.d, a.E, a.offsets, rows, a.status};
  EpiStoreBf16::Params ep{a.y_perm, a.d};
  return run_gemm_bn<EpiStoreBf16>(bn, ta, tb, td, sh, ep, a.sm_count, stream, bn);
}

// Expert GEMM-2 with the gate folded into the epilogue:
// y_perm[r] = gate[src_token[r], s] * (act Wd^T)[r], row_of[src_token[r], s] = r.
int launch_gemm2_gated(const FfnArgs& a, cudaStream_t stream) {
  CUtensorMap ta, tb, td;
  const int rows = static_cast<int>(a.rows);
  const int bn = pick_bn(a.d);
  if (!make_tmap_bf16_2d(&ta, a.act, a.I, a.rows, kBK, kBM)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&tb, a.w_down, a.I, static_cast<uint64_t>(a.E) * a.d, kBK, bn)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&td, a.y_perm, a.d, a.rows, kBK, 32)) return MOE_ERR_CUDA;
  GemmShape sh{a.I, a.I, a.d, a.E, a.offsets, rows, a.status};
  EpiStoreGated::Params ep{a.y_perm, a.d, a.src_token, a.row_of, a.gate, a.T, a.k};
  return run_gemm_bn<EpiStoreGated>(bn, ta, tb, td, sh, ep, a.sm_count, stream, bn);
}

// Self-test of the bounded waits: one 128 x 256 x 64 tile whose producer
// issues nothing, so the MMA and epilogue waits run out after `limit_ns`.
// Operands and output live in `scratch` (>= 112 KB); nothing is loaded or stored.
int launch_selftest_timeout(uint16_t* scratch, int* status, uint64_t limit_ns, cudaStream_t stream) {
  CUtensorMap ta, tb, td;
  uint16_t* a = scratch;                 // [128, 64]
  uint16_t* b = scratch + 128 * 64;      // [256, 64]
  uint16_t* d = scratch + 384 * 64;      // [128, 256]
  if (!make_tmap_bf16_2d(&ta, a, 64, 128, kBK, kBM)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&tb, b, 64, 256, kBK, 256)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&td, d, 256, 128, kBK, 32)) return MOE_ERR_CUDA;
  GemmShape sh{64, 64, 256, 1, nullptr, 128, status, nullptr, 0, limit_ns, 1};
  EpiStoreBf16::Params ep{d, 256};
  return run_gemm<256, EpiStoreBf16>(ta, tb, td, sh, ep, 1, stream, 256);
}

// w13[e, 128b + j] = j < 64 ? w_gate[e, 64b + j] : w_up[e, 64b + j - 64]   (rows of d)
__global__ void __launch_bounds__(256) prepare_w13_kernel(const uint4* __restrict__ wg, const uint4* __restrict__ wu,
                                                          uint4* __restrict__ w13, int64_t n_rows, int I,
                                                          int d_vec) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = wid; r < n_rows; r += nw) {       // r = e * 2I + row
    const int64_t e = r / (2 * I);
    const int row = static_cast<int>(r - e * 2 * I);
    const int b = row >> 7, j = row & 127;
    const uint4* src = (j < 64 ? wg : wu) + (e * I + b * 64 + (j & 63)) * d_vec;
    uint4* dst = w13 + r * d_vec;
    for (int c = lane; c < d_vec; c += 32) dst[c] = __ldg(src + c);
  }
}

int launch_prepare_w13(const uint16_t* w_gate, const uint16_t* w_up, uint16_t* w13, int E, int I, int d,
                       cudaStream_t stream) {
  const int64_t n_rows = static_cast<int64_t>(E) * 2 * I;
  const int64_t want = (n_rows + 7) / 8;
  const int grid = static_cast<int>(want < 4096 ? want : 4096);
  prepare_w13_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const uint4*>(w_gate),
                                               reinterpret_cast<const uint4*>(w_up), reinterpret_cast<uint4*>(w13),
                                               n_rows, I, d / 8);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
