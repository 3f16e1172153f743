// Fused router: latent projection, summed head scores, softmax and top-k in
// one persistent tcgen05 kernel (the multi-head latent routing of
// "MAGI-2 Preview" (heyaiwiki), Architecture table, "Routing" row and FAQ "What is
// MagiMoE?").  The latent vector h never leaves the SM:
// per 128-token tile and per head j,
//   1. h_j = x W_lat[j]^T accumulates in TMEM columns [0, head_dim) (fp32),
//   2. the epilogue warps read it back 64 columns at a time and write the bf16
//      hi/lo pair (hi = bf16(h), lo = bf16(h - hi)) into a 128-byte-swizzled
//      shared-memory operand (one chunk buffer: the shared memory goes to a
//      four-stage operand ring instead, which measured faster than three
//      stages with two chunk buffers),
//   3. s += [h_hi | h_lo] W_head[:, head j]^T accumulates into TMEM columns
//      [256, 256 + E) over all heads (the head sum is the K reduction),
// and after the last head the epilogue applies bias, top-k and gates.
//
// Roles (192 threads, one CTA per SM): warp 0 lane 0 loads with TMA (x and
// W_lat slices for the latent MMAs, W_head chunks for the score MMAs, one
// ring), warp 1 lane 0 issues tcgen05.mma, warps 2..5 convert and select.
// Every wait is bounded as in the GEMM engine.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "epilogues.cuh"
#include "gemm_tc.cuh"
#include "internal.h"
#include "moe.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kRStages = 4;  // four 48 KB stages: three measured 9% slower on the clip
constexpr int kRABytes = kBM * kBK * 2;          // x slice: 128 rows x 64
constexpr int kRBBytes = 256 * kBK * 2;          // W_lat head slice or W_head chunk: <= 256 rows x 64
constexpr int kRStageBytes = kRABytes + kRBBytes;
constexpr int kHsBytes = kBM * 128;              // one 128 x 64 bf16 operand chunk
constexpr int kRDynBytes = kRStages * kRStageBytes + 2 * kHsBytes + 1024;
constexpr uint32_t kLogitCol = 256;              // TMEM column of the score accumulator

struct FusedArgs {
  int T, d, n_heads, head_dim, E;
  int groups;         // G work items per token tile, each owning n_heads / G heads
  float* partial;     // G > 1: [G, T, E] fp32 partial scores (summed by topk_combine_kernel)
  TopKParams tp;      // G == 1: the epilogue selects directly
  int* status;
  uint64_t wait_ns;
};

template <int BNE>
__global__ void __launch_bounds__(kGemmThreads, 1)
router_fused_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_wlat,
                    const __grid_constant__ CUtensorMap tmap_whead, FusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* hs = smem + kRStages * kRStageBytes;  // one chunk buffer: [hi][lo]

  __shared__ __align__(8) uint64_t full_bar[kRStages];
  __shared__ __align__(8) uint64_t empty_bar[kRStages];
  __shared__ __align__(8) uint64_t h_full, h_free, lg_full, lg_free, drain_bar;
  __shared__ __align__(8) uint64_t hs_full[2], hs_free[2];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (a.T + kBM - 1) / kBM;
  const int n_items = m_tiles * a.groups;
  const int hpg = a.n_heads / a.groups;
  const int num_kb = a.d / kBK;
  const int chunks = a.head_dim / 64;
  const uint32_t lat_bytes = kRABytes + static_cast<uint32_t>(a.head_dim) * 128u;
  const uint32_t head_bytes = static_cast<uint32_t>(BNE) * 128u;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < kRStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&h_full), 1);
    ptx::mbar_init(ptx::smem_u32(&h_free), 128);
    ptx::mbar_init(ptx::smem_u32(&lg_full), 1);
    ptx::mbar_init(ptx::smem_u32(&lg_free), 128);
    ptx::mbar_init(ptx::smem_u32(&drain_bar), 1);
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ptx::smem_u32(&hs_full[b]), 128);
      ptx::mbar_init(ptx::smem_u32(&hs_free[b]), 1);
    }
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&s_tmem), 512);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmap_x);
    ptx::prefetch_tmap(&tmap_wlat);
    ptx::prefetch_tmap(&tmap_whead);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = s_tmem;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const uint64_t pol = ptx::policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, filled = 0, last_par = 0;
      bool ok = true;
      auto next_slot = [&](uint32_t bytes) -> uint32_t {  // returns the stage's shared address, or 0
        if (!ptx::mbar_wait(ptx::smem_u32(&empty_bar[stage]), phase ^ 1, &s_abort, a.wait_ns)) return 0;
        ptx::mbar_arrive_expect_tx(ptx::smem_u32(&full_bar[stage]), bytes);
        filled |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (phase << stage);
        return ptx::smem_u32(smem + stage * kRStageBytes);
      };
      auto advance = [&]() {
        if (++stage == kRStages) { stage = 0; phase ^= 1; }
      };
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const int row0 = (item / a.groups) * kBM;
        const int h0 = (item % a.groups) * hpg;
        for (int h = h0; h < h0 + hpg && ok; ++h) {
          for (int kb = 0; kb < num_kb; ++kb) {
            const uint32_t sa = next_slot(lat_bytes);
            if (sa == 0) { ok = false; break; }
            const uint32_t fb = ptx::smem_u32(&full_bar[stage]);
            ptx::tma_load_2d(sa, &tmap_x, kb * kBK, row0, fb, pol);
            ptx::tma_load_2d(sa + kRABytes, &tmap_wlat, kb * kBK, h * a.head_dim, fb, pol);
            advance();
          }
          for (int c = 0; c < chunks && ok; ++c) {
            const uint32_t sa = next_slot(head_bytes);
            if (sa == 0) { ok = false; break; }
            ptx::tma_load_2d(sa + kRABytes, &tmap_whead, h * a.head_dim + c * 64, 0,
                             ptx::smem_u32(&full_bar[stage]), pol);
            advance();
          }
        }
      }
      if (!ok) {
        atomicOr(a.status, MOE_DEV_TIMEOUT);
        s_abort = 1;
      }
      for (int s = 0; s < kRStages; ++s) {
        if (filled & (1u << s)) {
          const volatile int never = 0;
          if (!ptx::mbar_wait(ptx::smem_u32(&full_bar[s]), (last_par >> s) & 1u, &never, a.wait_ns))
            atomicOr(a.status, MOE_DEV_TIMEOUT);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc_lat = ptx::idesc_bf16_m128(a.head_dim);
      constexpr uint32_t idesc_lg = ptx::idesc_bf16_m128(BNE);
      const uint32_t t_h = tmem_base, t_lg = tmem_base + kLogitCol;
      int stage = 0;
      uint32_t phase = 0, nh = 0, nc = 0, nt = 0;
      bool ok = true;
      auto wait = [&](uint64_t& bar, uint32_t parity) {
        if (!ok) return false;
        if (!ptx::mbar_wait(ptx::smem_u32(&bar), parity, &s_abort, a.wait_ns)) ok = false;
        ptx::tc_fence_after();
        return ok;
      };
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        for (int h = 0; h < hpg && ok; ++h) {
          if (!wait(h_free, (nh & 1) ^ 1)) break;
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!wait(full_bar[stage], phase)) break;
            const uint32_t sa = ptx::smem_u32(smem + stage * kRStageBytes);
#pragma unroll
            for (int kk = 0; kk < kBK / kUK; ++kk)
              ptx::mma_bf16(t_h, ptx::sw128_desc(sa + kk * 32), ptx::sw128_desc(sa + kRABytes + kk * 32), idesc_lat,
                            (kb | kk) != 0 ? 1u : 0u);
            ptx::mma_commit(ptx::smem_u32(&empty_bar[stage]));
            if (++stage == kRStages) { stage = 0; phase ^= 1; }
          }
          if (!ok) break;
          ptx::mma_commit(ptx::smem_u32(&h_full));
          ++nh;
          for (int c = 0; c < chunks; ++c) {
            const int b = 0;  // one chunk buffer (its hi and lo halves)
            if (!wait(hs_full[b], nc & 1)) break;
            const bool first = (h == 0 && c == 0);
            if (first && !wait(lg_free, (nt & 1) ^ 1)) break;
            if (!wait(full_bar[stage], phase)) break;
            const uint32_t sb = ptx::smem_u32(smem + stage * kRStageBytes) + kRABytes;
            const uint32_t hi = ptx::smem_u32(hs + (2 * b) * kHsBytes), lo = hi + kHsBytes;
#pragma unroll
            for (int kk = 0; kk < kBK / kUK; ++kk)
              ptx::mma_bf16(t_lg, ptx::sw128_desc(hi + kk * 32), ptx::sw128_desc(sb + kk * 32), idesc_lg,
                            (first && kk == 0) ? 0u : 1u);
#pragma unroll
            for (int kk = 0; kk < kBK / kUK; ++kk)
              ptx::mma_bf16(t_lg, ptx::sw128_desc(lo + kk * 32), ptx::sw128_desc(sb + kk * 32), idesc_lg, 1u);
            ptx::mma_commit(ptx::smem_u32(&empty_bar[stage]));
            ptx::mma_commit(ptx::smem_u32(&hs_free[b]));
            if (++stage == kRStages) { stage = 0; phase ^= 1; }
            ++nc;
          }
        }
        if (!ok) break;
        ptx::mma_commit(ptx::smem_u32(&lg_full));
        ++nt;
      }
      if (!ok) {
        atomicOr(a.status, MOE_DEV_TIMEOUT);
        s_abort = 1;
      }
      ptx::mma_commit(ptx::smem_u32(&drain_bar));
      const volatile int never = 0;
      if (!ptx::mbar_wait(ptx::smem_u32(&drain_bar), 0, &never, a.wait_ns)) atomicOr(a.status, MOE_DEV_TIMEOUT);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // tile row = TMEM lane
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    uint32_t nh = 0, nc = 0, nt = 0;
    bool ok = true;
    auto wait = [&](uint64_t& bar, uint32_t parity) {
      const bool got = ptx::mbar_wait(ptx::smem_u32(&bar), parity, &s_abort, a.wait_ns);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) atomicOr(a.status, MOE_DEV_TIMEOUT);
        s_abort = 1;
        ok = false;
      }
      ptx::tc_fence_after();
      return ok;
    };
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const int tile = item / a.groups, g = item % a.groups;
      for (int h = 0; h < hpg && ok; ++h) {
        if (!wait(h_full, nh & 1)) break;
        ++nh;
        for (int c = 0; c < chunks; ++c) {
          uint32_t phi[32], plo[32];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float v[32];
            __syncwarp();
            tmem_ld32(lane_addr + c * 64 + half * 32, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float h0 = v[2 * i], h1 = v[2 * i + 1];
              const float b0 = __bfloat162float(__float2bfloat16_rn(h0));
              const float b1 = __bfloat162float(__float2bfloat16_rn(h1));
              phi[half * 16 + i] = pack_bf16x2(b0, b1);
              plo[half * 16 + i] = pack_bf16x2(h0 - b0, h1 - b1);
            }
          }
          if (c == chunks - 1) {  // every TMEM read of h_j is done: the next head may overwrite it
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_u32(&h_free));
          }
          const int b = 0;
          if (!wait(hs_free[b], (nc & 1) ^ 1)) break;
          const uint32_t hi = ptx::smem_u32(hs + (2 * b) * kHsBytes) + static_cast<uint32_t>(r) * 128u;
          const uint32_t lo = hi + kHsBytes;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t off = (static_cast<uint32_t>(j) ^ (static_cast<uint32_t>(r) & 7u)) << 4;
            ptx::st_shared_v4(hi + off, make_uint4(phi[4 * j], phi[4 * j + 1], phi[4 * j + 2], phi[4 * j + 3]));
            ptx::st_shared_v4(lo + off, make_uint4(plo[4 * j], plo[4 * j + 1], plo[4 * j + 2], plo[4 * j + 3]));
          }
          ptx::fence_proxy_async_smem();  // generic-proxy writes -> tensor-core (async proxy) reads
          ptx::mbar_arrive(ptx::smem_u32(&hs_full[b]));
          ++nc;
        }
      }
      if (!ok) break;
      if (!wait(lg_full, nt & 1)) break;
      ++nt;
      const int row = tile * kBM + r;
      if (a.groups == 1) {
        topk_row<BNE>(a.tp, lane_addr + kLogitCol, row, row < a.T);
      } else {  // this head group's partial scores for the row
        float* dst = a.partial + (static_cast<int64_t>(g) * a.T + row) * a.E;
#pragma unroll 1
        for (int col = 0; col < BNE; col += 16) {
          uint32_t u[16];
          __syncwarp();
          ptx::tmem_ld16(lane_addr + kLogitCol + col, u);
          ptx::tmem_ld_wait();
          if (row < a.T) {
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              if (col + j < a.E)  // E is a multiple of 4 whenever groups > 1
                *reinterpret_cast<float4*>(dst + col + j) =
                    make_float4(__uint_as_float(u[j]), __uint_as_float(u[j + 1]), __uint_as_float(u[j + 2]),
                                __uint_as_float(u[j + 3]));
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&lg_free));
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, 512);
  }
}

// Sums the G head-group partial scores of one token in group order, adds the
// bias and selects the top k (value descending, ties to the lower index) with
// k rounds of a warp arg-max; gates = softmax over the chosen k.
// One warp per token; lane l owns experts l, l + 32, ...
__global__ void __launch_bounds__(256) topk_combine_kernel(const float* __restrict__ partial, int groups, int T,
                                                           int E, TopKParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = wid; t < T; t += nw) {
    int e_lo, e_hi;
    expert_range(p, static_cast<int>(t), true, &e_lo, &e_hi);
    float v[kMaxExperts / 32];
#pragma unroll
    for (int j = 0; j < kMaxExperts / 32; ++j) {
      const int e = lane + 32 * j;
      float s = -INFINITY;
      if (e < E) {
        s = 0.f;
        for (int g = 0; g < groups; ++g) s += __ldg(partial + (static_cast<int64_t>(g) * T + t) * E + e);
        if (p.bias != nullptr) s += __ldg(p.bias + e);
        if (p.logits != nullptr) p.logits[t * E + e] = s;
      }
      v[j] = (e >= e_lo && e < e_hi) ? s : -INFINITY;
    }
    float sel_v[kMaxTopK];
    int sel_e[kMaxTopK];
#pragma unroll
    for (int i = 0; i < kMaxTopK; ++i) { sel_v[i] = -INFINITY; sel_e[i] = -1; }
#pragma unroll
    for (int i = 0; i < kMaxTopK; ++i) {
      if (i >= p.k) break;
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < kMaxExperts / 32; ++j) {
        const int e = lane + 32 * j;
        if (e < E && (v[j] > bv || (v[j] == bv && e < be))) { bv = v[j]; be = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
      }
      sel_v[i] = bv;
      sel_e[i] = (be < E && bv > -INFINITY) ? be : -1;
#pragma unroll
      for (int j = 0; j < kMaxExperts / 32; ++j)
        if (lane + 32 * j == be) v[j] = -INFINITY;
    }
    if (lane == 0) write_topk(p, static_cast<int>(t), sel_v, sel_e);
  }
}

template <int BNE>
int run_fused(const RouteArgs& a, int head_dim, cudaStream_t stream) {
  CUtensorMap tx, tl, th;
  if (!make_tmap_bf16_2d(&tx, a.x, a.d, a.T, kBK, kBM)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&tl, a.w_lat, a.d, a.L, kBK, head_dim)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&th, a.w_head, a.L, a.E, kBK, BNE)) return MOE_ERR_CUDA;
  FusedArgs fa{};
  fa.T = static_cast<int>(a.T);
  fa.d = a.d;
  fa.head_dim = head_dim;
  fa.n_heads = a.L / head_dim;
  fa.E = a.E;
  fa.tp = make_topk_params(a);
  fa.status = a.status;
  fa.wait_ns = kWaitLimitNs;
  // Head groups per token tile (G | n_heads).  Every tile re-reads its x slice
  // once per head, so the slices of the tiles in flight must stay in L2: take
  // at least the smallest G whose live slices fit in about a third of L2.
  // When there are fewer tiles than SMs, take the largest G that still gives
  // one work item per SM.  Partial scores need E % 4 == 0 and G * E <= L (they
  // live in the two-stage router's latent buffer).
  const int64_t m_tiles = (a.T + kBM - 1) / kBM;
  const double slice = static_cast<double>(kBM) * a.d * 2;
  int G = 1;
  if (a.E % 4 == 0 && a.partial != nullptr) {
    int g_l2 = 0, g_par = 1;
    for (int g = 1; g <= fa.n_heads; ++g) {
      if (fa.n_heads % g || static_cast<int64_t>(g) * a.E > a.L) continue;
      const int64_t live_tiles = std::min<int64_t>(m_tiles, std::max(1, a.sm_count / g));
      if (g_l2 == 0 && live_tiles * slice <= 40.0e6) g_l2 = g;
      if (m_tiles * g <= a.sm_count) g_par = g;
      if (g_l2 == 0) G = g;  // largest admissible so far, if nothing fits L2
    }
    G = std::max(g_l2 > 0 ? g_l2 : G, g_par);
  }
  fa.groups = G;
  fa.partial = a.partial;
  auto kern = router_fused_kernel<BNE>;
  static std::atomic<uint64_t> smem_set{0};
  if (!smem_attr_ready(kern, kRDynBytes, smem_set)) return MOE_ERR_CUDA;
  const int64_t items = m_tiles * G;
  const int grid = static_cast<int>(items < a.sm_count ? items : a.sm_count);
  kern<<<grid, kGemmThreads, kRDynBytes, stream>>>(tx, tl, th, fa);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  if (G > 1) {
    const int64_t want = (a.T + 7) / 8;
    const int cgrid = static_cast<int>(want < a.sm_count * 8LL ? want : a.sm_count * 8LL);
    topk_combine_kernel<<<cgrid, 256, 0, stream>>>(a.partial, G, static_cast<int>(a.T), a.E, fa.tp);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace

bool route_fused_supported(int head_dim) { return head_dim % 64 == 0 && head_dim >= 64 && head_dim <= 256; }

int launch_route_fused(const RouteArgs& a, int head_dim, cudaStream_t stream) {
  if (!route_fused_supported(head_dim)) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int E = a.E;
  if (E <= 16) return run_fused<16>(a, head_dim, stream);
  if (E <= 32) return run_fused<32>(a, head_dim, stream);
  if (E <= 64) return run_fused<64>(a, head_dim, stream);
  if (E <= 128) return run_fused<128>(a, head_dim, stream);
  return run_fused<256>(a, head_dim, stream);
}

}  // namespace moe
